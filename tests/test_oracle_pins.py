"""Pins for the CPU oracle against facts fixed outside the oracle itself:
hand-derived closed forms (tests/golden), brute force on tiny inputs with
plain Python integers, exact rational arithmetic, invariants of the
definitions, and library routines for the special cases they cover.

Runs on CPU only (no GPU marker)."""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from ternary_w2a8_linear_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.strip() for c in line.split(";")]


# ---------------------------------------------------------------------------
# Activation quantiser
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", list(_rows("quant_act_closed_forms.txt")))
def test_quant_act_golden(case):
    xs, qs, rs, amax = case
    x = np.array([[float(v) for v in xs.split()]], dtype=np.float32)
    q, a_scale, rowsum = oracle.quant_act(x)
    assert q[0].tolist() == [int(v) for v in qs.split()]
    assert int(rowsum[0]) == int(rs)
    expect_scale = np.float32(float(amax)) / np.float32(127) if float(amax) else np.float32(0)
    assert a_scale[0] == expect_scale


def test_quant_act_one_hot():
    for v in (1e-3, 0.7, -3.25, 1e4, -1e-20):
        x = np.zeros((1, 37), dtype=np.float32)
        x[0, 11] = v
        q, a_scale, rowsum = oracle.quant_act(x)
        expect = np.zeros(37, dtype=np.int8)
        expect[11] = 127 if v > 0 else -127
        assert np.array_equal(q[0], expect)
        assert rowsum[0] == expect[11]


def test_quant_act_rational_bound():
    """Each code is within 1/2 (+ the fp32 rounding of s and of x*s) of the
    exact rational x*127/amax; the largest-magnitude entry maps to +-127."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 300)).astype(np.float32)
    x[2] *= np.float32(1e-3)
    x[3, 17] = np.float32(55.0)
    q, a_scale, rowsum = oracle.quant_act(x)
    for m in range(x.shape[0]):
        amax = Fraction(float(np.max(np.abs(x[m]))))
        for k in range(x.shape[1]):
            exact = Fraction(float(x[m, k])) * 127 / amax
            assert abs(Fraction(int(q[m, k])) - exact) <= Fraction(1, 2) + Fraction(1, 2**14)
            if x[m, k] == 0:
                assert q[m, k] == 0
            else:
                assert q[m, k] == 0 or np.sign(q[m, k]) == np.sign(x[m, k])
        k_max = int(np.argmax(np.abs(x[m])))
        assert abs(int(q[m, k_max])) == 127
        assert int(rowsum[m]) == sum(int(v) for v in q[m])
        assert a_scale[m] == np.float32(np.max(np.abs(x[m]))) / np.float32(127)


def test_quant_act_monotone_and_odd():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((3, 513)).astype(np.float32)
    q, _, _ = oracle.quant_act(x)
    qn, _, rn = oracle.quant_act(-x)
    assert np.array_equal(qn, -q)
    for m in range(3):
        order = np.argsort(x[m], kind="stable")
        assert np.all(np.diff(q[m][order].astype(int)) >= 0)


def test_quant_act_power_of_two_scaling():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 200)).astype(np.float32)
    q, a, r = oracle.quant_act(x)
    for j in (-7, -1, 3, 10):
        q2, a2, r2 = oracle.quant_act((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(q2, q) and np.array_equal(r2, r)
        assert np.array_equal(a2, (a * np.float32(2.0 ** j)).astype(np.float32))


def test_quant_act_bf16_widening():
    vals = np.array([[1.0, -2.5, 0.0078125, 3.0e38, -1.0e-30]], dtype=np.float32)
    bits = inputs.to_bf16_bits(vals)
    widened = oracle.bf16_bits_to_f32(bits)
    import torch
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(widened, ref)


# ---------------------------------------------------------------------------
# bf16 rounding helper against torch's conversion (a library routine)
# ---------------------------------------------------------------------------
def test_f32_to_bf16_matches_torch():
    import torch
    rng = np.random.default_rng(10)
    x = np.concatenate([
        rng.standard_normal(10000).astype(np.float32) * np.float32(1e3),
        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 0.0, -0.0, 2**-130, 65504.0], dtype=np.float32),
    ])
    ours = oracle.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------
# Absmean ternarisation
# ---------------------------------------------------------------------------
def test_ternarize_constant_magnitude():
    rng = np.random.default_rng(11)
    sgn = np.where(rng.random((9, 33)) < 0.5, -1.0, 1.0).astype(np.float32)
    for c in (0.125, 0.7, 3.0):
        T, g = oracle.ternarize_absmean(sgn * np.float32(c))
        assert g == np.float32(c)
        assert np.array_equal(T, sgn.astype(np.int8))


def test_ternarize_ties_and_clamp():
    W = np.array([[1.0, 3.0, -1.0, -3.0]], dtype=np.float32)  # mean|W| = 2 -> ratios +-0.5, +-1.5
    T, g = oracle.ternarize_absmean(W)
    assert g == np.float32(2.0)
    assert T.tolist() == [[0, 1, 0, -1]]
    W = np.array([[2.0, -2.0, 1.0, 3.0, -1.0, 0.0]], dtype=np.float32)  # mean 1.5
    T, g = oracle.ternarize_absmean(W)
    assert g == np.float32(1.5)
    assert T.tolist() == [[1, -1, 1, 1, -1, 0]]


def test_ternarize_sum_exact_then_rounded():
    """mean|W| must not depend on the summation order.  For
    W = [2^30, 64, 2^-23, 2^-23] the exact sum 2^30 + 64 + 2^-22 is an fp64
    number; divided by 4 it is 2^28 + 16 + 2^-24, just above the fp32 midpoint
    2^28 + 16 between 2^28 and 2^28 + 32, so gamma = 2^28 + 32.  Adding the
    terms left to right in fp64 loses both 2^-23 (each a tie to even) and
    would give the midpoint, rounded down to 2^28."""
    W = np.array([[2.0 ** 30, 64.0, 2.0 ** -23, 2.0 ** -23]], dtype=np.float32)
    T, g = oracle.ternarize_absmean(W)
    assert g == np.float32(2.0 ** 28 + 32)
    assert T.tolist() == [[1, 0, 0, 0]]
    seq = np.float64(0.0)
    for v in W.ravel().astype(np.float64):
        seq += v
    assert np.float32(seq / 4) == np.float32(2.0 ** 28)  # the order-dependent value differs


def test_ternarize_gamma_against_exact_rationals():
    """gamma against the sum of |W| taken in exact rational arithmetic, rounded
    once to fp64 (Fraction -> float rounds correctly), over a wide range of
    magnitudes, subnormals and zeros included."""
    from fractions import Fraction
    rng = np.random.default_rng(23)
    for trial in range(6):
        n = int(rng.integers(1, 400))
        mag = np.exp2(rng.uniform(-140, 100, n)).astype(np.float32)
        W = (mag * np.where(rng.random(n) < 0.5, -1, 1)).astype(np.float32).reshape(1, n)
        W[0, rng.random(n) < 0.1] = 0.0
        if trial == 0:
            W[0, :3] = np.float32(1e-45)  # the smallest subnormal
        exact = sum((Fraction(float(abs(v))) for v in W.ravel()), Fraction(0))
        want = max(np.float32(np.float64(float(exact)) / np.float64(n)), np.float32(1e-5))
        _, g = oracle.ternarize_absmean(W)
        assert g == want


def test_ternarize_epsilon():
    T, g = oracle.ternarize_absmean(np.zeros((3, 4), dtype=np.float32))
    assert g == np.float32(1e-5) and not T.any()
    T, g = oracle.ternarize_absmean(np.full((2, 2), 1e-7, dtype=np.float32))
    assert g == np.float32(1e-5) and not T.any()


# ---------------------------------------------------------------------------
# Integer accumulation: brute force with plain Python integers
# ---------------------------------------------------------------------------
def _brute_acc(T, q):
    N, K = len(T), len(T[0])
    M = len(q)
    return [[sum(int(T[n][k]) * int(q[m][k]) for k in range(K)) for n in range(N)] for m in range(M)]


def test_gemm_exhaustive_tiny():
    rng = np.random.default_rng(12)
    q = rng.integers(-127, 128, size=(2, 3)).astype(np.int8)
    for vals in itertools.product((-1, 0, 1), repeat=6):
        T = np.array(vals, dtype=np.int8).reshape(2, 3)
        assert oracle.gemm_acc(T, q).tolist() == _brute_acc(T.tolist(), q.tolist())


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (4, 2, 9), (16, 3, 4), (2, 8, 1)])
def test_gemm_brute_force_shapes(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    T = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    assert oracle.gemm_acc(T, q).tolist() == _brute_acc(T.tolist(), q.tolist())


def test_gemm_invariants():
    rng = np.random.default_rng(13)
    K = 48
    q = rng.integers(-127, 128, size=(5, K)).astype(np.int8)
    assert not oracle.gemm_acc(np.zeros((7, K), np.int8), q).any()
    eye = np.eye(K, dtype=np.int8)
    assert np.array_equal(oracle.gemm_acc(eye, q), q.astype(np.int64))
    assert np.array_equal(oracle.gemm_acc(-eye, q), -q.astype(np.int64))
    perm = rng.permutation(K)
    P = eye[perm]
    assert np.array_equal(oracle.gemm_acc(P, q), q[:, perm].astype(np.int64))
    ones = np.ones((3, 11008), dtype=np.int8)
    q127 = np.full((2, 11008), 127, dtype=np.int8)
    assert np.all(oracle.gemm_acc(ones, q127) == 127 * 11008)


def test_gemm_rejects_int32_overflow():
    # int32 overflow needs > 16.9 M terms of 127; fake it with a wide int input
    with pytest.raises(OverflowError):
        oracle.gemm_acc(np.ones((1, 2), np.int64) * 2**30, np.ones((1, 2), np.int64) * 2)


# ---------------------------------------------------------------------------
# Dequant epilogue: exact rationals
# ---------------------------------------------------------------------------
def test_dequant_exact_rational():
    rng = np.random.default_rng(14)
    acc = rng.integers(-400000, 400000, size=(4, 50))
    acc[0, :3] = 0
    a_scale = (rng.random(4).astype(np.float32) * np.float32(0.1)).astype(np.float32)
    w_scale = np.float32(0.0312)
    y = oracle.dequant(acc, a_scale, w_scale)
    assert y.dtype == np.float32
    assert np.all(y[0, :3] == 0)
    for m in range(4):
        for n in range(50):
            exact = Fraction(int(acc[m, n])) * Fraction(float(a_scale[m])) * Fraction(float(w_scale))
            got = Fraction(float(y[m, n]))
            ulp = Fraction(float(np.spacing(np.float32(abs(float(exact)))))) if exact else Fraction(0)
            assert abs(got - exact) <= ulp


def test_dequant_power_of_two_scaling():
    rng = np.random.default_rng(15)
    acc = rng.integers(-10**6, 10**6, size=(3, 40))
    a = rng.random(3).astype(np.float32)
    y = oracle.dequant(acc, a, np.float32(0.02))
    y2 = oracle.dequant(acc, a, np.float32(0.02) * np.float32(8))
    assert np.array_equal(y2, (y * np.float32(8)).astype(np.float32))


def test_dequant_bf16_is_rounded_f32():
    import torch
    rng = np.random.default_rng(16)
    acc = rng.integers(-10**5, 10**5, size=(2, 300))
    a = rng.random(2).astype(np.float32)
    y32 = oracle.dequant(acc, a, np.float32(0.03))
    yb = oracle.dequant(acc, a, np.float32(0.03), out="bf16")
    ref = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, ref)


def test_linear_activation_sign_and_scale():
    T, w, x = inputs.random_problem(17, 3, 40, 70)
    y, acc, q, a, r = oracle.w2a8_linear(T, w, x)
    yn, accn, qn, _, _ = oracle.w2a8_linear(T, w, -x)
    assert np.array_equal(accn, -acc) and np.array_equal(qn, -q)
    assert np.array_equal(yn, -y)
    y4, acc4, _, _, _ = oracle.w2a8_linear(T, w, (x * np.float32(4)).astype(np.float32))
    assert np.array_equal(acc4, acc) and np.array_equal(y4, (y * np.float32(4)).astype(np.float32))


def test_linear_row_independence():
    T, w, x = inputs.random_problem(18, 6, 33, 90)
    y, acc, *_ = oracle.w2a8_linear(T, w, x)
    for m in range(6):
        y1, acc1, *_ = oracle.w2a8_linear(T, w, x[m:m + 1])
        assert np.array_equal(acc1[0], acc[m]) and np.array_equal(y1[0], y[m])


# ---------------------------------------------------------------------------
# Packed format: hand-derived words, round trip, trailer
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", list(_rows("pack_words.txt")))
def test_pack_golden_words(case):
    shape, entries, words = case
    N, K = (int(v) for v in shape.split())
    T = np.zeros((N, K), dtype=np.int8)
    if entries != "-":
        for e in entries.split():
            n, k, t = (int(v) for v in e.split(":"))
            T[n, k] = t
    pk = oracle.pack_tiles(T)
    assert pk.size == oracle.packed_bytes(N, K)
    body = pk[:-16].view(np.uint32)
    for w in words.split():
        idx, val = w.split(":")
        assert body[int(idx)] == int(val, 16), (idx, hex(int(body[int(idx)])))
    assert oracle.read_trailer(pk, N, K) == (oracle.TRAILER_MAGIC, N, K, 0)


@pytest.mark.parametrize("N,K", [(1, 1), (5, 17), (128, 128), (129, 300), (640, 2560), (300, 1000)])
def test_pack_round_trip(N, K):
    T = inputs.ternary(np.random.default_rng(N + K), (N, K), None)
    pk = oracle.pack_tiles(T)
    assert np.array_equal(oracle.unpack_tiles(pk, N, K), T)
    nt, kt = -(-N // 128), -(-K // 128)
    assert pk.size == nt * kt * 4096 + 16


def test_pack_counts_invalid():
    T = np.zeros((3, 40), dtype=np.int8)
    T[0, 0] = 2
    T[2, 39] = -128
    pk = oracle.pack_tiles(T)
    assert oracle.read_trailer(pk, 3, 40)[3] == 2


def test_unpack_rejects_code_three():
    pk = oracle.pack_tiles(np.zeros((1, 16), np.int8))
    pk[0] = 0xFF
    with pytest.raises(ValueError):
        oracle.unpack_tiles(pk, 1, 16)


def test_ternary_code_without_division():
    """The device pack computes the ternary code of w under scale g (a normal
    fp32 >= 1e-5) as (w > g/2) - (w < -g/2) instead of clamp(rint(w / g)).
    This checks that identity against the oracle's definition (fp32 IEEE
    division, round half to even, clamp) on random weights and on every float
    next to the boundaries +-g/2 and +-3g/2, for many g."""
    rng = np.random.default_rng(2024)
    gs = np.concatenate([np.float32([1e-5, 2.0 ** -17, 1.0, 0.75, 3.0, 1e30]),
                         (np.exp2(rng.uniform(-16, 20, 400))).astype(np.float32)])
    for g in gs:
        g = np.float32(g)
        h = np.float32(g * np.float32(0.5))
        assert np.float64(h) * 2 == np.float64(g)  # g / 2 is exact
        pts = []
        for c in (h, np.float32(3 * h), np.float32(g)):
            v = c
            lo = c
            for _ in range(3):
                v = np.nextafter(v, np.float32(np.inf))
                lo = np.nextafter(lo, np.float32(0))
                pts += [v, lo]
            pts.append(c)
        w = np.array(pts + [np.float32(0), np.float32(1e-45), np.float32(3e38)], dtype=np.float32)
        w = np.concatenate([w, -w, (rng.standard_normal(2000) * g).astype(np.float32)])
        with np.errstate(over="ignore"):
            ref = np.clip(np.rint((w / g).astype(np.float32)), -1, 1).astype(np.int8)
        got = (w > h).astype(np.int8) - (w < -h).astype(np.int8)
        assert np.array_equal(got, ref), (g, w[got != ref][:4])


def _rn32(r: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 value (ties to even), exactly;
    written from the format definition (24-bit significand), normal range."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    n, rem = divmod(a, ulp)
    if rem > ulp / 2 or (rem == ulp / 2 and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_chain_dequant_order():
    """dequant_chain is RN32(RN32(acc * a_scale) * w_scale), checked with exact
    rationals; on these samples that order differs from the single fp64
    rounding of dequant at least once, so the order is really pinned."""
    rng = np.random.default_rng(606)
    M = 400
    acc = rng.integers(-2 ** 20, 2 ** 20, size=(M, 1))
    a = (rng.uniform(1e-4, 1e-1, M)).astype(np.float32)
    w = np.float32(0.0137)
    got = oracle.dequant_chain(acc, a, w)
    single = oracle.dequant(acc, a, w)
    differs = 0
    for m in range(M):
        t = _rn32(Fraction(int(acc[m, 0])) * Fraction(float(a[m])))
        ref = _rn32(t * Fraction(float(w)))
        assert Fraction(float(got[m, 0])) == ref, m
        differs += got[m, 0] != single[m, 0]
    assert differs > 0


def test_chain_identity_is_a_fixed_point():
    """T = I, w_scale = 1: the first layer re-scales the codes (y = q * a_scale,
    whose absmax is 127 * a_scale), so every later layer quantises back to the
    same codes and acc == q; the recorded amax is the output's row absmax."""
    K = 300
    x = np.random.default_rng(607).standard_normal((5, K)).astype(np.float32)
    I = np.eye(K, dtype=np.int8)
    res = oracle.linear_chain([(I, np.float32(1.0))] * 4, x)
    for l, r in enumerate(res):
        assert np.array_equal(r["acc"], r["q"].astype(np.int64))
        assert np.array_equal(r["amax"], np.max(np.abs(r["y"]), axis=1))
        if l:
            assert np.array_equal(r["q"], res[0]["q"])


def test_chain_negation_alternates_sign():
    """T = -I, w_scale = 1/2, fp32 outputs: y = -q * a_scale / 2 (the halving
    is exact), so each layer's codes are the negation of the previous layer's.
    (With bf16 outputs the rounding of q * a_scale to 8 bits can move a code by
    one, so no such identity holds there.)"""
    K = 257
    x = np.random.default_rng(608).standard_normal((3, K)).astype(np.float32)
    negI = -np.eye(K, dtype=np.int8)
    res = oracle.linear_chain([(negI, np.float32(0.5))] * 5, x, out="f32")
    for l in range(1, 5):
        assert np.array_equal(res[l]["q"], -res[l - 1]["q"]), l


# ---------------------------------------------------------------------------
# FP8 (E4M3) "fast" draft projection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", list(_rows("e4m3_closed_forms.txt")))
def test_e4m3_round_golden(case):
    x, r, _ = case
    got = oracle.e4m3_round(np.array([float(x)], dtype=np.float32))[0]
    assert got == float(r)


def test_e4m3_grid_has_127_nonnegative_values():
    # exponent fields 0..15 x mantissas 0..7, minus the one NaN code (S.1111.111)
    a = np.linspace(0.0, 500.0, 2_000_001, dtype=np.float32)
    fine = np.ldexp(np.arange(0, 2 ** 14, dtype=np.float64), -14).astype(np.float32)  # dense near zero
    vals = np.unique(oracle.e4m3_round(np.concatenate([a, fine])))
    assert len(vals) == 127
    assert vals[0] == 0.0 and vals[1] == 2.0 ** -9 and vals[-1] == 448.0
    # every value is j * 2^(E-3) with 8 <= j <= 15 above 2^-6, j * 2^-9 below
    for v in vals[1:]:
        e = max(int(np.floor(np.log2(v))), -6)
        j = v / 2.0 ** (e - 3)
        assert j == int(j) and (j <= 15) and (j >= 8 or e == -6)


def test_e4m3_round_matches_torch_float8_cast():
    # library routine: torch's fp32 -> float8_e4m3fn conversion (round to
    # nearest even) on values inside the finite range, including every midpoint
    torch = pytest.importorskip("torch")
    grid = np.unique(oracle.e4m3_round(np.linspace(0, 448, 400_001, dtype=np.float32)))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    rnd = np.random.default_rng(11).standard_normal(200_000).astype(np.float32) * np.float32(40)
    x = np.concatenate([grid.astype(np.float32), mids, -mids, rnd, rnd * np.float32(1e-3)])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    assert np.array_equal(oracle.e4m3_round(x), ref)


@pytest.mark.parametrize("case", list(_rows("quant_act_fp8_closed_forms.txt")))
def test_quant_act_fp8_golden(case):
    xs, es, amax = case
    x = np.array([[float(v) for v in xs.split()]], dtype=np.float32)
    e, a_scale = oracle.quant_act_fp8(x)
    assert e[0].tolist() == [float(v) for v in es.split()]
    expect = np.float32(float(amax)) / np.float32(448) if float(amax) else np.float32(0)
    assert a_scale[0] == expect


def test_quant_act_fp8_one_hot_and_power_of_two_scaling():
    rng = np.random.default_rng(5)
    for _ in range(20):
        K = int(rng.integers(1, 300))
        x = np.zeros((1, K), dtype=np.float32)
        k0 = int(rng.integers(0, K))
        x[0, k0] = np.float32(rng.standard_normal())
        e, _ = oracle.quant_act_fp8(x)
        assert e[0, k0] == np.sign(x[0, k0]) * 448.0
        assert np.count_nonzero(e) == 1
    x = rng.standard_normal((4, 777)).astype(np.float32)
    e0, s0 = oracle.quant_act_fp8(x)
    for j in (-7, -1, 3, 9):
        ej, sj = oracle.quant_act_fp8((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(ej, e0)
        assert np.array_equal(sj, (s0 * np.float32(2.0 ** j)).astype(np.float32))


def test_gemm_acc_fp8_brute_force():
    rng = np.random.default_rng(17)
    for _ in range(30):
        M, N, K = (int(v) for v in rng.integers(1, 5, size=3))
        T = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
        x = rng.standard_normal((M, K)).astype(np.float32)
        e, _ = oracle.quant_act_fp8(x)
        acc = oracle.gemm_acc_fp8(T, e)
        for m, n in itertools.product(range(M), range(N)):
            exact = sum(Fraction(int(T[n, k])) * Fraction(float(e[m, k])) for k in range(K))
            assert Fraction(float(acc[m, n])) == exact


def test_fp8_linear_identity_and_negation():
    rng = np.random.default_rng(23)
    K = 96
    x = rng.standard_normal((3, K)).astype(np.float32)
    I = np.eye(K, dtype=np.int8)
    _, acc, e, _ = oracle.fp8_linear(I, np.float32(1), x)
    assert np.array_equal(acc, e)
    _, acc_n, _, _ = oracle.fp8_linear(-I, np.float32(1), x)
    assert np.array_equal(acc_n, -e)
    _, acc_x, e_x, _ = oracle.fp8_linear(I, np.float32(1), -x)
    assert np.array_equal(e_x, -e) and np.array_equal(acc_x, -acc)
    assert np.array_equal(oracle.fp8_linear(np.zeros((5, K), np.int8), np.float32(0.5), x)[1], np.zeros((3, 5)))


def test_fp8_linear_dequant_exact_rational():
    rng = np.random.default_rng(29)
    T = rng.integers(-1, 2, size=(7, 200)).astype(np.int8)
    x = rng.standard_normal((2, 200)).astype(np.float32)
    w = np.float32(0.0371)
    y, acc, _, a_scale = oracle.fp8_linear(T, w, x)
    for m in range(2):
        for n in range(7):
            exact = Fraction(float(acc[m, n])) * Fraction(float(a_scale[m])) * Fraction(float(w))
            assert y[m, n] == np.float32(float(exact))  # one rounding of the exact product
