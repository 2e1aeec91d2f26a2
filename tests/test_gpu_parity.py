"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element, on seeded inputs at sizes that span several tiles plus a
ragged tail.  int8 codes, row sums, int32 accumulators and packed bytes are
bit-exact; fp32 outputs within 1e-5 relative (exact zero where acc == 0);
bf16 outputs within one bf16 ulp of the oracle's fp32 value rounded to bf16."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import (act_f32_for_oracle, assert_bf16_within_ulp, assert_f32_close, bf16_bits,
                      bf16_tensor, dev_tensor, reference)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


# ------------------------------------------------------------------ pack --
@pytest.mark.parametrize("N,K", [(1, 1), (5, 17), (128, 128), (129, 300), (640, 2560), (300, 1000),
                                 (2560, 2560), (257, 4097)])
def test_pack_bytes_bitexact(N, K):
    T = inputs.ternary(np.random.default_rng(N * 7 + K), (N, K), 0.5)
    pk = L.pack(dev_tensor(T)).cpu().numpy()
    ref = oracle.pack_tiles(T)
    assert pk.shape == ref.shape
    assert np.array_equal(pk, ref)
    assert np.array_equal(oracle.unpack_tiles(pk, N, K), T)


def test_pack_strided_source():
    T = inputs.ternary(np.random.default_rng(3), (200, 300), None)
    big = np.zeros((200, 384), dtype=np.int8)
    big[:, :300] = T
    t = dev_tensor(big)[:, :300]
    assert t.stride(0) == 384
    assert np.array_equal(L.pack(t).cpu().numpy(), oracle.pack_tiles(T))


def test_pack_rejects_non_ternary():
    T = np.zeros((3, 40), dtype=np.int8)
    T[1, 7] = 2
    T[2, 39] = -5
    with pytest.raises(L.BitmtpError) as e:
        L.pack(dev_tensor(T))
    assert e.value.status == L.ERR_NOT_TERNARY


# ------------------------------------------------------------- quant_act --
def _check_quant(x_np, is_bf16):
    x_dev = bf16_tensor(x_np) if is_bf16 else dev_tensor(x_np)
    q, a, r = L.quant_act(x_dev)
    q_ref, a_ref, r_ref = oracle.quant_act(act_f32_for_oracle(x_np, is_bf16))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(a.cpu().numpy(), a_ref)
    assert np.array_equal(r.cpu().numpy(), r_ref)


@pytest.mark.parametrize("M,K", [(1, 1), (3, 17), (16, 2560), (5, 6912), (2, 11008), (16, 300),
                                 (3, 32768), (1, 32767)])
@pytest.mark.parametrize("is_bf16", [False, True])
def test_quant_act_bitexact(M, K, is_bf16):
    rng = np.random.default_rng(M * 1000 + K)
    x = rng.standard_normal((M, K), dtype=np.float32)
    x[rng.random((M, K)) < 0.01] *= np.float32(20)
    if M > 2:
        x[1] = 0.0                       # all-zero row
        x[2] = 0.0
        x[2, K // 2] = -3.75             # one-hot row
    _check_quant(inputs.to_bf16_bits(x) if is_bf16 else x, is_bf16)


def test_quant_act_golden_rows():
    rows = [[127, 2.5, -3.5, 0.5, 1.5], [1, 0.5, -0.25, 2 ** -8, 0], [3, -3, 1, 0, 0]]
    _check_quant(np.array(rows, dtype=np.float32), False)


# ------------------------------------------------------------------ gemm --
def run_gemm(T, w_scale, x_np, x_kind, out_dtype, flags=0, M=None, pk=None):
    N, K = T.shape
    if pk is None:
        pk = L.pack(dev_tensor(T))
    if x_kind == "bf16":
        x = bf16_tensor(x_np)
    else:
        x = dev_tensor(x_np)
    a_scale = None
    if x_kind == "q8":
        x, a_scale = x, None
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    y, acc = L.gemm(pk, w_scale, N, K, x, a_scale=a_scale, out_dtype=tdt, acc=True, flags=flags)
    return y, acc


def check_gemm(T, w_scale, x_np, is_bf16, out_dtype, flags=0, pk=None):
    y, acc = run_gemm(T, w_scale, x_np, "bf16" if is_bf16 else "f32", out_dtype, flags, pk=pk)
    y_ref, acc_ref, _, _ = reference(T, w_scale, x_np, is_bf16)
    acc_np = acc.cpu().numpy()
    assert np.array_equal(acc_np, acc_ref.astype(np.int32)), _first_diff(acc_np, acc_ref)
    if out_dtype == "f32":
        assert_f32_close(y.cpu().numpy(), y_ref, acc_ref)
    else:
        assert_bf16_within_ulp(bf16_bits(y), y_ref)


def _first_diff(a, b):
    d = np.argwhere(a != b)
    if not len(d):
        return ""
    i = tuple(d[0])
    return f"first acc mismatch at {i}: got {a[i]} ref {b[i]} ({len(d)} of {a.size})"


PATHS = {"tc": L.FLAG_FORCE_TC, "dp": L.FLAG_FORCE_DP, "auto": 0}
SHAPES = [(1, 1), (7, 5), (130, 129), (300, 1000), (640, 2560), (257, 2049), (1000, 3000)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("path", ["tc", "dp"])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_gemm_small_widths(N, K, path, M):
    T, w, x = inputs.random_problem(N + K + M, M, N, K, p_zero=0.4)
    check_gemm(T, w, x, False, "f32", PATHS[path])


@pytest.mark.parametrize("N,K", [(130, 129), (640, 2560), (1000, 3000), (2560, 6912)])
@pytest.mark.parametrize("M", list(range(5, 17)))
def test_gemm_tensor_path_widths(N, K, M):
    T, w, x = inputs.random_problem(10 * M + N + K, M, N, K, outliers=True)
    check_gemm(T, w, x, False, "f32", PATHS["tc"])


@pytest.mark.parametrize("K", [128, 256, 384])
@pytest.mark.parametrize("M", [8, 16])
def test_tensor_path_many_short_segments(K, M):
    """One to three k tiles per row tile and several row tiles per CTA: every
    CTA runs a run of short segments, most of them a single MMA batch, so the
    two MMA-issuing warps take turns segment by segment and one of them passes
    whole segments without issuing.  Exact accumulators against the oracle."""
    N = 128 * 700 + 37
    T, w, x = inputs.random_problem(7000 + K + M, M, N, K, p_zero=0.3, outliers=True)
    check_gemm(T, w, x, False, "f32", PATHS["tc"])


@pytest.mark.parametrize("path", ["tc", "dp"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_gemm_bf16_activations(path, out_dtype):
    M = 4 if path == "dp" else 11
    T, w, xb = inputs.random_problem(99, M, 900, 2600, p_zero=0.5, x_kind="bf16", outliers=True)
    check_gemm(T, w, xb, True, out_dtype, PATHS[path])


@pytest.mark.parametrize("path", ["tc", "dp"])
def test_gemm_q8_matches_raw(path):
    M = 3
    T, w, x = inputs.random_problem(5, M, 700, 1500)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    q, a, _ = L.quant_act(xd)
    y8, acc8 = L.gemm(pk, w, 700, 1500, q, a_scale=a, acc=True, flags=PATHS[path])
    yr, accr = L.gemm(pk, w, 700, 1500, xd, acc=True, flags=PATHS[path])
    assert torch.equal(acc8, accr) and torch.equal(y8, yr)
    y_ref, acc_ref, _, _ = reference(T, w, x, False)
    assert np.array_equal(acc8.cpu().numpy(), acc_ref)


def test_width_consistency():
    """Rows computed in a block of 16 equal the same rows computed alone."""
    T, w, x = inputs.random_problem(21, 16, 1100, 2300, outliers=True)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    y16, a16 = L.gemm(pk, w, 1100, 2300, xd, acc=True)
    for m in range(16):
        y1, a1 = L.gemm(pk, w, 1100, 2300, xd[m:m + 1], acc=True)
        assert torch.equal(a1[0], a16[m]) and torch.equal(y1[0], y16[m])
    for M in (2, 3, 5, 8, 13):
        yM, aM = L.gemm(pk, w, 1100, 2300, xd[:M], acc=True)
        assert torch.equal(aM, a16[:M]) and torch.equal(yM, y16[:M])


def test_strided_operands():
    M, N, K = 6, 500, 1000
    T, w, x = inputs.random_problem(31, M, N, K)
    pk = L.pack(dev_tensor(T))
    xbig = torch.zeros((M, 1040), dtype=torch.float32, device="cuda")
    xbig[:, :K] = dev_tensor(x)
    ybig = torch.full((M, 520), -7.0, dtype=torch.float32, device="cuda")
    abig = torch.full((M, 515), -7, dtype=torch.int32, device="cuda")
    L.gemm(pk, w, N, K, xbig[:, :K], y=ybig[:, :N], acc=abig[:, :N])
    y_ref, acc_ref, _, _ = reference(T, w, x, False)
    assert np.array_equal(abig[:, :N].cpu().numpy(), acc_ref)
    assert_f32_close(ybig[:, :N].cpu().numpy(), y_ref, acc_ref)
    assert torch.all(ybig[:, N:] == -7.0) and torch.all(abig[:, N:] == -7)


def test_degenerate_cases():
    N, K = 300, 700
    rng = np.random.default_rng(41)
    # all-zero weights -> exact zeros
    T0 = np.zeros((N, K), dtype=np.int8)
    x = rng.standard_normal((5, K), dtype=np.float32)
    check_gemm(T0, np.float32(0.03), x, False, "f32")
    # zero activation rows -> exact zeros in those rows
    T, w, x = inputs.random_problem(42, 5, N, K)
    x[0] = 0
    x[3] = 0
    check_gemm(T, w, x, False, "f32")
    # identity weights: acc == q
    Ti = np.eye(256, dtype=np.int8)
    xi = rng.standard_normal((9, 256), dtype=np.float32)
    y, acc = run_gemm(Ti, np.float32(1.0), xi, "f32", "f32")
    q_ref, _, _ = oracle.quant_act(xi)
    assert np.array_equal(acc.cpu().numpy(), q_ref.astype(np.int32))
    # all +1 weights and constant positive rows: acc == 127 * K exactly
    K2 = 11008
    T1 = np.ones((128, K2), dtype=np.int8)
    xc = np.full((16, K2), 0.37, dtype=np.float32)
    y, acc = run_gemm(T1, np.float32(0.02), xc, "f32", "f32", L.FLAG_FORCE_TC)
    assert torch.all(acc == 127 * K2)
    # empty block is a no-op
    pk = L.pack(dev_tensor(T))
    yz = torch.full((0, N), 1.0, device="cuda")
    L.gemm(pk, w, N, K, torch.zeros((0, K), device="cuda"), y=yz)


@pytest.mark.parametrize("K", [32768, 32767])
@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_gemm_max_in_features(K, M):
    """The largest in-feature count the library accepts (one dp4a width and the
    three tensor widths): 256 k-tiles per row, the last one ragged for K=32767."""
    T, w, x = inputs.random_problem(7000 + 10 * M + K % 2, M, 130, K, outliers=True)
    check_gemm(T, w, x, False, "f32")


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_gemm_max_in_features_extreme_sums(M):
    """All +1 (then all -1) weights against constant rows at the maximum K: every
    activation code is 127 and acc = +-127 * 32768, the largest magnitude a
    call can produce."""
    K = 32768
    xc = np.full((M, K), -0.61, dtype=np.float32)
    for sign in (1, -1):
        T = np.full((130, K), sign, dtype=np.int8)
        y, acc = run_gemm(T, np.float32(0.02), xc, "f32", "f32")
        assert torch.all(acc == -sign * 127 * K)


def test_pdl_flag_same_result():
    T, w, x = inputs.random_problem(51, 8, 2560, 2560)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    y0, a0 = L.gemm(pk, w, 2560, 2560, xd, acc=True)
    ys = [L.gemm(pk, w, 2560, 2560, xd, acc=True, flags=L.FLAG_PDL) for _ in range(4)]
    torch.cuda.synchronize()
    for y1, a1 in ys:
        assert torch.equal(a0, a1) and torch.equal(y0, y1)


def test_grouped_launch_two_roles():
    """Verify rows through one projection and draft rows through another, one launch."""
    rng = np.random.default_rng(61)
    x = rng.standard_normal((16, 1200), dtype=np.float32)
    Tv, wv = inputs.ternary(rng, (3000, 1200), 0.5), np.float32(0.021)
    Td, wd = inputs.ternary(rng, (700, 1200), 0.2), np.float32(0.037)
    xd = dev_tensor(x)
    q, a, _ = L.quant_act(xd)
    pv, pd = L.pack(dev_tensor(Tv)), L.pack(dev_tensor(Td))
    yv = torch.empty((4, 3000), device="cuda")
    ydd = torch.empty((12, 700), device="cuda", dtype=torch.bfloat16)
    av = torch.empty((4, 3000), device="cuda", dtype=torch.int32)
    ad = torch.empty((12, 700), device="cuda", dtype=torch.int32)
    L.gemm_grouped([
        dict(pk=pv, w_scale=wv, N=3000, K=1200, x=q[:4], a_scale=a[:4], y=yv, acc=av),
        dict(pk=pd, w_scale=wd, N=700, K=1200, x=q[4:], a_scale=a[4:], y=ydd, acc=ad),
    ])
    yv_ref, accv, _, _ = reference(Tv, wv, x[:4], False)
    yd_ref, accd, _, _ = reference(Td, wd, x[4:], False)
    assert np.array_equal(av.cpu().numpy(), accv)
    assert np.array_equal(ad.cpu().numpy(), accd)
    assert_f32_close(yv.cpu().numpy(), yv_ref, accv)
    assert_bf16_within_ulp(bf16_bits(ydd), yd_ref)


def test_workspace_reuse_across_shapes():
    """One workspace, zero-filled once, shared by alternating shapes (whose
    activation sections overlap each other's) gives exact results every time."""
    probs = [inputs.random_problem(71, 8, 2560, 6912), inputs.random_problem(72, 3, 11008, 4096),
             inputs.random_problem(73, 1, 640, 2560)]
    packed = [L.pack(dev_tensor(T)) for T, _, _ in probs]
    nb = max(L.bitmtp_linear_workspace_bytes(T.shape[0], T.shape[1], x.shape[0]) for T, _, x in probs)
    ws = torch.zeros((nb,), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for (T, w, x), pk in zip(probs, packed):
            N, K = T.shape
            y, acc = L.gemm(pk, w, N, K, dev_tensor(x), acc=True, flags=L.FLAG_PDL, workspace_tensor=ws)
            y_ref, acc_ref, _, _ = reference(T, w, x, False)
            assert np.array_equal(acc.cpu().numpy(), acc_ref), (rep, N, K)
            assert_f32_close(y.cpu().numpy(), y_ref, acc_ref)
    assert L.bitmtp_linear_device_error() == 0


@pytest.mark.parametrize("M", [1, 8, 16])
def test_workspace_flags_left_zero(M):
    """Row tiles split between CTAs hand their partial sums over through the
    workspace slots and ready flags; every launch must leave the flags at zero
    for the next one (the slots need no clearing)."""
    N, K = 2560, 6912
    T, w, x = inputs.random_problem(81 + M, M, N, K)
    pk = L.pack(dev_tensor(T))
    nb = L.bitmtp_linear_workspace_bytes(N, K, M)
    ws = torch.zeros((nb,), dtype=torch.uint8, device="cuda")
    y, acc = L.gemm(pk, w, N, K, dev_tensor(x), acc=True, workspace_tensor=ws)
    torch.cuda.synchronize()
    flags_end = 256 + (320 * 4 + 255) // 256 * 256
    slots_end = flags_end + 320 * 16 * 128 * 4
    assert int(torch.count_nonzero(ws[:flags_end])) == 0
    assert int(torch.count_nonzero(ws[flags_end:slots_end])) > 0  # some row tiles were split
    _, acc_ref, _, _ = reference(T, w, x, False)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
