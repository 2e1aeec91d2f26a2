"""GPU parity of the device absmean ternarisation + pack
(bitmtp_linear_ternarize_pack, through the C ABI) against the oracle: the
per-tensor scale bit for bit and the packed bytes byte for byte, on normal
weights of several shapes (ragged tiles included), strided and unaligned
rows, a wide range of magnitudes with subnormals and zeros, the summation-
order case, ties, the epsilon floor and a full-size projection, which then
feeds the GEMM."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_f32_close, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


def _bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


def _check(W: np.ndarray, W_dev: torch.Tensor | None = None):
    pk, g = L.ternarize_pack(dev_tensor(W) if W_dev is None else W_dev)
    T_ref, g_ref = oracle.ternarize_absmean(W)
    assert _bits(g) == _bits(g_ref), (g, g_ref)
    assert np.array_equal(pk.cpu().numpy(), oracle.pack_tiles(T_ref))
    return pk, g, T_ref


@pytest.mark.parametrize("N,K", [(1, 1), (5, 17), (130, 129), (300, 1000), (640, 2560), (257, 4097),
                                 (3000, 300)])
def test_normal_weights(N, K):
    W = (np.random.default_rng(N * 31 + K).standard_normal((N, K)) * 0.02).astype(np.float32)
    _check(W)


def test_wide_magnitude_range_subnormals_and_zeros():
    rng = np.random.default_rng(5)
    N, K = 200, 777
    mag = np.exp2(rng.uniform(-149, 100, (N, K))).astype(np.float32)
    W = (mag * np.where(rng.random((N, K)) < 0.5, -1, 1)).astype(np.float32)
    W[rng.random((N, K)) < 0.05] = 0.0
    W[0, :5] = np.float32(1e-45)
    _check(W)


def test_fixed_scale_window_boundaries():
    """Entries at and next to the edges of the window [2^-14, 8) that the
    absmean pass sums at a fixed scale, mixed with entries outside it (tiny,
    subnormal, zero, large) and with ordinary weights, in a matrix large enough
    for many blocks and threads: the scale bit for bit."""
    rng = np.random.default_rng(77)
    N, K = 513, 1031
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    edges = np.array([2.0 ** -14, np.nextafter(np.float32(2.0 ** -14), np.float32(0)),
                      np.nextafter(np.float32(2.0 ** -14), np.float32(1)), np.nextafter(np.float32(8), np.float32(0)),
                      8.0, np.nextafter(np.float32(8), np.float32(9)), 7.99999, 1e-30, 1e-44, 0.0, 1e6, 3.0e38,
                      2.0 ** -14 + 2.0 ** -37, 0.5 + 2.0 ** -24], dtype=np.float32)
    idx = rng.integers(0, N * K, size=4000)
    W.reshape(-1)[idx] = edges[rng.integers(0, len(edges), size=idx.size)] * np.where(rng.random(idx.size) < 0.5, -1, 1)
    _check(W)


def test_summation_order_case():
    W = np.array([[2.0 ** 30, 64.0, 2.0 ** -23, 2.0 ** -23]], dtype=np.float32)
    pk, g, T = _check(W)
    assert g == 2.0 ** 28 + 32
    assert T.tolist() == [[1, 0, 0, 0]]


def test_ties_and_epsilon():
    _check(np.array([[1.0, 3.0, -1.0, -3.0]], dtype=np.float32))        # ratios +-0.5, +-1.5
    _check(np.array([[2.0, -2.0, 1.0, 3.0, -1.0, 0.0]], dtype=np.float32))
    pk, g, T = _check(np.zeros((3, 40), dtype=np.float32))
    assert g == np.float32(1e-5) and not T.any()
    _check(np.full((2, 2), 1e-7, dtype=np.float32))


def _plant_boundaries(W: np.ndarray, g: np.float32) -> np.ndarray:
    """Copy of W (all entries positive in the planting region) with entries at
    and next to the code boundaries +-g/2 and +-3g/2, placed in pairs whose
    exact sum of magnitudes is unchanged, so that mean|W| -- and g -- stay the
    same.  Partner values are chosen so that the pair sum stays exact."""
    W = W.copy()
    h = np.float32(g * np.float32(0.5))
    up, dn = np.float32(np.inf), np.float32(0.0)
    targets = [h, np.nextafter(h, up), np.nextafter(h, dn), np.float32(3 * h),
               np.nextafter(np.float32(3 * h), up), np.nextafter(np.float32(3 * h), dn)]
    flat = W.reshape(-1)
    i = 0
    placed = 0
    for t in targets:
        for sign in (1, -1):
            while True:
                a, b = flat[i], flat[i + 1]
                i += 2
                tot = np.float64(abs(a)) + np.float64(abs(b))
                rest = np.float32(tot - np.float64(t))
                if rest > 0 and np.float64(rest) + np.float64(t) == tot:
                    flat[i - 2] = np.float32(sign * t)
                    flat[i - 1] = np.float32(np.sign(b) * rest) if b != 0 else rest
                    placed += 1
                    break
    assert placed == 2 * len(targets)
    return W


def test_code_boundaries_exact():
    """Weights exactly at +-g/2 (code 0), one ulp beyond (code +-1), one ulp
    inside (code 0), and the same around +-3g/2 (code +-1): the packed codes
    match the oracle's division and round-half-even byte for byte."""
    W0 = (np.abs(np.random.default_rng(91).standard_normal((256, 512))) * 0.02 + 0.001).astype(np.float32)
    _, g = oracle.ternarize_absmean(W0)
    W = _plant_boundaries(W0, g)
    T, g2 = oracle.ternarize_absmean(W)
    assert _bits(g2) == _bits(g)
    h = np.float32(g * np.float32(0.5))
    assert (W == h).sum() == 1 and (W == -h).sum() == 1  # the boundaries are really there
    assert T[W == h].tolist() == [0] and T[W == np.nextafter(h, np.float32(np.inf))].tolist() == [1]
    _check(W)


def test_grouped_matches_oracle_per_matrix():
    """One grouped call over matrices of different shapes and layouts (flat,
    strided, unaligned rows, ragged tiles) gives every matrix's oracle scale and
    packing."""
    rng = np.random.default_rng(31)
    shapes = [(640, 2560), (130, 129), (300, 1000), (257, 4097), (1, 1), (64, 128), (1000, 300)]
    Ws, devs = [], []
    for i, (N, K) in enumerate(shapes):
        W = (rng.standard_normal((N, K)) * (0.01 + 0.01 * i)).astype(np.float32)
        Ws.append(W)
        if i == 2:  # strided rows, 16-byte aligned
            big = dev_tensor(np.zeros((N, K + 4), dtype=np.float32))
            big[:, :K] = dev_tensor(W)
            devs.append(big[:, :K])
        elif i == 3:  # odd row pitch
            big = dev_tensor(np.zeros((N, K + 1), dtype=np.float32))
            big[:, :K] = dev_tensor(W)
            devs.append(big[:, :K])
        else:
            devs.append(dev_tensor(W))
    out = L.ternarize_pack_grouped(devs)
    for W, (pk, g) in zip(Ws, out):
        T_ref, g_ref = oracle.ternarize_absmean(W)
        assert _bits(g) == _bits(g_ref)
        assert np.array_equal(pk.cpu().numpy(), oracle.pack_tiles(T_ref))


def test_grouped_non_finite_in_one_matrix():
    """A NaN in one matrix of the group is reported; the other matrices are
    still packed exactly."""
    rng = np.random.default_rng(32)
    Ws = [(rng.standard_normal((200, 333)) * 0.02).astype(np.float32) for _ in range(3)]
    Ws[1][17, 5] = np.nan
    devs = [dev_tensor(W) for W in Ws]
    N, K = Ws[0].shape
    nb = L.packed_bytes(N, K)
    outs = [(torch.empty(nb, dtype=torch.uint8, device="cuda"), torch.empty(1, dtype=torch.float32, device="cuda"))
            for _ in Ws]
    descs = [L.TernDesc(L._ptr(W), N, K, K, L._ptr(pk), nb, L._ptr(g)) for W, (pk, g) in zip(devs, outs)]
    wb = L.bitmtp_linear_ternarize_workspace_bytes_grouped(3)
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    st = L.bitmtp_linear_ternarize_pack_grouped((L.TernDesc * 3)(*descs), 3, L._ptr(ws), wb, L._stream(None))
    assert st == L.ERR_NOT_FINITE
    for i in (0, 2):
        T_ref, g_ref = oracle.ternarize_absmean(Ws[i])
        assert _bits(outs[i][1].item()) == _bits(g_ref)
        assert np.array_equal(outs[i][0].cpu().numpy(), oracle.pack_tiles(T_ref))


def test_strided_and_unaligned_rows():
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((150, 300)) * 0.05).astype(np.float32)
    for pad in (4, 1):  # 16-byte aligned rows (vector loads), then odd row pitch
        big = np.zeros((150, 300 + pad), dtype=np.float32)
        big[:, :300] = W
        t = dev_tensor(big)[:, :300]
        assert t.stride(0) == 300 + pad
        _check(W, t)


def test_non_finite_rejected():
    W = np.ones((4, 40), dtype=np.float32)
    for bad in (np.nan, np.inf, -np.inf):
        W[2, 7] = bad
        with pytest.raises(L.BitmtpError) as e:
            L.ternarize_pack(dev_tensor(W))
        assert e.value.status == L.ERR_NOT_FINITE


def test_full_size_projection_then_gemm():
    """The gate projection of the BitNet-2B layer set (2560 -> 6912) from fp32
    weights, then a width-8 linear on the result against the oracle."""
    _, K, N = inputs.BITNET2B_PROJ[4]
    W = (np.random.default_rng(77).standard_normal((N, K)) * 0.02).astype(np.float32)
    pk, g, T = _check(W)
    x = np.random.default_rng(78).standard_normal((8, K)).astype(np.float32)
    y, acc = L.gemm(pk, g, N, K, dev_tensor(x), acc=True)
    y_ref, acc_ref, _, _, _ = oracle.w2a8_linear(T, np.float32(g), x, "f32")
    assert np.array_equal(acc.cpu().numpy(), acc_ref.astype(np.int32))
    assert_f32_close(y.cpu().numpy(), y_ref, acc_ref)
