"""FP8 "fast" draft projections (BITMTP_FLAG_FP8) against the oracle.

The activations are quantised per row to E4M3 and multiplied with the ternary
weights on the tensor cores, accumulating in fp32.  What is compared:

* bit for bit, where the arithmetic leaves no freedom:
  - T = identity: each accumulator is one product T * e = e, so the fp32
    accumulators returned in ``acc`` are exactly the oracle's E4M3 values --
    the quantiser (scale, rounding, saturation, zero rows) checked bit for bit;
  - activations whose E4M3 values are multiples of 32 in [256, 448] (and
    amax = 448, so s = 1): every partial sum (of (T+1)*e and -e) is a multiple
    of 32 below 2^24 * 32, exact in fp32 whatever the order, so acc and y equal
    the oracle exactly;
* otherwise within the bound the header states for the fp32 accumulation,
  which adds sum_k (T+1)*e and -sum_k e (2 * ceil(K/32) MMAs of 32 products):
  |acc - sum_k T*e| <= (2 * ceil(K/32) + 2) * 2^-23 * sum_k (T+2)*|e|, and y
  within that bound times a_scale * w_scale plus the dequant roundings (two
  fp32 roundings, then the bf16 rounding for bf16 output)."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_fp8_within_bound, bf16_bits, bf16_tensor, dev_tensor, fp8_reference

pytestmark = pytest.mark.gpu

WAIT_CODES = set(range(0x101, 0x109))


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


def _x_dev(x, is_bf16):
    return bf16_tensor(x) if is_bf16 else dev_tensor(x)


def _run(T, w, x, is_bf16, out=torch.float32, flags=0, amax=None, ws=None):
    N, K = T.shape
    pk = L.pack(dev_tensor(T))
    xd = _x_dev(x, is_bf16)
    M = xd.shape[0]
    y = torch.empty((M, N), dtype=out, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    nb = L.bitmtp_linear_workspace_bytes(N, K, max(M, 1))
    if ws is None:
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    st = L.bitmtp_linear_gemm(L._ptr(pk), float(w), N, K, M, L.make_act(xd, None, amax), L.make_out(y, acc),
                              L._ptr(ws), ws.numel(), flags | L.FLAG_FP8, L._stream(None))
    assert st == L.OK, L.status_string(st)
    torch.cuda.synchronize()
    yh = bf16_bits(y) if out == torch.bfloat16 else y.cpu().numpy()
    return yh, acc.view(torch.float32).cpu().numpy()


def _oracle(T, w, x, is_bf16):
    return fp8_reference(T, w, x, is_bf16)


def _check_within_bound(K, w, y, acc, ref, out):
    return assert_fp8_within_bound(K, w, y, acc, ref, out == torch.bfloat16)


# ---------------------------------------------------------------------------
# Bit-exact cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K,is_bf16", [(1, 128, False), (7, 300, True), (16, 2560, False), (16, 2560, True),
                                         (3, 6912, True)])
def test_fp8_codes_exact_through_identity(M, K, is_bf16):
    rng = np.random.default_rng(900 + M + K)
    x = rng.standard_normal((M, K), dtype=np.float32)
    x[rng.random((M, K)) < 0.01] *= np.float32(20)
    x[rng.random((M, K)) < 0.05] *= np.float32(1e-4)  # values rounding to E4M3 subnormals and zero
    if M > 2:
        x[1] = 0.0                                   # zero row: e = 0, a_scale = 0
        x[2] = 0.0
        x[2, K // 2] = np.float32(-3.5)              # one-hot row: -448 there
    xin = inputs.to_bf16_bits(x) if is_bf16 else x
    T = np.eye(K, dtype=np.int8)
    w = np.float32(0.03125)
    y, acc = _run(T, w, xin, is_bf16)
    _, acc_ref, e, a_scale, _ = _oracle(T, w, xin, is_bf16)
    assert np.array_equal(acc.astype(np.float64), e)
    assert np.array_equal(acc.astype(np.float64), acc_ref)
    # y = RN32(RN32(e * a_scale) * w) with w a power of two: exact products after one rounding
    y_k = (e.astype(np.float32) * a_scale[:, None]).astype(np.float32) * w
    assert np.array_equal(y, y_k.astype(np.float32))


def _binade_activations(rng, M, K):
    """E4M3 values that are multiples of 32 in [256, 448], zeros, and one 448
    per row (amax = 448, so the scale is exactly 1 and e = x)."""
    mags = np.arange(256, 449, 32, dtype=np.float32)
    x = rng.choice(mags, size=(M, K)) * rng.choice(np.array([-1, 1], np.float32), size=(M, K))
    x[rng.random((M, K)) < 0.3] = 0.0
    x[np.arange(M), rng.integers(0, K, size=M)] = np.float32(448)
    return x.astype(np.float32)


@pytest.mark.parametrize("M,N,K,is_bf16,out", [
    (1, 2560, 2560, False, torch.float32),
    (3, 1000, 300, True, torch.float32),
    (8, 2560, 6912, True, torch.bfloat16),
    (16, 6912, 2560, False, torch.float32),
    (16, 384, 32768, True, torch.float32),      # the largest K: partial sums < 3 * 448 * 2^15 < 2^24 * 32
    (12, 130, 4100, False, torch.bfloat16),     # ragged N and K tails
])
def test_fp8_exact_binade_sums(M, N, K, is_bf16, out):
    rng = np.random.default_rng(7000 + M * 31 + K)
    x = _binade_activations(rng, M, K)
    xin = inputs.to_bf16_bits(x) if is_bf16 else x
    T = inputs.ternary(rng, (N, K), 0.5)
    w = np.float32(0.0234375)
    y, acc = _run(T, w, xin, is_bf16, out)
    y_ref, acc_ref, e, a_scale, _ = _oracle(T, w, xin, is_bf16)
    assert np.array_equal(e, x.astype(np.float64)) and np.all(a_scale == 1)
    assert np.array_equal(acc.astype(np.float64), acc_ref)
    if out == torch.bfloat16:
        assert np.array_equal(y, oracle.f32_to_bf16_bits(y_ref))
    else:
        assert np.array_equal(y, y_ref)


# ---------------------------------------------------------------------------
# Random data: within the fp32 accumulation bound
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K,p0,is_bf16,out", [
    (1, 2560, 2560, 0.5, True, torch.bfloat16),
    (2, 640, 2560, None, False, torch.float32),
    (4, 2560, 6912, 0.5, True, torch.bfloat16),
    (5, 1000, 300, None, False, torch.float32),
    (8, 6912, 2560, 0.5, True, torch.float32),
    (12, 2560, 2560, 0.2, False, torch.bfloat16),
    (16, 2560, 6912, 0.8, True, torch.bfloat16),
    (16, 256, 32768, None, False, torch.float32),
    (16, 129, 129, None, False, torch.float32),
])
def test_fp8_random_within_accumulation_bound(M, N, K, p0, is_bf16, out):
    T, w, x = inputs.random_problem(3100 + M * 7 + K, M, N, K, p_zero=p0, x_kind="bf16" if is_bf16 else "f32",
                                    outliers=True)
    y, acc = _run(T, w, x, is_bf16, out)
    ratio = _check_within_bound(K, w, y, acc, _oracle(T, w, x, is_bf16), out)
    print(f"max |acc error| / bound = {ratio:.3g}")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_fp8_grouped_layer_set(M):
    probs, refs = [], []
    for p in range(len(inputs.BITNET2B_PROJ)):
        _, K, N = inputs.BITNET2B_PROJ[p]
        T, w = inputs.bitnet2b_weights(p)
        x = inputs.bitnet2b_act(p, M)
        probs.append(dict(pk=L.pack(dev_tensor(T)), w_scale=float(w), N=N, K=K, x=bf16_tensor(x),
                          y=torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                          acc=torch.empty((M, N), dtype=torch.int32, device="cuda")))
        refs.append((T, w, x, K))
    L.gemm_grouped(probs, flags=L.FLAG_FP8 | L.FLAG_PDL)
    torch.cuda.synchronize()
    for pr, (T, w, x, K) in zip(probs, refs):
        _check_within_bound(K, w, bf16_bits(pr["y"]), pr["acc"].view(torch.float32).cpu().numpy(),
                            _oracle(T, w, x, True), torch.bfloat16)


def test_fp8_amax_handoff_gives_the_same_codes():
    """A layer chain hands the rows' absmax to the next call: the FP8
    quantiser then skips its absmax pass and must give the same values."""
    M, K = 9, 2560
    rng = np.random.default_rng(77)
    x = inputs.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    T = np.eye(K, dtype=np.int8)
    amax = torch.from_numpy(np.max(np.abs(oracle.bf16_bits_to_f32(x)), axis=1).astype(np.float32)).cuda()
    _, acc_a = _run(T, np.float32(1), x, True, amax=amax)
    _, acc_b = _run(T, np.float32(1), x, True)
    _, _, e, _, _ = _oracle(T, np.float32(1), x, True)
    assert np.array_equal(acc_a.astype(np.float64), e)
    assert np.array_equal(acc_a, acc_b)


def test_fp8_withheld_chunk_times_out_then_next_call_is_exact():
    M, N, K = 8, 2560, 6912
    rng = np.random.default_rng(4242)
    x = _binade_activations(rng, M, K)
    T = inputs.ternary(rng, (N, K), 0.5)
    nb = L.bitmtp_linear_workspace_bytes(N, K, M)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = L.bitmtp_linear_gemm(L._ptr(pk), 0.5, N, K, M, L.make_act(xd), L.make_out(y), L._ptr(ws), nb,
                              L.FLAG_FP8 | L.FLAG_TEST_WITHHOLD, L._stream(None))
    assert st == L.OK
    assert L.bitmtp_linear_device_error() in WAIT_CODES
    assert L.bitmtp_linear_device_error() == 0
    ws.zero_()
    _, acc = _run(T, np.float32(0.5), x, False, ws=ws)
    _, acc_ref, _, _, _ = _oracle(T, np.float32(0.5), x, False)
    assert np.array_equal(acc.astype(np.float64), acc_ref)


def test_fp8_through_the_noalloc_entry():
    """The FP8 flag through the entry point that allocates nothing: identity
    weights, so the accumulators are the E4M3 values exactly."""
    M, K = 6, 1000
    rng = np.random.default_rng(515)
    x = rng.standard_normal((M, K), dtype=np.float32)
    T = np.eye(K, dtype=np.int8)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    y = torch.empty((M, K), dtype=torch.float32, device="cuda")
    acc = torch.empty((M, K), dtype=torch.int32, device="cuda")
    st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), 1.0, K, K, M, L.make_act(xd), L.make_out(y, acc),
                                      L.FLAG_FP8, L._stream(None))
    assert st == L.OK, L.status_string(st)
    torch.cuda.synchronize()
    _, _, e, _, _ = fp8_reference(T, np.float32(1), x, False)
    assert np.array_equal(acc.view(torch.float32).cpu().numpy().astype(np.float64), e)
