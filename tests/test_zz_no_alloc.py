"""GPU test of bitmtp_linear_gemm_noalloc, the entry point for callers that may
not allocate device memory (code inside another runtime's launch hook, loops
that cannot afford cudaMalloc's stalls, processes whose memory belongs to an
allocator they cannot reach).  It runs the same GEMM kernel as
bitmtp_linear_gemm but keeps its split-row-tile counters and partial sums in
the library's own static device array instead of a caller workspace.

Each case calls the new entry point twice in a row through the C ABI and
compares both results with bitmtp_linear_gemm on the same inputs: int32
accumulators bit-exact, fp32 outputs within 1e-5 relative, bf16 outputs within
one bf16 ulp.  The file is named to be collected last, and it needs nothing
from earlier tests: its first call also performs the per-device set-up."""
import numpy as np
import pytest
import torch

from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_f32_close, bf16_bits, bf16_tensor, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


# (N, K, M, activation kind, output dtype, with int32 accumulators):
# 16 rows on the 16-row tensor tile with row tiles split between CTAs,
# 5 rows on the 8-row tensor tile, 1 row on the dp4a path, 16 rows at the
# maximum in-feature count.
CASES = [
    (2560, 6912, 16, "bf16", torch.float32, True),
    (2560, 2560, 5, "f32", torch.bfloat16, False),
    (640, 2560, 1, "bf16", torch.float32, True),
    (1000, 3000, 9, "f32", torch.float32, True),
    (130, 32768, 16, "f32", torch.float32, True),  # the largest K the array holds
]


def _setup(case, seed):
    N, K, M, xk, out_dtype, want_acc = case
    T, w, x = inputs.random_problem(seed, M, N, K, p_zero=0.5, x_kind=xk, outliers=True)
    pk = L.pack(dev_tensor(T))
    xd = bf16_tensor(x) if xk == "bf16" else dev_tensor(x)
    return pk, float(w), xd


def _outputs(case):
    N, _, M, _, out_dtype, want_acc = case
    y = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    acc = torch.full((M, N), -12345, dtype=torch.int32, device="cuda") if want_acc else None
    return y, acc


def _run_existing(case, pk, w, xd):
    N, K, M = case[:3]
    y, acc = _outputs(case)
    nb = L.bitmtp_linear_workspace_bytes(N, K, M)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    st = L.bitmtp_linear_gemm(L._ptr(pk), w, N, K, M, L.make_act(xd), L.make_out(y, acc),
                              L._ptr(ws), nb, 0, L._stream(None))
    assert st == L.OK, L.status_string(st)
    torch.cuda.synchronize()
    return y, acc


def _run_noalloc(case, pk, w, xd):
    N, K, M = case[:3]
    y, acc = _outputs(case)
    st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), w, N, K, M, L.make_act(xd), L.make_out(y, acc),
                                      0, L._stream(None))
    assert st == L.OK, L.status_string(st)
    return y, acc


def _assert_same(case, got, ref):
    y, acc = got
    y_ref, acc_ref = ref
    if acc is not None:
        assert np.array_equal(acc.cpu().numpy(), acc_ref.cpu().numpy())
    if y.dtype == torch.float32:
        assert_f32_close(y.cpu().numpy(), y_ref.cpu().numpy())
    else:
        g = bf16_bits(y).astype(np.int32)
        r = bf16_bits(y_ref).astype(np.int32)
        g = np.where(g & 0x8000, 0x8000 - g, g)
        r = np.where(r & 0x8000, 0x8000 - r, r)
        assert np.abs(g - r).max() <= 1


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_noalloc_matches_workspace_entry_twice(ci):
    case = CASES[ci]
    pk, w, xd = _setup(case, 900 + ci)
    ref = _run_existing(case, pk, w, xd)
    first = _run_noalloc(case, pk, w, xd)
    second = _run_noalloc(case, pk, w, xd)
    torch.cuda.synchronize()
    _assert_same(case, first, ref)
    _assert_same(case, second, ref)
    assert L.bitmtp_linear_device_error() == 0


def test_noalloc_alternating_shapes():
    """Calls of different shapes back to back on one stream share the array;
    each still matches the workspace entry point."""
    probs = [(CASES[i], *_setup(CASES[i], 950 + i)) for i in (0, 2, 1, 0)]
    refs = [_run_existing(c, pk, w, xd) for c, pk, w, xd in probs]
    outs = [_run_noalloc(c, pk, w, xd) for c, pk, w, xd in probs]
    torch.cuda.synchronize()
    for (c, *_), got, ref in zip(probs, outs, refs):
        _assert_same(c, got, ref)


def test_noalloc_pdl_side_stream_mixed_shapes():
    """Back-to-back calls of mixed shapes with programmatic dependent launch on
    a side stream (each call's weight prefetch overlaps the previous call)
    share the array; each matches the workspace entry point bit for bit."""
    probs = [(CASES[i], *_setup(CASES[i], 970 + i)) for i in (0, 1, 2, 3, 0, 2)]
    refs = [_run_existing(c, pk, w, xd) for c, pk, w, xd in probs]
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    with torch.cuda.stream(side):
        for c, pk, w, xd in probs:
            N, K, M = c[:3]
            y, acc = _outputs(c)
            st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), w, N, K, M, L.make_act(xd), L.make_out(y, acc),
                                              L.FLAG_PDL, L._stream(side))
            assert st == L.OK, L.status_string(st)
            outs.append((y, acc))
    side.synchronize()
    for (c, *_), (y, acc), (y_ref, acc_ref) in zip(probs, outs, refs):
        if acc is not None:
            assert torch.equal(acc, acc_ref)
        assert torch.equal(y, y_ref)
    assert L.bitmtp_linear_device_error(side) == 0


def test_noalloc_rejects_beyond_limits():
    """The shape check: a width beyond BITMTP_MAX_M is rejected before anything
    is enqueued.  (Every shape inside the library's limits fits the array, so
    its size check cannot be reached through valid shapes.)"""
    case = CASES[0]
    pk, w, xd = _setup(case, 990)
    y, acc = _outputs(case)
    st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), w, 2560, 6912, L.MAX_M + 1, L.make_act(xd),
                                      L.make_out(y, acc), 0, L._stream(None))
    assert st == L.ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.isnan(y).all()  # nothing was enqueued
