"""The bounded-wait error path on the GPU, made to run without a fault.

Every wait of the GEMM kernel (on an mbarrier, or on another CTA's ready
flag) gives up after a time bound; the kernel then records a code in the
device error word, skips its remaining work, waits (bounded) for its own bulk
copies and MMAs, frees its tensor memory and exits.  BITMTP_FLAG_TEST_WITHHOLD
makes CTA 0 never request its first chunk of packed weights and lowers every
bound of the launch to 1 ms, so a consumer wait runs out on a barrier that
nothing completes.  The test checks that the host reads the wait's code from
bitmtp_linear_device_error (and that reading clears it), and that the next
normal call on the same device and workspace -- zero-filled again, as the
header asks after an error -- matches the oracle.  Both compute paths run it:
the dp4a path (no tensor memory) and the tensor path (its tensor memory must
be freed for the next launch to allocate)."""
import numpy as np
import pytest
import torch

from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_f32_close, dev_tensor, reference

pytestmark = pytest.mark.gpu

# the kernel's wait codes (weights, activation tiles, A full, A empty, D,
# ring slot, contributor flag, contributor slot)
WAIT_CODES = set(range(0x101, 0x109))


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


@pytest.mark.parametrize("M,flags", [(4, L.FLAG_FORCE_DP), (8, L.FLAG_FORCE_TC)])
def test_withheld_chunk_times_out_then_next_call_is_exact(M, flags):
    N, K = 2560, 6912
    T, w, x = inputs.random_problem(1234 + M, M, N, K, p_zero=0.5, outliers=True)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    nb = L.bitmtp_linear_workspace_bytes(N, K, M)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    assert L.bitmtp_linear_device_error() == 0

    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = L.bitmtp_linear_gemm(L._ptr(pk), float(w), N, K, M, L.make_act(xd), L.make_out(y),
                              L._ptr(ws), nb, flags | L.FLAG_TEST_WITHHOLD, L._stream(None))
    assert st == L.OK, L.status_string(st)
    code = L.bitmtp_linear_device_error()  # synchronises the stream
    assert code in WAIT_CODES, hex(code)
    assert L.bitmtp_linear_device_error() == 0  # read and cleared

    # the same device, workspace (zero-filled again) and path work exactly
    ws.zero_()
    for _ in range(2):
        y2, acc2 = L.gemm(pk, w, N, K, xd, acc=True, flags=flags, workspace_tensor=ws)
        y_ref, acc_ref, _, _ = reference(T, w, x, False)
        assert np.array_equal(acc2.cpu().numpy(), acc_ref)
        assert_f32_close(y2.cpu().numpy(), y_ref, acc_ref)
    assert L.bitmtp_linear_device_error() == 0


def test_noalloc_recovers_after_reported_error():
    """After an error has been reported, the next no-alloc call clears its
    built-in flags itself and is exact."""
    M, N, K = 8, 2560, 2560
    T, w, x = inputs.random_problem(4321, M, N, K, p_zero=0.5)
    pk = L.pack(dev_tensor(T))
    xd = dev_tensor(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), float(w), N, K, M, L.make_act(xd), L.make_out(y),
                                      L.FLAG_TEST_WITHHOLD, L._stream(None))
    assert st == L.OK
    assert L.bitmtp_linear_device_error() in WAIT_CODES
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    for _ in range(2):
        st = L.bitmtp_linear_gemm_noalloc(L._ptr(pk), float(w), N, K, M, L.make_act(xd), L.make_out(y, acc),
                                          0, L._stream(None))
        assert st == L.OK
        _, acc_ref, _, _ = reference(T, w, x, False)
        assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert L.bitmtp_linear_device_error() == 0
