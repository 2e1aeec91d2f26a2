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
be freed for the next launch to allocate), and so does the dp4a path's
one-launch layer-chain mode (quantising warps, the output-absmax zeroing word
and its reset)."""
import numpy as np
import pytest
import torch

from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
import oracle
from gpu_util import assert_f32_close, bf16_tensor, dev_tensor, reference

pytestmark = pytest.mark.gpu

# the kernel's wait codes (weights, activation tiles, A full, A empty, D,
# ring slot, contributor flag, contributor slot, the one-launch mode's zeroed
# output absmax)
WAIT_CODES = set(range(0x101, 0x10A))


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


def test_one_launch_chain_call_times_out_then_next_call_is_exact():
    """The one-launch mode (rows' absmax handed over, width 4) on a call with
    eleven ring chunks per CTA, so warp 5 quantises too, and an output absmax,
    so the zeroing word is in play: the withheld chunk ends the launch with a
    wait code, and after the workspace is zero-filled again the same call is
    exact, twice (the second time on the word the first one reset)."""
    M, N, K = 4, 32000, 6912
    rng = np.random.default_rng(2468)
    T = inputs.ternary(rng, (N, K), 0.5)
    x = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    amax_in = dev_tensor(np.max(np.abs(oracle.bf16_bits_to_f32(x)), axis=1).astype(np.float32))
    pk = L.pack(dev_tensor(T))
    xd = bf16_tensor(x)
    nb = L.bitmtp_linear_workspace_bytes(N, K, M)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    amax_out = torch.empty(M, dtype=torch.float32, device="cuda")
    act, out = L.make_act(xd, amax=amax_in), L.make_out(y, acc, amax=amax_out)
    st = L.bitmtp_linear_gemm(L._ptr(pk), 0.03, N, K, M, act, out, L._ptr(ws), nb,
                              L.FLAG_PDL | L.FLAG_TEST_WITHHOLD, L._stream(None))
    assert st == L.OK, L.status_string(st)
    code = L.bitmtp_linear_device_error()
    assert code in WAIT_CODES, hex(code)
    assert L.bitmtp_linear_device_error() == 0

    ws.zero_()
    q, _, _ = oracle.quant_act_bf16(x)
    acc_ref = oracle.gemm_acc(T, q)
    for _ in range(2):
        st = L.bitmtp_linear_gemm(L._ptr(pk), 0.03, N, K, M, act, out, L._ptr(ws), nb, L.FLAG_PDL,
                                  L._stream(None))
        assert st == L.OK
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), acc_ref.astype(np.int32))
        assert int(ws[:1536].abs().sum()) == 0
    assert L.bitmtp_linear_device_error() == 0
