"""GPU parity of the layer-chained step: each linear's output is the next
linear's input, its epilogues reduce the output rows' absmax (first phase)
and the next call's preparation takes it instead of its own absmax pass
(second phase).  Every layer's stored output, accumulators and row absmax
are compared with the oracle's chain (``linear_chain``, which takes the
dequant in the kernel's fixed order) bit for bit, and the same chain without
the handed-over absmax gives the same bits."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import bf16_bits, dev_tensor

pytestmark = pytest.mark.gpu

SHAPES = [(1024, 1024), (1024, 2048), (2048, 1024), (1024, 1024)]  # (K, N) per layer


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


def _layers(seed):
    out = []
    for i, (K, N) in enumerate(SHAPES):
        T, w, _ = inputs.random_problem(seed + i, 1, N, K, p_zero=0.4)
        out.append((T, w))
    return out


def _run_chain(layers, x0, out_dtype, handoff, flags):
    """The chain through the C ABI; returns per layer (y, acc, amax) tensors."""
    M = x0.shape[0]
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    ws = L.workspace(L.bitmtp_linear_workspace_bytes(max(N for _, N in SHAPES), max(K for K, _ in SHAPES), M),
                     x0.device)
    pks = [L.pack(dev_tensor(T)) for T, _ in layers]  # packed first: the calls then run back to back
    x, x_amax = x0, None
    res = []
    for (T, w), (K, N), pk in zip(layers, SHAPES, pks):
        y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        amax = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
        act = L.make_act(x, amax=x_amax if handoff else None)
        out = L.make_out(y, acc, amax=amax)
        st = L.bitmtp_linear_gemm(L._ptr(pk), float(w), N, K, M, act, out, L._ptr(ws), ws.numel(), flags,
                                  L._stream(None))
        assert st == L.OK, L.status_string(st)
        res.append((y, acc, amax, pk))
        x, x_amax = y, amax
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_chain_matches_oracle(M, out_dtype):
    layers = _layers(9100 + M)
    x0 = np.random.default_rng(9200 + M).standard_normal((M, SHAPES[0][0])).astype(np.float32)
    ref = oracle.linear_chain(layers, x0, out=out_dtype)
    outs = {}
    for handoff in (True, False):
        got = _run_chain(layers, dev_tensor(x0), out_dtype, handoff, L.FLAG_PDL)
        for l, ((y, acc, amax, _), r) in enumerate(zip(got, ref)):
            assert np.array_equal(acc.cpu().numpy(), r["acc"].astype(np.int32)), (handoff, l)
            yb = y.cpu().numpy() if out_dtype == "f32" else bf16_bits(y)
            ry = r["y"]
            if out_dtype == "f32":
                assert np.array_equal(yb.view(np.uint32), ry.view(np.uint32)), (handoff, l)
            else:
                assert np.array_equal(yb, ry), (handoff, l)
            assert np.array_equal(amax.cpu().numpy().view(np.uint32), r["amax"].view(np.uint32)), (handoff, l)
        outs[handoff] = [t[0].cpu() for t in got]
    for a, b in zip(outs[True], outs[False]):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))


def test_chain_tensor_and_dp_paths_agree():
    """Width 4 on the dp4a path and on the forced tensor path give the same
    chain."""
    M = 4
    layers = _layers(9300)
    x0 = np.random.default_rng(9301).standard_normal((M, SHAPES[0][0])).astype(np.float32)
    a = _run_chain(layers, dev_tensor(x0), "bf16", True, L.FLAG_PDL | L.FLAG_FORCE_DP)
    b = _run_chain(layers, dev_tensor(x0), "bf16", True, L.FLAG_PDL | L.FLAG_FORCE_TC)
    for (ya, _, ma, _), (yb, _, mb, _) in zip(a, b):
        assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
        assert torch.equal(ma, mb)
