"""GPU parity of the layer-chained step: each linear's output is the next
linear's input, its epilogues reduce the output rows' absmax (first phase)
and the next call's preparation takes it instead of its own absmax pass
(second phase).  Every layer's stored output, accumulators and row absmax
are compared with the oracle's chain (``linear_chain``, which takes the
dequant in the kernel's fixed order) bit for bit, and the same chain without
the handed-over absmax gives the same bits.

At widths 1-4 (the dp4a path) a call whose every problem brings its rows'
absmax runs as one launch: no preparation kernel, the GEMM quantises its own
activation tiles.  Its single calls, grouped calls over mixed K, unaligned
and ragged rows, calls without an output absmax, and a chain replayed from a
CUDA graph (the workspace's sync words back at zero after every launch) are
compared with the oracle bit for bit; so are the same handed-over-absmax
calls at widths 5-16 (the tensor paths, with the preparation kernel)."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import bf16_bits, bf16_tensor, dev_tensor

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
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 16])
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


# ---------------------------------------------------------------------------
# Fused calls (dp4a path, handed-over absmax): single and grouped
# ---------------------------------------------------------------------------
def _act_on_device(x, is_bf16, offset):
    """x ([M, K] fp32 values or bf16 bits) on the device; offset > 0 places
    the rows at that element offset inside wider rows (not 16-byte aligned)."""
    M, K = x.shape
    src = bf16_tensor(x) if is_bf16 else dev_tensor(x)
    if offset == 0:
        return src
    buf = torch.zeros((M, K + offset + 5), dtype=src.dtype, device="cuda")
    buf[:, offset:offset + K] = src
    return buf[:, offset:offset + K]


def _row_amax(x, is_bf16):
    xf = oracle.bf16_bits_to_f32(x) if is_bf16 else x.astype(np.float32)
    return np.max(np.abs(xf), axis=1).astype(np.float32) if xf.shape[1] else np.zeros(xf.shape[0], np.float32)


def _expect(T, w, x, is_bf16, out_dtype):
    q, a_scale, _ = oracle.quant_act_bf16(x) if is_bf16 else oracle.quant_act(x)
    acc = oracle.gemm_acc(T, q)
    y = oracle.dequant_chain(acc, a_scale, w, out_dtype)
    yf = oracle.bf16_bits_to_f32(y) if out_dtype == "bf16" else y
    return acc, y, np.max(np.abs(yf), axis=1).astype(np.float32)


def _check(got_y, got_acc, got_amax, exp, out_dtype):
    acc, y, amax = exp
    assert np.array_equal(got_acc.cpu().numpy(), acc.astype(np.int32))
    if out_dtype == "f32":
        assert np.array_equal(got_y.cpu().numpy().view(np.uint32), y.view(np.uint32))
    else:
        assert np.array_equal(bf16_bits(got_y), y)
    if got_amax is not None:
        assert np.array_equal(got_amax.cpu().numpy().view(np.uint32), amax.view(np.uint32))


@pytest.mark.parametrize("M,N,K,is_bf16,offset,out_dtype,with_amax_out", [
    (1, 2560, 2560, True, 0, "bf16", True),
    (2, 1000, 300, False, 1, "f32", True),      # ragged K, unaligned rows
    (3, 130, 1000, True, 3, "bf16", True),      # ragged N and K, unaligned rows
    (4, 2560, 6912, True, 0, "f32", False),     # no output absmax
    (4, 384, 32768, False, 0, "bf16", True),    # the largest K
    (2, 6912, 2560, False, 0, "bf16", True),
    # several ring chunks per CTA (the later ones quantised by warp 5), the
    # ring wrapping around, fp32 and unaligned rows among them
    (4, 32000, 6912, True, 0, "bf16", True),
    (1, 32000, 6912, False, 1, "f32", True),
    (3, 20000, 1000, False, 0, "bf16", True),
    (2, 16000, 2560, True, 5, "f32", False),
    # the tensor paths (the preparation kernel takes the handed-over absmax)
    (5, 2560, 2560, True, 0, "bf16", True),
    (8, 1000, 300, False, 1, "f32", True),
    (9, 130, 1000, True, 3, "bf16", True),
    (16, 2560, 6912, True, 0, "f32", True),
    (16, 384, 2560, False, 0, "bf16", False),
    (8, 32000, 2560, True, 0, "bf16", True),
    (16, 11008, 4096, False, 1, "f32", True),
])
def test_fused_call_matches_oracle(M, N, K, is_bf16, offset, out_dtype, with_amax_out):
    rng = np.random.default_rng(9400 + M * 13 + K)
    T = inputs.ternary(rng, (N, K), 0.4)
    w = np.float32(0.0371)
    xf = rng.standard_normal((M, K)).astype(np.float32)
    xf[rng.random((M, K)) < 0.01] *= np.float32(25)
    if M > 2:
        xf[1] = 0.0                                  # zero row: codes 0, a_scale 0
    x = inputs.to_bf16_bits(xf) if is_bf16 else xf
    xd = _act_on_device(x, is_bf16, offset)
    amax_in = dev_tensor(_row_amax(x, is_bf16))
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    amax_out = torch.full((M,), -1.0, dtype=torch.float32, device="cuda") if with_amax_out else None
    ws = L.workspace(L.bitmtp_linear_workspace_bytes(N, K, M), xd.device)
    for _ in range(2):  # the second call on the same workspace: sync words reset
        st = L.bitmtp_linear_gemm(L._ptr(L.pack(dev_tensor(T))), float(w), N, K, M, L.make_act(xd, amax=amax_in),
                                  L.make_out(y, acc, amax=amax_out), L._ptr(ws), ws.numel(), L.FLAG_PDL,
                                  L._stream(None))
        assert st == L.OK, L.status_string(st)
        torch.cuda.synchronize()
        _check(y, acc, amax_out, _expect(T, w, x, is_bf16, out_dtype), out_dtype)
        assert int(ws[:1536].abs().sum()) == 0  # sync words and flags left at zero


@pytest.mark.parametrize("M", [1, 3, 4, 8, 12, 16])
def test_fused_grouped_mixed_k(M):
    rng = np.random.default_rng(9500 + M)
    if M <= 4:
        shapes = [(2560, 2560), (6912, 2560), (300, 1000), (2560, 6912)]  # (K, N)
    else:  # the tensor paths
        shapes = [(1024, 1024), (300, 1000), (2048, 512), (1000, 130)]
    probs, exps = [], []
    for i, (K, N) in enumerate(shapes):
        T = inputs.ternary(rng, (N, K), 0.5)
        w = np.float32(0.02 + 0.01 * i)
        x = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
        probs.append(dict(pk=L.pack(dev_tensor(T)), w_scale=float(w), N=N, K=K, x=bf16_tensor(x),
                          amax=dev_tensor(_row_amax(x, True)),
                          y=torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                          acc=torch.empty((M, N), dtype=torch.int32, device="cuda"),
                          amax_out=torch.full((M,), -1.0, dtype=torch.float32, device="cuda")))
        exps.append(_expect(T, w, x, True, "bf16"))
    L.gemm_grouped(probs, flags=L.FLAG_PDL)
    torch.cuda.synchronize()
    for pr, exp in zip(probs, exps):
        _check(pr["y"], pr["acc"], pr["amax_out"], exp, "bf16")


@pytest.mark.parametrize("M", [2, 4])
def test_fused_grouped_mixed_kinds_several_chunks(M):
    """One-launch grouped call over bf16 and fp32 rows (aligned and not), with
    about 13 tiles per CTA: warp 5 quantises chunks that hold tiles of two
    problems of different kinds."""
    rng = np.random.default_rng(9700 + M)
    specs = [(2560, 16000, True, 0), (6912, 2560, False, 0), (1000, 8000, False, 1), (300, 6000, True, 3)]
    probs, exps = [], []
    for i, (K, N, is_bf16, offset) in enumerate(specs):
        T = inputs.ternary(rng, (N, K), 0.45)
        w = np.float32(0.015 + 0.005 * i)
        xf = rng.standard_normal((M, K)).astype(np.float32)
        x = inputs.to_bf16_bits(xf) if is_bf16 else xf
        probs.append(dict(pk=L.pack(dev_tensor(T)), w_scale=float(w), N=N, K=K, x=_act_on_device(x, is_bf16, offset),
                          amax=dev_tensor(_row_amax(x, is_bf16)),
                          y=torch.empty((M, N), dtype=torch.float32, device="cuda"),
                          acc=torch.empty((M, N), dtype=torch.int32, device="cuda"),
                          amax_out=torch.full((M,), -1.0, dtype=torch.float32, device="cuda")))
        exps.append(_expect(T, w, x, is_bf16, "f32"))
    L.gemm_grouped(probs, flags=L.FLAG_PDL)
    torch.cuda.synchronize()
    for pr, exp in zip(probs, exps):
        _check(pr["y"], pr["acc"], pr["amax_out"], exp, "f32")


def test_fused_chain_replayed_from_a_graph():
    """The 4-layer chain at width 2, captured once with PDL and replayed three
    times on one workspace: every replay gives the oracle's chain and leaves
    the workspace's sync words and flags at zero."""
    M = 2
    layers = _layers(9600)
    x0 = np.random.default_rng(9601).standard_normal((M, SHAPES[0][0])).astype(np.float32)
    ref = oracle.linear_chain(layers, x0, out="bf16")
    xd = dev_tensor(x0)
    pks = [L.pack(dev_tensor(T)) for T, _ in layers]
    ws = L.workspace(L.bitmtp_linear_workspace_bytes(max(N for _, N in SHAPES), max(K for K, _ in SHAPES), M),
                     xd.device)
    bufs = [(torch.empty((M, N), dtype=torch.bfloat16, device="cuda"), torch.empty((M, N), dtype=torch.int32,
             device="cuda"), torch.zeros(M, dtype=torch.float32, device="cuda")) for _, N in SHAPES]
    stream = torch.cuda.Stream()

    def run():
        x, xa = xd, None
        for (T, w), (K, N), pk, (y, acc, am) in zip(layers, SHAPES, pks, bufs):
            st = L.bitmtp_linear_gemm(L._ptr(pk), float(w), N, K, M, L.make_act(x, amax=xa),
                                      L.make_out(y, acc, amax=am), L._ptr(ws), ws.numel(), L.FLAG_PDL,
                                      L._stream(torch.cuda.current_stream()))
            assert st == L.OK, L.status_string(st)
            x, xa = y, am

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    for _ in range(3):
        for y, acc, am in bufs:
            y.fill_(float("nan"))
            acc.zero_()
            am.fill_(-1.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        for (y, acc, am), r in zip(bufs, ref):
            assert np.array_equal(acc.cpu().numpy(), r["acc"].astype(np.int32))
            assert np.array_equal(bf16_bits(y), r["y"])
            assert np.array_equal(am.cpu().numpy().view(np.uint32), r["amax"].view(np.uint32))
        assert int(ws[:1536].abs().sum()) == 0
