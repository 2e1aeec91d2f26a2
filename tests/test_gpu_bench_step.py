"""GPU parity of the exact step the benchmark times, and of the tensor path's
fp32 accumulator on adversarial sums.

The benchmark's step is one grouped call of the seven BitNet-2B projections
(mixed in-features 2560 and 6912) per block width, every call with
programmatic dependent launch, replayed from a CUDA graph while the weights
rotate over distinct copies, all calls sharing one workspace.  Here that
graph is captured the same way, over two weight copies and the widths 1, 2,
4, 8, 12 and 16, and every output is compared with the oracle: int32
accumulators bit-exact, bf16 outputs within one bf16 ulp of the oracle's fp32
value rounded to bf16.

The tensor path computes sum_k u * h and sum_k u * l (u = T + 1 in {0, 1, 2},
q = 16 h + l) in the fp32 accumulator of tcgen05.mma kind::f8f6f4 with inputs
scaled by 2^-9; the result is exact only if the accumulator keeps every bit up
to 2^20 units.  The adversarial case drives it there with large same-sign sums
whose low bits vary: all-+1 (or +1 on a random half) weights against codes in
[64, 127] that are not constant, at the largest in-feature count."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_bf16_within_ulp, bf16_bits, bf16_tensor, dev_tensor

pytestmark = pytest.mark.gpu

WIDTHS = (1, 2, 4, 8, 12, 16)
COPIES = 2


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


def _oracle_rows16(T, w, xb):
    """Oracle for the 16 seeded rows; rows are quantised independently, so the
    first M rows of this result are the oracle for width M."""
    xf = oracle.bf16_bits_to_f32(xb)
    q, a, _ = oracle.quant_act(xf)
    acc = oracle.gemm_acc(T, q)
    y = oracle.dequant(acc, a, w)
    return acc, y


@pytest.mark.parametrize("with_acc", [False, True])
def test_bench_step_graph_pdl_rotating_copies(with_acc):
    proj = inputs.BITNET2B_PROJ
    xs_np = [inputs.bitnet2b_act(p, 16) for p in range(len(proj))]
    xs = [bf16_tensor(x) for x in xs_np]
    weights, refs = [], []
    for c in range(COPIES):
        row, rrow = [], []
        for p in range(len(proj)):
            T, w = inputs.bitnet2b_weights(p, layer=c)
            row.append((L.pack(dev_tensor(T)), float(w)))
            rrow.append(_oracle_rows16(T, w, xs_np[p]))
        weights.append(row)
        refs.append(rrow)
    # outputs per (copy, width, projection)
    ys, accs = {}, {}
    for c in range(COPIES):
        for M in WIDTHS:
            for p, (_, K, N) in enumerate(proj):
                ys[(c, M, p)] = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                accs[(c, M, p)] = (torch.full((M, N), -1, dtype=torch.int32, device="cuda")
                                   if with_acc else None)
    descs = {}
    for c in range(COPIES):
        for M in WIDTHS:
            d = []
            for p, (_, K, N) in enumerate(proj):
                pk, w = weights[c][p]
                d.append(L.GemmDesc(pk.data_ptr(), w, N, K, M, L.Act(L.BF16, xs[p].data_ptr(), K, None),
                                    L.make_out(ys[(c, M, p)], accs[(c, M, p)])))
            descs[(c, M)] = ((L.GemmDesc * len(d))(*d), len(d))
    nb = max(L.bitmtp_linear_workspace_bytes_grouped(list(a[:n])) for a, n in descs.values())
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    cs = L.ctypes.c_void_p(stream.cuda_stream)
    lib = L.load()

    def step(c):
        for M in WIDTHS:
            arr, n = descs[(c, M)]
            st = lib.bitmtp_linear_gemm_grouped(arr, n, L.ctypes.c_void_p(ws.data_ptr()), nb, L.FLAG_PDL, cs)
            assert st == L.OK, L.status_string(st)

    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step(0)  # warm call outside the capture, as the benchmark does
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in range(COPIES):
                step(c)
        for v in ys.values():
            v.fill_(float("nan"))
        for _ in range(2):
            g.replay()
    stream.synchronize()
    for c in range(COPIES):
        for M in WIDTHS:
            for p in range(len(proj)):
                acc_ref, y_ref = refs[c][p]
                if with_acc:
                    got = accs[(c, M, p)].cpu().numpy()
                    assert np.array_equal(got, acc_ref[:M].astype(np.int32)), (c, M, p)
                assert_bf16_within_ulp(bf16_bits(ys[(c, M, p)]), y_ref[:M])


@pytest.mark.parametrize("M", [8, 16])
@pytest.mark.parametrize("wkind", ["all_plus", "half_plus"])
def test_tensor_accumulator_large_odd_sums(M, wkind):
    K, N = 32768, 130
    rng = np.random.default_rng(4242 + M)
    x = rng.uniform(0.5, 1.0, size=(M, K)).astype(np.float32)  # codes in [64, 127], not constant
    if wkind == "all_plus":
        T = np.ones((N, K), dtype=np.int8)
    else:
        T = (rng.random((N, K)) < 0.5).astype(np.int8)
    w = np.float32(0.013)
    pk = L.pack(dev_tensor(T))
    y, acc = L.gemm(pk, w, N, K, dev_tensor(x), acc=True, flags=L.FLAG_FORCE_TC)
    q, a, _ = oracle.quant_act(x)
    assert q.min() >= 64 and len(np.unique(q)) > 32
    acc_ref = oracle.gemm_acc(T, q)
    # large same-sign sums: above 2^20, so the h and l partial sums reach 2^18..2^20 units
    assert acc_ref.max() > 2 ** 20
    got = acc.cpu().numpy()
    assert np.array_equal(got, acc_ref.astype(np.int32)), np.argwhere(got != acc_ref)[:3]
