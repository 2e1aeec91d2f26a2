"""GPU parity on the five benchmark workloads at full size, in the launch
configuration the benchmark uses (programmatic dependent launch between
consecutive linears).  Workloads 1, 2 and 5 compare every output; the 30-layer
and 36-layer stacks compare every output of their first and last layers and 64
sampled output features of every other projection."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_bf16_within_ulp, assert_f32_close, bf16_bits, bf16_tensor, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


def _compare(T, w, x_f32, q_ref_src, acc_gpu, y_gpu, out_dtype, cols=None):
    q, a, _ = oracle.quant_act(x_f32)
    Tc = T if cols is None else T[cols]
    acc_ref = oracle.gemm_acc(Tc, q)
    y_ref = oracle.dequant(acc_ref, a, w)
    acc_g = acc_gpu if cols is None else acc_gpu[:, cols]
    y_g = y_gpu if cols is None else y_gpu[:, cols]
    assert np.array_equal(acc_g, acc_ref.astype(np.int32))
    if out_dtype == torch.float32:
        assert_f32_close(y_g, y_ref, acc_ref)
    else:
        assert_bf16_within_ulp(y_g, y_ref)


def _run(T, w, x_dev, M, out_dtype):
    N, K = T.shape
    pk = L.pack(dev_tensor(T))
    y, acc = L.gemm(pk, w, N, K, x_dev[:M], out_dtype=out_dtype, acc=True, flags=L.FLAG_PDL)
    yh = y.cpu().numpy() if out_dtype == torch.float32 else bf16_bits(y)
    return acc.cpu().numpy(), yh


@pytest.mark.parametrize("M", [1, 4])
def test_single_linear_2560(M):
    T, w, x = inputs.single_linear(M)
    acc, y = _run(T, w, dev_tensor(x), M, torch.float32)
    _compare(T, w, x, None, acc, y, torch.float32)


@pytest.mark.parametrize("proj", range(len(inputs.BITNET2B_PROJ)))
def test_bitnet2b_layer_set(proj):
    T, w = inputs.bitnet2b_weights(proj)
    xb = inputs.bitnet2b_act(proj, 16)
    xd = bf16_tensor(xb)
    xf = oracle.bf16_bits_to_f32(xb)
    N, K = T.shape
    pk = L.pack(dev_tensor(T))
    for M in (1, 2, 4, 8):
        for out_dtype in (torch.bfloat16, torch.float32):
            y, acc = L.gemm(pk, w, N, K, xd[:M], out_dtype=out_dtype, acc=True, flags=L.FLAG_PDL)
            yh = y.cpu().numpy() if out_dtype == torch.float32 else bf16_bits(y)
            _compare(T, w, xf[:M], None, acc.cpu().numpy(), yh, out_dtype)


def _stack(weights_fn, act_fn, nlayers, nproj, widths, full_layers, seed):
    rng = np.random.default_rng(seed)
    for layer in range(nlayers):
        for p in range(nproj):
            T, w = weights_fn(p, layer)
            N, K = T.shape
            pk = L.pack(dev_tensor(T))
            xb = act_fn(p, 16, layer)
            xd = bf16_tensor(xb)
            xf = oracle.bf16_bits_to_f32(xb)
            cols = None if layer in full_layers else np.sort(rng.choice(N, 64, replace=False))
            for M in widths:
                y, acc = L.gemm(pk, w, N, K, xd[:M], out_dtype=torch.bfloat16, acc=True, flags=L.FLAG_PDL)
                _compare(T, w, xf[:M], None, acc.cpu().numpy(), bf16_bits(y), torch.bfloat16, cols)
            del pk


@pytest.mark.slow
def test_bitnet2b_30_layer_stack():
    _stack(lambda p, l: inputs.bitnet2b_weights(p, layer=l),
           lambda p, M, l: inputs.bitnet2b_act(p, M, layer=l),
           inputs.BITNET2B_LAYERS, len(inputs.BITNET2B_PROJ), (4,), {0, inputs.BITNET2B_LAYERS - 1}, 303)


@pytest.mark.slow
def test_large_36_layer_stack():
    _stack(inputs.large_weights, inputs.large_act, inputs.LARGE_LAYERS, len(inputs.LARGE_PROJ),
           (8, 12, 16), {0, inputs.LARGE_LAYERS - 1}, 404)


@pytest.mark.parametrize("sparsity_idx", range(len(inputs.ROLE_SPARSITY)))
def test_role_dependent_grouped(sparsity_idx):
    x = inputs.role_act(sparsity_idx)
    xd = dev_tensor(x)
    q, a, _ = L.quant_act(xd)
    probs, refs = [], []
    for g, (_, row0, rows, K, N) in enumerate(inputs.ROLE_GROUPS):
        T, w = inputs.role_weights(sparsity_idx, g)
        pk = L.pack(dev_tensor(T))
        y = torch.empty((rows, N), dtype=torch.float32, device="cuda")
        acc = torch.empty((rows, N), dtype=torch.int32, device="cuda")
        probs.append(dict(pk=pk, w_scale=w, N=N, K=K, x=q[row0:row0 + rows], a_scale=a[row0:row0 + rows],
                          y=y, acc=acc))
        refs.append((T, w, x[row0:row0 + rows]))
    L.gemm_grouped(probs, flags=L.FLAG_PDL)
    q_ref, a_ref, _ = oracle.quant_act(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    for p, (T, w, xr) in zip(probs, refs):
        _compare(T, w, xr, None, p["acc"].cpu().numpy(), p["y"].cpu().numpy(), torch.float32)
