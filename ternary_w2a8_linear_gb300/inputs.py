"""Seeded synthetic inputs for the W2A8 ternary linear.

This module only draws random data (numpy PCG64 with fixed seeds, and torch's
seeded generator on the device for the benchmark's large stacks); it holds
none of the linear's arithmetic.  Tests and the benchmark feed the same
arrays to the CUDA path and to the CPU oracle.

The pages measure only end-to-end decoding of trained models on task suites;
none of that is available here, so every workload below is synthetic, shaped
like the ternary backbones the pages run (BitNet b1.58-2B class layer shapes),
with the value distributions stated per workload.
"""
from __future__ import annotations

import numpy as np

# (name, K in-features, N out-features)
BITNET2B_PROJ = [
    ("q", 2560, 2560), ("k", 2560, 640), ("v", 2560, 640), ("o", 2560, 2560),
    ("gate", 2560, 6912), ("up", 2560, 6912), ("down", 6912, 2560),
]
BITNET2B_LAYERS = 30

LARGE_PROJ = [
    ("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024), ("o", 4096, 4096),
    ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096),
]
LARGE_LAYERS = 36

MAX_ROWS = 16


def ternary(rng: np.random.Generator, shape, p_zero: float | None) -> np.ndarray:
    """Ternary int8 matrix.  p_zero None: uniform over {-1, 0, +1};
    otherwise P(0) = p_zero and P(+1) = P(-1) = (1 - p_zero) / 2."""
    if p_zero is None:
        return rng.integers(-1, 2, size=shape, dtype=np.int8)
    # 16-bit uniform draw through a lookup table: P(0) = round(p_zero * 2^16) / 2^16
    z = int(round(p_zero * 65536))
    h = z + (65536 - z) // 2
    lut = np.full(65536, -1, dtype=np.int8)
    lut[:z] = 0
    lut[z:h] = 1
    return lut[rng.integers(0, 65536, size=shape, dtype=np.uint16)]


def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 data to bf16 (torch's round-to-nearest-even) -> uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal_with_outliers_bf16(rng: np.random.Generator, shape, frac=0.01, mult=20.0) -> np.ndarray:
    """bf16 bits of N(0,1) data where each element is multiplied by ``mult``
    with probability ``frac``."""
    x = rng.standard_normal(shape, dtype=np.float32)
    hit = rng.random(shape, dtype=np.float32) < frac
    x[hit] *= np.float32(mult)
    return to_bf16_bits(x)


# ---------------------------------------------------------------------------
# Workload 1: single 2560 -> 2560 linear, uniform ternary, fp32 activations.
# ---------------------------------------------------------------------------
def single_linear(M: int):
    """T uniform over {-1,0,1} (seed 0), w_scale 0.02, x fp32 N(0,1) (seed 100+M)."""
    T = ternary(np.random.default_rng(0), (2560, 2560), None)
    x = normal_f32(np.random.default_rng(100 + M), (M, 2560))
    return T, np.float32(0.02), x


# ---------------------------------------------------------------------------
# Workload 2/3: BitNet-2B-shaped projections, P(0)=0.5, bf16 activations with
# 1% outliers x20.  Layer-set copy / layer index selects distinct weights.
# ---------------------------------------------------------------------------
def bitnet2b_weights(proj_idx: int, layer: int | None = None):
    """Weights of one BitNet-2B projection.  layer None: the single layer set
    (seed 2000 + proj); otherwise layer ``layer`` of the 30-layer stack
    (seed 3000 + 10*layer + proj).  w_scale ~ U[0.01, 0.05]."""
    _, K, N = BITNET2B_PROJ[proj_idx]
    seed = 2000 + proj_idx if layer is None else 3000 + 10 * layer + proj_idx
    rng = np.random.default_rng(seed)
    T = ternary(rng, (N, K), 0.5)
    w_scale = np.float32(rng.uniform(0.01, 0.05))
    return T, w_scale


def bitnet2b_dense_weights(proj_idx: int) -> np.ndarray:
    """fp32 weights [N, K] of one BitNet-2B projection before ternarisation:
    N(0, 0.02^2), seed 6000 + proj (input of the device ternarisation)."""
    _, K, N = BITNET2B_PROJ[proj_idx]
    rng = np.random.default_rng(6000 + proj_idx)
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)


def bitnet2b_act(proj_idx: int, M: int, layer: int | None = None) -> np.ndarray:
    """bf16 bits [M, K]; the first M of 16 seeded rows (seed 2100 + proj, or
    7000 + 10*layer + proj for the 30-layer stack)."""
    _, K, _ = BITNET2B_PROJ[proj_idx]
    seed = 2100 + proj_idx if layer is None else 7000 + 10 * layer + proj_idx
    x = normal_with_outliers_bf16(np.random.default_rng(seed), (MAX_ROWS, K))
    return np.ascontiguousarray(x[:M])


# ---------------------------------------------------------------------------
# Workload 4: hidden 4096 / FFN 11008 shapes, 36 layers, P(0)=1/3, bf16 N(0,1).
# ---------------------------------------------------------------------------
def large_weights(proj_idx: int, layer: int):
    _, K, N = LARGE_PROJ[proj_idx]
    rng = np.random.default_rng(4000 + 10 * layer + proj_idx)
    T = ternary(rng, (N, K), None)  # uniform == P(0) = 1/3, +-1 equally likely
    w_scale = np.float32(rng.uniform(0.01, 0.05))
    return T, w_scale


def large_act(proj_idx: int, M: int, layer: int) -> np.ndarray:
    _, K, _ = LARGE_PROJ[proj_idx]
    x = normal_f32(np.random.default_rng(8000 + 10 * layer + proj_idx), (MAX_ROWS, K))
    return np.ascontiguousarray(to_bf16_bits(x)[:M])


# ---------------------------------------------------------------------------
# Workload 5: role-dependent output projection at width 16.
# rows 0-3 (verify): 2560 -> 32000; rows 4-15 (draft): 2560 -> 2560.
# ---------------------------------------------------------------------------
ROLE_SPARSITY = (0.2, 0.5, 0.8)
ROLE_GROUPS = (("verify", 0, 4, 2560, 32000), ("draft", 4, 12, 2560, 2560))  # name, row0, rows, K, N


def role_weights(sparsity_idx: int, group: int):
    _, _, _, K, N = ROLE_GROUPS[group]
    rng = np.random.default_rng(5000 + 10 * sparsity_idx + group)
    T = ternary(rng, (N, K), ROLE_SPARSITY[sparsity_idx])
    w_scale = np.float32(rng.uniform(0.01, 0.05))
    return T, w_scale


def role_act(sparsity_idx: int) -> np.ndarray:
    return normal_f32(np.random.default_rng(5500 + sparsity_idx), (MAX_ROWS, 2560))


# ---------------------------------------------------------------------------
# Generic random problems for parity tests.
# ---------------------------------------------------------------------------
def random_problem(seed: int, M: int, N: int, K: int, p_zero=None, x_kind: str = "f32",
                   outliers: bool = False):
    """Returns (T int8 [N,K], w_scale fp32, x) with x fp32 [M,K] or bf16 bits."""
    rng = np.random.default_rng(seed)
    T = ternary(rng, (N, K), p_zero)
    w_scale = np.float32(rng.uniform(0.01, 0.05))
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        x[rng.random((M, K), dtype=np.float32) < 0.01] *= np.float32(20.0)
    if x_kind == "bf16":
        return T, w_scale, to_bf16_bits(x)
    return T, w_scale, x


# ---------------------------------------------------------------------------
# Device-side generators for the benchmark's large stacks (hundreds of
# millions of weights per layer set), drawn with torch's seeded generator on
# the GPU.  Same distributions as above; different streams from the numpy
# ones, so the benchmark draws the layers it checks against the oracle with
# the numpy generators and the rest with these.
# ---------------------------------------------------------------------------
def device_ternary(seed: int, shape, p_zero: float | None, device):
    """Ternary int8 tensor on `device`.  p_zero None: uniform over {-1, 0, +1};
    otherwise P(0) = p_zero (to 2^-16) and P(+1) = P(-1)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if p_zero is None:
        return (torch.randint(0, 3, shape, generator=g, device=device, dtype=torch.int8) - 1).contiguous()
    z = int(round(p_zero * 65536))
    h = z + (65536 - z) // 2
    r = torch.randint(0, 65536, shape, generator=g, device=device, dtype=torch.int32)
    t = torch.where(r < z, 0, torch.where(r < h, 1, -1))
    return t.to(torch.int8).contiguous()


def device_normal_bf16(seed: int, shape, device, outlier_frac: float = 0.0, mult: float = 20.0):
    """bf16 N(0, 1) tensor on `device`; each element multiplied by `mult`
    with probability `outlier_frac`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        hit = torch.rand(shape, generator=g, device=device) < outlier_frac
        x = torch.where(hit, x * mult, x)
    return x.to(torch.bfloat16).contiguous()
