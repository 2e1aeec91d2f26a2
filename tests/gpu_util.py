"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI binding, and compare with the oracle at the stated
tolerances (bit-exact integers; fp32 within 1e-5 relative with exact zeros;
bf16 within one bf16 ulp of the oracle's fp32 value rounded to bf16)."""
import math

import numpy as np
import torch

import oracle

FP32_RTOL = 1e-5


def dev_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def act_f32_for_oracle(x: np.ndarray, is_bf16: bool) -> np.ndarray:
    return oracle.bf16_bits_to_f32(x) if is_bf16 else x


def assert_f32_close(got: np.ndarray, ref: np.ndarray, acc: np.ndarray | None = None):
    got = np.asarray(got, dtype=np.float32)
    ref = np.asarray(ref, dtype=np.float32)
    assert got.shape == ref.shape
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    tol = FP32_RTOL * np.abs(ref.astype(np.float64))
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"fp32 mismatch at {tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                             f"({int(bad.sum())} elements)")
    if acc is not None:
        assert np.all(got[acc == 0] == 0)


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b)


def assert_bf16_within_ulp(got_bits: np.ndarray, ref_f32: np.ndarray):
    ref_bits = oracle.f32_to_bf16_bits(ref_f32)
    d = np.abs(_ordered(got_bits) - _ordered(ref_bits))
    if (d > 1).any():
        i = np.argwhere(d > 1)[0]
        raise AssertionError(f"bf16 mismatch at {tuple(i)}: got {hex(int(got_bits[tuple(i)]))} "
                             f"ref {hex(int(ref_bits[tuple(i)]))}")


def reference(T, w_scale, x, x_is_bf16):
    """Oracle result (y fp32, acc int64, q, a_scale)."""
    y, acc, q, a_scale, _ = oracle.w2a8_linear(T, w_scale, x, "f32", x_is_bf16=x_is_bf16)
    return y, acc, q, a_scale


# ---------------------------------------------------------------------------
# FP8 ("fast" draft projection) results: the fp32 accumulation adds
# 2 * ceil(K/32) MMA results (sum_k (T+1)*e and -sum_k e per k step), so
# |acc - sum_k T*e| <= (2 * ceil(K/32) + 2) * 2^-23 * sum_k (T+2)*|e|; y within
# that times a_scale * w_scale plus two fp32 roundings (and the bf16 rounding).
# ---------------------------------------------------------------------------
def fp8_reference(T, w, x, is_bf16):
    """Oracle (y fp32, exact acc, e, a_scale) and S = sum_k (T+2)*|e| per output."""
    y, acc, e, a_scale = oracle.fp8_linear(T, w, x, "f32", x_is_bf16=is_bf16)
    S = np.abs(e) @ (T.astype(np.float64) + 2).T
    return y, acc, e, a_scale, S


def fp8_acc_bound(K, S):
    return (2 * math.ceil(K / 32) + 2) * 2.0 ** -23 * S


def assert_fp8_within_bound(K, w, y, acc, ref, bf16_out):
    """y: fp32 values or bf16 bit patterns; acc: the fp32 accumulators (or
    None).  Returns the largest |acc error| / bound seen."""
    y_ref, acc_ref, _, a_scale, S = ref
    B = fp8_acc_bound(K, S)
    ratio = 0.0
    if acc is not None:
        err = np.abs(acc.astype(np.float64) - acc_ref)
        assert np.all(err <= B), f"acc beyond bound: max ratio {float(np.max(err / np.maximum(B, 1e-300))):.3g}"
        ratio = float(np.max(err / np.maximum(B, 1e-300))) if err.size else 0.0
    scale = a_scale.astype(np.float64)[:, None] * float(np.float32(w))
    yr = np.abs(y_ref.astype(np.float64))
    tol32 = B * scale * (1 + 2.0 ** -21) + 2.0 ** -21 * yr
    yv = oracle.bf16_bits_to_f32(y).astype(np.float64) if bf16_out else np.asarray(y, dtype=np.float64)
    tol = tol32 + (2.0 ** -8 * (yr + tol32) if bf16_out else 0.0)
    yerr = np.abs(yv - y_ref.astype(np.float64))
    assert np.all(yerr <= tol), f"y beyond bound at {tuple(np.argwhere(yerr > tol)[0])}"
    assert np.all(yv[S == 0] == 0)  # every product and correction term zero: exact zero
    return ratio
