"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI binding, and compare with the oracle at the stated
tolerances (bit-exact integers; fp32 within 1e-5 relative with exact zeros;
bf16 within one bf16 ulp of the oracle's fp32 value rounded to bf16)."""
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
