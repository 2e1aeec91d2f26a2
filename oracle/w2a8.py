"""Plain CPU oracle for the W2A8 ternary linear.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and this module shares no code, table or constant
generator with that path.

What is computed, and where it comes from
-----------------------------------------
The pages ("BitMTP: When Multi-Token Prediction Meets Low-Bit Large Language
Models", AI summary) describe the backbone as BitNet b1.58-style ternary
("What This Paper Is About"; "Overview": ultra-low-bit ternary / 1.58-bit
backbones), run in the "W2A8 setting (2-bit weights, 8-bit activations)"
("Main Findings", first bullet) through "packed W2A8 execution" and
width-specialised packed low-bit operators ("Methodology in Plain English",
third and last paragraphs).  The pages print no formula.  This library's
specification fills that in with the BitNet b1.58 definitions, which this
oracle writes out directly:

* weights: T in {-1, 0, +1} with one fp32 per-tensor absmean scale,
  W ~= w_scale * T  (``ternarize_absmean``);
* activations: per row, amax = max|x|, s = 127 / amax, q = round-half-even(x*s)
  in fp32, a_scale = amax / 127  (``quant_act``);
* integer accumulation acc[m, n] = sum_k T[n, k] * q[m, k]  (``gemm_acc``);
* dequant epilogue y = acc * a_scale[m] * w_scale  (``dequant``).

Readings taken where the pages are silent: a zero row gives all-zero codes
and a_scale 0; codes are clamped to +-127; s is multiplied, not divided; the
weight epsilon is 1e-5; mean|W| is the exact sum rounded once to fp64; bf16
widens exactly; dequant is evaluated in fp64 and rounded once to fp32, then
to bf16 for bf16 output.

The packed-weight format (``pack_tiles`` / ``unpack_tiles``) is this library's
own internal layout, not the pages'; it is restated here from its written
definition so that the device pack kernel can be checked byte for byte.

The FP8 "fast" draft projection (``quant_act_fp8``, ``gemm_acc_fp8``,
``fp8_linear``) follows the reading stated at its definition.

Precision: the quantiser is fp32 (the specification fixes it); accumulation is
exact int64; dequant is fp64 then rounded to fp32 (``dequant``), or, inside a
layer chain, two fp32 roundings in a fixed order (``dequant_chain``).
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64

QMAX = 127
WEIGHT_EPS = F32(1e-5)


# ---------------------------------------------------------------------------
# bf16 helpers (bf16 values are carried as their uint16 bit patterns)
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32."""
    b = np.asarray(bits).astype(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(F32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16, round-to-nearest-even, returning uint16 bits.

    Finite inputs only (the oracle never produces non-finite values)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=F32)).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# A2: absmean ternarisation (BitNet b1.58 weight quantiser)
# ---------------------------------------------------------------------------
def ternarize_absmean(W: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """T = clamp(round_half_even(W / gamma), -1, 1), gamma = max(mean|W|, 1e-5).

    mean|W|: the exact sum of |W|, rounded once to fp64 (math.fsum, so that
    the value does not depend on a summation order), divided by the count in
    fp64 and rounded once to fp32.  The division W / gamma and the rounding
    are fp32 IEEE operations.  Returns (T int8 [N, K], w_scale fp32) with
    W ~= w_scale * T."""
    W = np.asarray(W, dtype=F32)
    if W.size == 0:
        raise ValueError("empty weight matrix")
    if not np.all(np.isfinite(W)):
        raise ValueError("non-finite weight")
    total = math.fsum(np.abs(W.astype(F64)).ravel())
    gamma = F32(F64(total) / F64(W.size))
    gamma = max(gamma, WEIGHT_EPS)
    ratio = (W / gamma).astype(F32)
    T = np.clip(np.rint(ratio), -1, 1).astype(np.int8)
    return T, F32(gamma)


# ---------------------------------------------------------------------------
# A3: per-row absmax int8 activation quantiser
# ---------------------------------------------------------------------------
def quant_act(x: np.ndarray):
    """Quantise each row of x (fp32 [M, K]) to int8 codes by absmax.

    Per row m, all in fp32 round-to-nearest-even:
      amax = max_k |x[m, k]|
      amax == 0  ->  q = 0, a_scale = 0, rowsum = 0
      otherwise  ->  s = 127 / amax;  q = clamp(rint(x * s), -127, 127);
                     a_scale = amax / 127;  rowsum = sum_k q  (int32)
    Returns (q int8 [M, K], a_scale fp32 [M], rowsum int32 [M])."""
    x = np.asarray(x, dtype=F32)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [M, K]")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite activation")
    M, K = x.shape
    q = np.zeros((M, K), dtype=np.int8)
    a_scale = np.zeros(M, dtype=F32)
    rowsum = np.zeros(M, dtype=np.int32)
    for m in range(M):
        row = x[m]
        amax = F32(np.max(np.abs(row))) if K else F32(0)
        if amax == 0:
            continue
        s = F32(F32(QMAX) / amax)
        v = (row * s).astype(F32)
        qm = np.clip(np.rint(v), -QMAX, QMAX).astype(np.int8)
        q[m] = qm
        a_scale[m] = F32(amax / F32(QMAX))
        rowsum[m] = np.int32(np.sum(qm.astype(np.int64)))
    return q, a_scale, rowsum


def quant_act_bf16(x_bits: np.ndarray):
    """``quant_act`` on bf16 activations given as uint16 bit patterns."""
    return quant_act(bf16_bits_to_f32(x_bits))


# ---------------------------------------------------------------------------
# A4: integer accumulation and the dequant epilogue
# ---------------------------------------------------------------------------
def gemm_acc(T: np.ndarray, q: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k T[n, k] * q[m, k], exact in int64.

    Raises if a result does not fit int32 (the device accumulator type)."""
    T = np.asarray(T)
    q = np.asarray(q)
    if T.ndim != 2 or q.ndim != 2 or T.shape[1] != q.shape[1]:
        raise ValueError("shape mismatch: T [N, K], q [M, K]")
    acc = q.astype(np.int64) @ T.astype(np.int64).T
    if acc.size and (acc.max() > np.iinfo(np.int32).max or acc.min() < np.iinfo(np.int32).min):
        raise OverflowError("accumulator exceeds int32")
    return acc


def dequant(acc: np.ndarray, a_scale: np.ndarray, w_scale, out: str = "f32") -> np.ndarray:
    """y[m, n] = acc[m, n] * a_scale[m] * w_scale, evaluated in fp64 and
    rounded once to fp32; ``out="bf16"`` then rounds that fp32 value to bf16
    (round-to-nearest-even) and returns uint16 bit patterns."""
    y64 = (np.asarray(acc, dtype=F64)
           * np.asarray(a_scale, dtype=F64)[:, None]
           * F64(F32(w_scale)))
    y32 = y64.astype(F32)
    if out == "f32":
        return y32
    if out == "bf16":
        return f32_to_bf16_bits(y32)
    raise ValueError(f"unknown output dtype {out!r}")


def w2a8_linear(T, w_scale, x, out: str = "f32", x_is_bf16: bool = False):
    """quant_act -> gemm_acc -> dequant.  Returns (y, acc, q, a_scale, rowsum)."""
    q, a_scale, rowsum = quant_act_bf16(x) if x_is_bf16 else quant_act(x)
    acc = gemm_acc(T, q)
    return dequant(acc, a_scale, w_scale, out), acc, q, a_scale, rowsum


# ---------------------------------------------------------------------------
# Layer chain: the output of one linear is the input of the next.  The next
# layer's codes are decided on the stored output values, so a chain needs one
# fixed dequant order on both sides; the pages fix none.  Reading taken:
# y = RN32(RN32(acc * a_scale) * w_scale), then RN to bf16 for bf16 output
# (the single fp64 rounding of ``dequant`` can differ from this by one fp32
# ulp, which can move a code of the next layer).  The stored output's row
# absmax is the next layer's amax.
# ---------------------------------------------------------------------------
def dequant_chain(acc: np.ndarray, a_scale: np.ndarray, w_scale, out: str = "f32") -> np.ndarray:
    """y[m, n] = RN32(RN32(acc[m, n] * a_scale[m]) * w_scale) (fp32 IEEE
    products; acc is exact in fp32); ``out="bf16"`` rounds that to bf16 and
    returns uint16 bit patterns."""
    acc = np.asarray(acc, dtype=np.int64)
    if acc.size and np.abs(acc).max() >= 2 ** 24:
        raise OverflowError("accumulator not exact in fp32")
    t = (acc.astype(F32) * np.asarray(a_scale, dtype=F32)[:, None]).astype(F32)
    y32 = (t * F32(w_scale)).astype(F32)
    if out == "f32":
        return y32
    if out == "bf16":
        return f32_to_bf16_bits(y32)
    raise ValueError(f"unknown output dtype {out!r}")


def linear_chain(layers, x0: np.ndarray, out: str = "f32", x0_is_bf16: bool = False):
    """Run the linears (T, w_scale) of ``layers`` one after another, each on
    the previous one's stored output (fp32, or bf16 bit patterns for
    ``out="bf16"``).  Returns one dict per layer: y (as stored), acc, q,
    a_scale and amax (max_n |y[m, n]| of the stored values, fp32)."""
    x, is_bf16 = x0, x0_is_bf16
    res = []
    for T, w_scale in layers:
        q, a_scale, _ = quant_act_bf16(x) if is_bf16 else quant_act(x)
        acc = gemm_acc(T, q)
        y = dequant_chain(acc, a_scale, w_scale, out)
        yf = bf16_bits_to_f32(y) if out == "bf16" else y
        amax = np.max(np.abs(yf), axis=1).astype(F32) if yf.shape[1] else np.zeros(yf.shape[0], F32)
        res.append(dict(y=y, acc=acc, q=q, a_scale=a_scale, amax=amax))
        x, is_bf16 = y, out == "bf16"
    return res


# ---------------------------------------------------------------------------
# "Fast" draft projections with FP8 activations.  The pages run cheaper "fast"
# projections for drafting and more careful "critical" ones for generation
# and verification, and on H20 "additionally" FP8 draft projections
# ("Methodology in Plain English", M1).  They give no formula.  Reading taken:
# the backbone weights stay ternary (packed 2-bit; -1, 0 and +1 are exact
# FP8 values) and the draft rows' activations are quantised per row to FP8
# E4M3 instead of int8, by absmax, with the same fp32 steps as ``quant_act``
# and 448 (the largest finite E4M3 value) in place of 127:
#   s = RN32(448 / amax);  e = E4M3(RN32(x * s));  a_scale = RN32(amax / 448);
# E4M3 here is the OCP FP8 format without infinities: sign, 4 exponent bits
# (bias 7), 3 mantissa bits; normal values 1.m * 2^E for E in -6..8 (largest
# 1.75 * 2^8 = 448), subnormal values j * 2^-9; conversion rounds to nearest,
# ties to even, and saturates at +-448.  The accumulation sum_k T * e is exact
# here (every e is a multiple of 2^-9 below 2^9 in magnitude, so the sum is an
# integer number of 2^-9 units below 2^33); the device accumulates in fp32,
# so its results agree within a bound, not bit for bit.
# ---------------------------------------------------------------------------
FP8_MAX = 448.0
FP8_MIN_EXP = -6        # smallest normal binade 2^-6
FP8_MANT_BITS = 3


def e4m3_round(v) -> np.ndarray:
    """Round fp32 (or exactly representable fp64) values to the E4M3 grid,
    round-to-nearest-even, saturating at +-448.  Returns fp64 values.

    The grid step in the binade [2^E, 2^(E+1)) is 2^(E-3) for E >= -6; below
    2^-6 (the subnormals) it is 2^-9.  Dividing by a power of two is exact, so
    rint (half to even) on the scaled value is the correctly rounded result."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1)
    binade = np.maximum(ex - 1, FP8_MIN_EXP)
    step = np.ldexp(1.0, binade - FP8_MANT_BITS)
    r = np.minimum(np.rint(a / step) * step, FP8_MAX)
    return np.where(v < 0, -r, r)


def quant_act_fp8(x: np.ndarray):
    """Quantise each row of x (fp32 [M, K]) to E4M3 values by absmax.

    Per row m, in fp32 round-to-nearest-even:
      amax = max_k |x[m, k]|
      amax == 0  ->  e = 0, a_scale = 0
      otherwise  ->  s = 448 / amax;  e = E4M3(x * s);  a_scale = amax / 448
    Returns (e fp64 [M, K] holding E4M3 values, a_scale fp32 [M])."""
    x = np.asarray(x, dtype=F32)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [M, K]")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite activation")
    M, K = x.shape
    e = np.zeros((M, K), dtype=F64)
    a_scale = np.zeros(M, dtype=F32)
    for m in range(M):
        row = x[m]
        amax = F32(np.max(np.abs(row))) if K else F32(0)
        if amax == 0:
            continue
        s = F32(F32(FP8_MAX) / amax)
        e[m] = e4m3_round((row * s).astype(F32))
        a_scale[m] = F32(amax / F32(FP8_MAX))
    return e, a_scale


def quant_act_fp8_bf16(x_bits: np.ndarray):
    """``quant_act_fp8`` on bf16 activations given as uint16 bit patterns."""
    return quant_act_fp8(bf16_bits_to_f32(x_bits))


def gemm_acc_fp8(T: np.ndarray, e: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k T[n, k] * e[m, k], exact: computed in int64 units of
    2^-9 (every E4M3 value is an integer multiple of 2^-9) and returned as
    fp64 (exact, below 2^33 units)."""
    T = np.asarray(T)
    e = np.asarray(e, dtype=F64)
    if T.ndim != 2 or e.ndim != 2 or T.shape[1] != e.shape[1]:
        raise ValueError("shape mismatch: T [N, K], e [M, K]")
    units = e * 512.0
    if units.size and not np.array_equal(units, np.rint(units)):
        raise ValueError("e is not on the E4M3 grid")
    acc_units = units.astype(np.int64) @ T.astype(np.int64).T
    return acc_units.astype(F64) / 512.0


def fp8_linear(T, w_scale, x, out: str = "f32", x_is_bf16: bool = False):
    """quant_act_fp8 -> gemm_acc_fp8 -> dequant (fp64, rounded once).
    Returns (y, acc, e, a_scale)."""
    e, a_scale = quant_act_fp8_bf16(x) if x_is_bf16 else quant_act_fp8(x)
    acc = gemm_acc_fp8(T, e)
    return dequant(acc, a_scale, w_scale, out), acc, e, a_scale


# ---------------------------------------------------------------------------
# Packed-weight format (this library's own layout; restated from its definition)
#
#   * rows are grouped in row tiles of 128, k in k tiles of 128; both padded
#     with T = 0;
#   * tile (rt, kt) is 4096 contiguous bytes at byte offset (rt*KT + kt)*4096;
#   * inside a tile, row r has eight 32-bit words j = 0..7; word j of row r is
#     stored at word index (j // 4)*512 + r*4 + (j % 4);
#   * word j holds k = kt*128 + 16*j + 2*p + e (p = 0..7, e = 0..1) as the
#     2-bit code u = T + 1 in bits 16*e + 2*p .. 16*e + 2*p + 1 (u = 3 never
#     occurs);
#   * a 16-byte trailer follows the tiles: uint32 {0x38413242, N, K, invalid},
#     invalid = number of entries of the source that were not in {-1, 0, 1}.
# ---------------------------------------------------------------------------
TILE_N = 128
TILE_K = 128
TILE_BYTES = 4096
TRAILER_MAGIC = 0x38413242


def packed_bytes(N: int, K: int) -> int:
    nt = -(-N // TILE_N)
    kt = -(-K // TILE_K)
    return nt * kt * TILE_BYTES + 16


def pack_tiles(T: np.ndarray) -> np.ndarray:
    """Pack ternary int8 T [N, K] into the tiled 2-bit format (uint8 bytes)."""
    T = np.asarray(T)
    N, K = T.shape
    nt, kt = -(-N // TILE_N), -(-K // TILE_K)
    invalid = int(np.count_nonzero((T < -1) | (T > 1)))
    Tp = np.zeros((nt * TILE_N, kt * TILE_K), dtype=np.int64)
    Tp[:N, :K] = T
    u = np.where((Tp >= -1) & (Tp <= 1), Tp + 1, 1).astype(np.uint64)
    # axes: [rt, r, kt, j, p, e]
    u = u.reshape(nt, TILE_N, kt, 8, 8, 2)
    shifts = (np.uint64(16) * np.arange(2, dtype=np.uint64)[None, :]
              + np.uint64(2) * np.arange(8, dtype=np.uint64)[:, None])  # [p, e]
    words = np.sum(u << shifts, axis=(4, 5)).astype(np.uint32)          # [rt, r, kt, j]
    words = words.reshape(nt, TILE_N, kt, 2, 4)                         # j = 4*half + jj
    tiles = np.transpose(words, (0, 2, 3, 1, 4))                        # [rt, kt, half, r, jj]
    body = np.ascontiguousarray(tiles).reshape(-1).view(np.uint8)
    trailer = np.array([TRAILER_MAGIC, N, K, invalid], dtype=np.uint32).view(np.uint8)
    return np.concatenate([body, trailer])


def unpack_tiles(pk: np.ndarray, N: int, K: int) -> np.ndarray:
    """Inverse of ``pack_tiles``: tiled bytes -> T int8 [N, K].

    Raises on a 2-bit code of 3 anywhere (including padding)."""
    pk = np.asarray(pk, dtype=np.uint8)
    nt, kt = -(-N // TILE_N), -(-K // TILE_K)
    body = pk[: nt * kt * TILE_BYTES].view(np.uint32).reshape(nt, kt, 2, TILE_N, 4)
    words = np.transpose(body, (0, 3, 1, 2, 4)).reshape(nt, TILE_N, kt, 8).astype(np.uint64)
    shifts = (np.uint64(16) * np.arange(2, dtype=np.uint64)[None, :]
              + np.uint64(2) * np.arange(8, dtype=np.uint64)[:, None])
    u = (words[..., None, None] >> shifts) & np.uint64(3)                # [rt, r, kt, j, p, e]
    if np.any(u == 3):
        raise ValueError("invalid 2-bit code 3 in packed weights")
    T = u.astype(np.int64).reshape(nt * TILE_N, kt * TILE_K) - 1
    return T[:N, :K].astype(np.int8)


def read_trailer(pk: np.ndarray, N: int, K: int) -> tuple[int, int, int, int]:
    nt, kt = -(-N // TILE_N), -(-K // TILE_K)
    off = nt * kt * TILE_BYTES
    t = np.asarray(pk, dtype=np.uint8)[off: off + 16].view(np.uint32)
    return int(t[0]), int(t[1]), int(t[2]), int(t[3])
