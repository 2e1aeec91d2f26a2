// quant.cuh -- the per-row absmax int8 quantiser, shared by the standalone
// quantisation kernel and the GEMM prologue so both give identical codes.
//
// Per row: amax = max|x|; s = RN(127 / amax); q = clamp(rint(RN(x * s)), -127, 127)
// (fp32, round half to even); a_scale = RN(amax / 127); zero row -> q = 0,
// a_scale = 0.  (BitNet b1.58 activation quantiser: the W2A8 setting's 8-bit
// activations, "BitMTP ..." AI summary, Main Findings.)
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace bitmtp {

__device__ __forceinline__ float load_act(const void* x, int kind, long long idx) {
    if (kind == BITMTP_F32) return static_cast<const float*>(x)[idx];
    const uint16_t b = static_cast<const uint16_t*>(x)[idx];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);  // exact bf16 widening
}

__device__ __forceinline__ float quant_scale(float amax) {
    return amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
}
__device__ __forceinline__ float dequant_scale(float amax) {
    return amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
}
// FP8 (E4M3) activations: the same steps with the largest finite E4M3 value,
// 448, in place of 127.
__device__ __forceinline__ float fp8_quant_scale(float amax) {
    return amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
}
__device__ __forceinline__ float fp8_dequant_scale(float amax) {
    return amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
}
__device__ __forceinline__ int quantize(float v, float s) {
    int q = __float2int_rn(__fmul_rn(v, s));
    return max(-127, min(127, q));
}

}  // namespace bitmtp
