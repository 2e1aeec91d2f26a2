// api.cu -- the C ABI (include/bitmtp_linear.h): argument validation, device
// checks, the width/shape dispatch table and the pack, absmean-ternarisation
// and activation-quantisation kernels.  The GEMM kernels live in gemm.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "internal.h"
#include "quant.cuh"
#include "ptx.cuh"

namespace bitmtp {

// Device error word: set by a kernel whose bounded wait expired.
__device__ int g_device_error = 0;

namespace {

constexpr uint32_t kTrailerMagic = 0x38413242u;

// ----------------------------------------------------------------- pack --
// Sources of ternary entries for the pack kernel: load16 gives the codes of
// entries k0..k0+15 of row n (zero beyond N or K).

// int8 T: entries outside {-1, 0, +1} are counted into `bad` and clamped.
struct Int8Source {
    const int8_t* T;
    long long ld;
    __device__ void load16(int n, int k0, int N, int K, int (&t)[16], int& bad) const {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const int k = k0 + kk;
            int v = 0;
            if (n < N && k < K) v = T[static_cast<long long>(n) * ld + k];
            if (v < -1 || v > 1) {
                ++bad;
                v = v < 0 ? -1 : 1;
            }
            t[kk] = v;
        }
    }
};

// fp32 W under the absmean scale g: clamp(round_half_even(RN(w / g)), -1, 1),
// computed without the division.  With g >= 1e-5 (a normal number) h = g / 2
// is exact, and the code is +1 exactly when w > h: for w = h the quotient is
// 0.5, which rounds (half to even) to 0; the next float above h, h + ulp(h),
// gives w / g = 0.5 + 2^-24 / m with m in [1, 2) the significand of h, which
// is above the rounding midpoint 0.5 + 2^-25 and so rounds to a float above
// 0.5, whose rint is at least 1; larger w only raise the quotient.  The
// negative side is the mirror image.
__device__ __forceinline__ int ternary_code(float w, float h) {
    return (w > h ? 1 : 0) - (w < -h ? 1 : 0);
}
// 16-byte load with an L2 eviction-priority hint.
__device__ __forceinline__ float4 ld_f4_hint(const float4* p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p), "l"(pol));
    return v;
}
struct F32Source {
    const float* W;
    long long ld;
    const float* g;  // device scalar written by absmean_finish_kernel
    bool vec;        // W 16-byte aligned and ld a multiple of 4: float4 loads
    __device__ void load16(int n, int k0, int N, int K, int (&t)[16], int&) const {
        const float gs = 0.5f * *g;  // exact: g is normal
        const float* row = W + static_cast<long long>(n) * ld;
        if (n < N && vec && k0 + 16 <= K) {
            // the second and last read of W (the absmean pass left it in L2)
            const uint64_t pol = policy_evict_first();
            const float4* p = reinterpret_cast<const float4*>(row + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = ld_f4_hint(p + i, pol);
                t[4 * i] = ternary_code(v.x, gs);
                t[4 * i + 1] = ternary_code(v.y, gs);
                t[4 * i + 2] = ternary_code(v.z, gs);
                t[4 * i + 3] = ternary_code(v.w, gs);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                t[kk] = (n < N && k0 + kk < K) ? ternary_code(row[k0 + kk], gs) : 0;
        }
    }
};

// One 4 KiB tile (row tile rt, k tile kt) by one block, four words a thread.
template <class Src>
__device__ __forceinline__ void pack_tile(const Src& src, int N, int K, int KT, int rt, int kt,
                                          uint32_t* __restrict__ pk, uint32_t* __restrict__ invalid) {
    uint32_t* tile = pk + (static_cast<size_t>(rt) * KT + kt) * (kTileBytes / 4);
    int bad = 0;
    for (int widx = threadIdx.x; widx < kTileBytes / 4; widx += blockDim.x) {
        const int half = widx >> 9;
        const int r = (widx & 511) >> 2;
        const int j = half * 4 + (widx & 3);
        int t[16];
        src.load16(rt * kTileN + r, kt * kTileK + 16 * j, N, K, t, bad);
        uint32_t word = 0;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            word |= static_cast<uint32_t>(t[kk] + 1) << (16 * (kk & 1) + 2 * (kk >> 1));
        tile[widx] = word;
    }
    // block-reduce the invalid count
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(invalid, static_cast<uint32_t>(bad));
}

// Grid (KT, NT): the int8 pack.
template <class Src>
__global__ void __launch_bounds__(256)
pack_kernel(Src src, int N, int K, int KT, uint32_t* __restrict__ pk, uint32_t* __restrict__ invalid) {
    pack_tile(src, N, K, KT, static_cast<int>(blockIdx.y), static_cast<int>(blockIdx.x), pk, invalid);
}

// A group of fp32 matrices to ternarise: per matrix its absmean blocks and
// pack tiles occupy consecutive ranges of the two grids.
struct TernMat {
    const float* W;
    long long ldw;
    int N, K, KT;
    int flat, vec;
    int blk_begin, blocks;  // absmean pass
    int tile_begin;         // pack pass: tiles tile_begin .. + NT * KT - 1
    uint32_t* pk;
    uint32_t* trailer;      // the packed buffer's last 16 bytes
    float* w_scale;
};
struct TernParams {
    TernMat m[BITMTP_MAX_GROUP];
    int n;
    unsigned long long* bins;  // [n][kHistBins]
    uint32_t* nonfinite;       // [n]
};

// --------------------------------------------------- absmean ternarisation --
// mean|W| is the exact sum of |W| rounded once to fp64, divided by the count
// in fp64 and rounded to fp32; no summation order enters.  An entry is
// m * 2^(e-150) with e = max(biased exponent, 1) and m its significand (the
// implicit bit included for normals).  Integer sums of such terms are exact
// and order-free:
// * each thread adds m << (e - b) into a 128-bit register accumulator, b
//   fixed by its first non-zero entry (b = e - 40, so exponents e - 40 ..
//   e + 23 fit; at most 2^22 entries per thread keep it below 2^110);
// * entries outside that window go to shared bins: bin j holds an integer
//   sum at scale 2^(j - kBinOff - 150), entry (m, e) into bin e + kBinOff;
// * at the end each thread adds its accumulator, in four 32-bit pieces, to
//   bins b + 32 i + kBinOff (i = 0..3), and each block adds its non-zero bins
//   into one global set of bins (zeroed by the host before the launch);
// * the common entries, |w| in [2^-14, 8), never reach the integer road: as
//   integers at the fixed scale 2^-37 they are summed exactly in fp32 pieces
//   (absmean_hist_kernel's add_fast) and added as two 32-bit pieces to bins
//   113 + kBinOff and 145 + kBinOff; the pass then runs on the
//   floating-point pipe instead of saturating the integer one.
// Bins 89..438 are the only ones used; bin 511 counts non-finite entries.  A
// bin stays below 2^39 * 2^24 + 2^17 * 2^32 < 2^64.
constexpr int kHistBins = 512;
constexpr int kBinOff = 128;
constexpr int kNonFiniteBin = 511;

// Blocks of the absmean pass for a matrix of N x K entries out of `total`
// entries in the group: the larger of its share of one full wave (per_sm
// resident blocks on every SM) and one block per 64 K entries up to
// a full wave; at least one, at most one per row on the row walk, and never
// fewer than keep a thread at or below 2^22 entries (the accumulator bound
// above).
int hist_blocks(int64_t N, int64_t K, int64_t total, bool flat, int sms, int per_sm) {
    const int64_t full = static_cast<int64_t>(std::max(per_sm, 1)) * std::max(sms, 1);
    const int64_t per_thread_max = static_cast<int64_t>(256) << 22;
    const int64_t min_blocks = (N * K + per_thread_max - 1) / per_thread_max;
    const int64_t share = (full * N * K + total - 1) / total;
    int64_t g = std::max<int64_t>(std::max<int64_t>(share, std::min<int64_t>(full, (N * K + 65535) / 65536)), 1);
    g = std::min<int64_t>(g, (N * K + 1023) / 1024);  // at least 4 entries a thread
    if (!flat) g = std::min<int64_t>(g, N);
    return static_cast<int>(std::max<int64_t>(std::max<int64_t>(g, min_blocks), 1));
}

// flat: W contiguous (ldw == K) and 16-byte aligned: a grid-stride walk over
// the whole matrix as float4, the last (N * K) % 4 entries one by one.
// Otherwise a grid-stride over rows; vec: rows 16-byte aligned (W aligned,
// ldw % 4 == 0), read as float4 with the row's last K % 4 entries one by
// one.  The loads ask L2 to keep W for the pack pass that reads it next.
__global__ void __launch_bounds__(256)
absmean_hist_kernel(const __grid_constant__ TernParams P) {
    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < P.n; ++i)
        if (static_cast<int>(blockIdx.x) >= P.m[i].blk_begin) mi = i;
    const TernMat& mt = P.m[mi];
    const float* __restrict__ W = mt.W;
    const long long ldw = mt.ldw;
    const int N = mt.N, K = mt.K;
    const bool flat = mt.flat != 0, vec = mt.vec != 0;
    const int blk = static_cast<int>(blockIdx.x) - mt.blk_begin;  // block within the matrix
    const int nblk = mt.blocks;
    unsigned long long* __restrict__ gbins = P.bins + static_cast<size_t>(mi) * kHistBins;
    __shared__ unsigned long long h[kHistBins];
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h[i] = 0ull;
    __syncthreads();
    unsigned long long acc_lo = 0ull, acc_hi = 0ull;
    int base = 0;
    bool have_base = false;
    auto add = [&](float w) {
        const uint32_t b = __float_as_uint(w) & 0x7FFFFFFFu;
        const int eb = static_cast<int>(b >> 23);
        if (eb == 255) {
            atomicAdd(&h[kNonFiniteBin], 1ull);
            return;
        }
        const unsigned long long m = (b & 0x7FFFFFu) | (eb ? 0x800000u : 0u);
        if (m == 0ull) return;
        const int e = eb ? eb : 1;
        if (!have_base) {
            base = e - 40;
            have_base = true;
        }
        const int d = e - base;
        if (d >= 0 && d < 64) {
            const unsigned long long lo = m << d;
            const unsigned long long hi = d > 40 ? (m >> (64 - d)) : 0ull;
            acc_lo += lo;
            acc_hi += hi + (acc_lo < lo ? 1ull : 0ull);
        } else {
            atomicAdd(&h[e + kBinOff], m);
        }
    };
    // The common entries, |w| in [2^-14, 8), on the floating-point pipe:
    // |w| * 2^37 = a * 2^20 + b exactly, with p = |w| * 2^17 (exact, below
    // 2^20), a = RN(p) (an integer, by adding and subtracting 1.5 * 2^23) and
    // b = (p - a) * 2^20 (p - a is exact by Sterbenz, as p >= 8, and a
    // multiple of 2^-20 in [-1/2, 1/2], so b is an integer of at most 2^19).
    // a and b are summed in fp32 over at most 16 entries (sums below 2^24 stay
    // exact), then flushed into 64-bit integers; sa * 2^20 + sb is the sum of
    // |w| * 2^37 over the thread's common entries.
    float fa = 0.f, fb = 0.f;
    unsigned long long sa = 0ull;
    long long sb = 0ll;
    auto add_fast = [&](float w) {
        const uint32_t bits = __float_as_uint(w) & 0x7FFFFFFFu;
        if (bits - 0x38800000u < 0x41000000u - 0x38800000u) {  // 2^-14 <= |w| < 8
            const float p = __fmul_rn(__uint_as_float(bits), 131072.f);
            const float a = __fadd_rn(__fadd_rn(p, 12582912.f), -12582912.f);
            fa = __fadd_rn(fa, a);
            fb = __fadd_rn(fb, __fmul_rn(__fadd_rn(p, -a), 1048576.f));
        } else if (bits != 0u) {  // zeros add nothing; the rest (NaN and inf too) as above
            add(w);
        }
    };
    auto flush = [&]() {  // at most 16 add_fast calls since the last flush
        sa += static_cast<unsigned long long>(__float2uint_rn(fa));
        sb += static_cast<long long>(__float2int_rn(fb));
        fa = 0.f;
        fb = 0.f;
    };
    const uint64_t pol = policy_evict_last();
    if (flat) {
        const long long total = static_cast<long long>(N) * K;
        const long long n4 = total / 4;
        const long long stride = static_cast<long long>(nblk) * blockDim.x;
        const long long first = static_cast<long long>(blk) * blockDim.x + threadIdx.x;
        const float4* W4 = reinterpret_cast<const float4*>(W);
        // four loads in flight before any of their entries is added (the
        // shared-memory atomics of the slow path would otherwise keep the
        // compiler from hoisting the next load above them)
        long long i = first;
        for (; i + 3 * stride < n4; i += 4 * stride) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = ld_f4_hint(W4 + i + u * stride, pol);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                add_fast(v[u].x);
                add_fast(v[u].y);
                add_fast(v[u].z);
                add_fast(v[u].w);
            }
            flush();
        }
        for (; i < n4; i += stride) {
            const float4 v = ld_f4_hint(W4 + i, pol);
            add_fast(v.x);
            add_fast(v.y);
            add_fast(v.z);
            add_fast(v.w);
            flush();
        }
        for (long long i1 = 4 * n4 + first; i1 < total; i1 += stride) add(W[i1]);
    } else {
        const int K4 = vec ? K / 4 : 0;
        for (int n = blk; n < N; n += nblk) {
            const float* row = W + static_cast<long long>(n) * ldw;
            const float4* row4 = reinterpret_cast<const float4*>(row);
            const int bd = static_cast<int>(blockDim.x);
            int k4 = threadIdx.x;
            for (; k4 + 3 * bd < K4; k4 += 4 * bd) {  // four loads in flight, as above
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = ld_f4_hint(row4 + k4 + u * bd, pol);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    add_fast(v[u].x);
                    add_fast(v[u].y);
                    add_fast(v[u].z);
                    add_fast(v[u].w);
                }
                flush();
            }
            for (; k4 < K4; k4 += bd) {
                const float4 v = ld_f4_hint(row4 + k4, pol);
                add_fast(v.x);
                add_fast(v.y);
                add_fast(v.z);
                add_fast(v.w);
                flush();
            }
            for (int k = 4 * K4 + threadIdx.x; k < K; k += blockDim.x) add(row[k]);
        }
    }
    {
        // the common entries' sum at the fixed scale 2^-37 (exponent 113),
        // non-negative and below 2^63, in two 32-bit pieces
        const unsigned long long fix = static_cast<unsigned long long>(static_cast<long long>(sa << 20) + sb);
        if (fix & 0xFFFFFFFFull) atomicAdd(&h[113 + kBinOff], fix & 0xFFFFFFFFull);
        if (fix >> 32) atomicAdd(&h[145 + kBinOff], fix >> 32);
    }
    if (have_base) {
        const unsigned long long piece[4] = {acc_lo & 0xFFFFFFFFull, acc_lo >> 32, acc_hi & 0xFFFFFFFFull, acc_hi >> 32};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (piece[i]) atomicAdd(&h[base + 32 * i + kBinOff], piece[i]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        if (h[i]) atomicAdd(&gbins[i], h[i]);
}

// 512-bit unsigned integer in 64-bit limbs, least significant first, in units
// of 2^-213: bin j adds at bit j - kBinOff - 150 + 213 = j - 65 (>= 24 for the
// bins in use; every bin below 511 fits, shift <= 445).
constexpr int kLimbs = 8;
constexpr int kUnitExp = -213;

// The limbs stay in registers: every limb index below is a compile-time
// constant (unrolled loops with predicates; a runtime index would move the
// array to local memory and make the one-thread sum ~10x slower).
__device__ __forceinline__ void wide_add_shifted(unsigned long long (&L)[kLimbs], unsigned long long v, int sh) {
    const int i = sh >> 6, o = sh & 63;  // sh <= 445: i + 1 < kLimbs
    const unsigned long long lo = v << o;
    const unsigned long long hi = o ? (v >> (64 - o)) : 0ull;
    unsigned long long carry = 0ull;
#pragma unroll
    for (int j = 0; j < kLimbs; ++j) {
        const unsigned long long add = (j == i) ? lo : (j == i + 1) ? hi : 0ull;
        const unsigned long long s1 = L[j] + add;
        const unsigned long long c1 = s1 < add ? 1ull : 0ull;
        const unsigned long long s2 = s1 + carry;
        const unsigned long long c2 = s2 < carry ? 1ull : 0ull;
        L[j] = (j >= i) ? s2 : L[j];
        carry = (j >= i) ? (c1 | c2) : 0ull;
    }
}

// L += R (two 512-bit integers; the sum fits, as every total here does).
__device__ __forceinline__ void wide_add(unsigned long long (&L)[kLimbs], const unsigned long long (&R)[kLimbs]) {
    unsigned long long carry = 0ull;
#pragma unroll
    for (int j = 0; j < kLimbs; ++j) {
        const unsigned long long s1 = L[j] + R[j];
        const unsigned long long c1 = s1 < R[j] ? 1ull : 0ull;
        const unsigned long long s2 = s1 + carry;
        const unsigned long long c2 = s2 < carry ? 1ull : 0ull;
        L[j] = s2;
        carry = c1 | c2;
    }
}

// 64 bits of L from bit pos (bits past the top read as 0).
__device__ __forceinline__ unsigned long long wide_bits(const unsigned long long (&L)[kLimbs], int pos) {
    const int i = pos >> 6, o = pos & 63;
    unsigned long long v = 0ull;
#pragma unroll
    for (int j = 0; j < kLimbs; ++j) {
        if (j == i) v |= L[j] >> o;
        if (j == i + 1 && o) v |= L[j] << (64 - o);
    }
    return v;
}

// L * 2^kUnitExp rounded to the nearest fp64, ties to even.
__device__ __forceinline__ double wide_to_double(const unsigned long long (&L)[kLimbs]) {
    int top = -1;
#pragma unroll
    for (int j = 0; j < kLimbs; ++j)
        if (L[j]) top = 64 * j + 63 - __clzll(static_cast<long long>(L[j]));
    if (top < 0) return 0.0;
    if (top < 53) return __dmul_rn(static_cast<double>(L[0]), 0x1p-213);  // exact (kUnitExp = -213)
    int lo = top - 52;  // the 53 bits [lo, top]
    unsigned long long mant = wide_bits(L, lo) & ((1ull << 53) - 1ull);
    const unsigned long long round = wide_bits(L, lo - 1) & 1ull;
    bool sticky = false;
    const int sb = lo - 1;  // bits [0, sb) below the round bit
#pragma unroll
    for (int j = 0; j < kLimbs; ++j) {
        const int b0 = 64 * j;
        if (b0 + 64 <= sb) sticky = sticky || L[j] != 0ull;
        else if (b0 < sb) sticky = sticky || (L[j] & ((1ull << (sb - b0)) - 1ull)) != 0ull;
    }
    if (round && (sticky || (mant & 1ull))) {
        ++mant;
        if (mant == (1ull << 53)) {
            mant >>= 1;
            ++lo;
        }
    }
    // mant * 2^(lo + kUnitExp), a normal fp64 (mant has its top bit at 52):
    // biased exponent lo + kUnitExp + 52 + 1023, fraction the low 52 bits
    const long long bexp = static_cast<long long>(lo + kUnitExp + 52 + 1023);
    return __longlong_as_double(static_cast<long long>((static_cast<unsigned long long>(bexp) << 52) |
                                                       (mant & ((1ull << 52) - 1ull))));
}

// One block of kHistBins threads: the exact sum from the global bins (warp 0:
// each lane adds every 32nd bin into its own 512-bit integer, then a shuffle
// tree adds the 32 partial sums; integer additions, so the order is free),
// gamma = max(RN32(RN64(sum) / count), 1e-5) into *w_scale, the non-finite
// flag, and the packed buffer's trailer {magic, N, K, 0}.
__global__ void __launch_bounds__(kHistBins)
absmean_finish_kernel(const __grid_constant__ TernParams P) {
    const int mi = static_cast<int>(blockIdx.x);
    const TernMat& mt = P.m[mi];
    const int N = mt.N, K = mt.K;
    uint32_t* __restrict__ trailer = mt.trailer;
    __shared__ unsigned long long H[kHistBins];
    const int e = threadIdx.x;
    H[e] = P.bins[static_cast<size_t>(mi) * kHistBins + e];
    __syncthreads();
    if (e >= 32) return;
    unsigned long long L[kLimbs] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
    for (int j = 65 + e; j < kNonFiniteBin; j += 32)
        if (H[j]) wide_add_shifted(L, H[j], j - 65);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        unsigned long long R[kLimbs];
#pragma unroll
        for (int k = 0; k < kLimbs; ++k) R[k] = __shfl_down_sync(0xffffffffu, L[k], off);
        if (e < off) wide_add(L, R);
    }
    if (e == 0) {
        const long long count = static_cast<long long>(N) * K;
        const double mean = __ddiv_rn(wide_to_double(L), static_cast<double>(count));
        *mt.w_scale = fmaxf(__double2float_rn(mean), 1e-5f);
        P.nonfinite[mi] = H[kNonFiniteBin] ? 1u : 0u;
        trailer[0] = kTrailerMagic;
        trailer[1] = static_cast<uint32_t>(N);
        trailer[2] = static_cast<uint32_t>(K);
        trailer[3] = 0u;
    }
}

// The fp32 pack of every tile of the group: block b is tile b - tile_begin of
// the matrix holding it.
__global__ void __launch_bounds__(256)
tern_pack_kernel(const __grid_constant__ TernParams P) {
    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < P.n; ++i)
        if (static_cast<int>(blockIdx.x) >= P.m[i].tile_begin) mi = i;
    const TernMat& mt = P.m[mi];
    const int t = static_cast<int>(blockIdx.x) - mt.tile_begin;
    pack_tile(F32Source{mt.W, mt.ldw, mt.w_scale, mt.vec != 0}, mt.N, mt.K, mt.KT, t / mt.KT, t % mt.KT, mt.pk,
              mt.trailer + 3);
}

// ------------------------------------------------------------ quant_act --
// One block per activation row.
__global__ void __launch_bounds__(256)
quant_act_kernel(const void* __restrict__ x, int kind, int K, long long ldx, int8_t* __restrict__ q,
                 long long ldq, float* __restrict__ a_scale, int32_t* __restrict__ rowsum) {
    __shared__ float red_f[8];
    __shared__ int red_i[8];
    const int m = blockIdx.x;
    const int tid = threadIdx.x;
    const long long xo = static_cast<long long>(m) * ldx;
    float a = 0.f;
    for (int k = tid; k < K; k += blockDim.x) a = fmaxf(a, fabsf(load_act(x, kind, xo + k)));
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((tid & 31) == 0) red_f[tid >> 5] = a;
    __syncthreads();
    float amax = red_f[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) amax = fmaxf(amax, red_f[w]);
    const float s = quant_scale(amax);
    int sum = 0;
    const long long qo = static_cast<long long>(m) * ldq;
    for (int k = tid; k < K; k += blockDim.x) {
        const int v = (amax > 0.f) ? quantize(load_act(x, kind, xo + k), s) : 0;
        q[qo + k] = static_cast<int8_t>(v);
        sum += v;
    }
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((tid & 31) == 0) red_i[tid >> 5] = sum;
    __syncthreads();
    if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red_i[w];
        a_scale[m] = dequant_scale(amax);
        if (rowsum) rowsum[m] = tot;
    }
}

// ------------------------------------------------------------- device --
// Per-device facts, looked up once per device: the first caller fills them
// and publishes `state` with release order; later callers read it with
// acquire order (concurrent first callers only repeat the same queries).
struct DevInfo {
    std::atomic<int> state{0};   // 0 unknown, 1 ok, -1 unsupported
    int sms = 0;
    int hist_per_sm = 1;         // resident absmean-pass blocks per SM (its register use decides)
    int* err = nullptr;
    std::atomic<int> dirty{0};   // the no-alloc scratch may hold flags of a launch that gave up
};
DevInfo g_dev[64];

int current_device(DevInfo** info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return BITMTP_ERR_UNSUPPORTED;
    }
    if (dev >= 64) return BITMTP_ERR_UNSUPPORTED;
    DevInfo& d = g_dev[dev];
    int st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return BITMTP_ERR_UNSUPPORTED;
        }
        if (major != 10 || minor != 3) {
            st = -1;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
                cudaGetLastError();
                return BITMTP_ERR_CUDA;
            }
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, absmean_hist_kernel, 256, 0) != cudaSuccess) {
                cudaGetLastError();
                return BITMTP_ERR_CUDA;
            }
            d.err = static_cast<int*>(p);
            d.sms = sms;
            d.hist_per_sm = std::max(per_sm, 1);
            st = 1;
        }
        d.state.store(st, std::memory_order_release);
    }
    if (st != 1) return BITMTP_ERR_UNSUPPORTED;
    *info = &d;
    return BITMTP_OK;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return BITMTP_OK;
    cudaGetLastError();
    return BITMTP_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validate one GEMM problem and fill its kernel descriptor (no CUDA calls).
int check_problem(const void* pk, float w_scale, int64_t N, int64_t K, int64_t M,
                  const bitmtp_act* act, const bitmtp_out* out, GemmProblem* g) {
    if (!act || !out) return BITMTP_ERR_INVALID;
    if (M < 0 || M > BITMTP_MAX_M || N < 0 || N > BITMTP_MAX_N || K < 1 || K > BITMTP_MAX_K)
        return BITMTP_ERR_SHAPE;
    if (M == 0 || N == 0) {
        g->M = 0;
        g->N = 0;
        return BITMTP_OK;
    }
    if (!pk) return BITMTP_ERR_INVALID;
    if (!aligned16(pk)) return BITMTP_ERR_ALIGN;
    if (act->kind != BITMTP_F32 && act->kind != BITMTP_BF16 && act->kind != BITMTP_Q8)
        return BITMTP_ERR_INVALID;
    if (!act->x || act->ldx < K) return BITMTP_ERR_INVALID;
    if (act->kind == BITMTP_Q8 && !act->a_scale) return BITMTP_ERR_INVALID;
    if (out->dtype != BITMTP_F32 && out->dtype != BITMTP_BF16) return BITMTP_ERR_INVALID;
    if (!out->y || out->ldy < N) return BITMTP_ERR_INVALID;
    if (out->acc && out->lda < N) return BITMTP_ERR_INVALID;
    if (!(w_scale == w_scale)) return BITMTP_ERR_INVALID;  // NaN scale
    g->pk = static_cast<const uint8_t*>(pk);
    g->x = act->x;
    g->a_scale_in = act->a_scale;
    g->y = out->y;
    g->acc = out->acc;
    g->ldx = act->ldx;
    g->ldy = out->ldy;
    g->lda = out->acc ? out->lda : 0;
    g->w_scale = w_scale;
    g->N = static_cast<int>(N);
    g->K = static_cast<int>(K);
    g->M = static_cast<int>(M);
    g->nt = static_cast<int>(ceil_div(N, kTileN));
    g->kt = static_cast<int>(ceil_div(K, kTileK));
    g->act_kind = act->kind;
    g->out_dtype = out->dtype;
    g->amax_in = act->kind == BITMTP_Q8 ? nullptr : act->amax;
    g->amax_out = out->amax;
    const int64_t esize = act->kind == BITMTP_F32 ? 4 : (act->kind == BITMTP_BF16 ? 2 : 1);
    g->vec_ok = (aligned16(act->x) && (act->ldx * esize) % 16 == 0) ? 1 : 0;
    return BITMTP_OK;
}

// Width-specialised operator choice (the analogue of picking packed low-bit
// operators by replay width and input/output dimensions), from measured call
// times on GB300: dp4a up to four rows, tensor cores with an 8-row activation
// tile up to 8 rows, 16 rows above.
int choose_path(int max_m, unsigned flags, int* dp_rows) {
    const int r = max_m <= 1 ? 1 : (max_m <= 2 ? 2 : 4);
    if (flags & BITMTP_FLAG_FP8) {  // every width on the FP8 tensor path
        *dp_rows = 1;
        return (flags & BITMTP_FLAG_FORCE_DP) ? -1 : kPathF8;
    }
    if (flags & BITMTP_FLAG_FORCE_DP) {
        if (max_m > 4) return -1;
        *dp_rows = r;
        return kPathDP;
    }
    if (!(flags & BITMTP_FLAG_FORCE_TC) && max_m <= 4) {
        *dp_rows = r;
        return kPathDP;
    }
    return max_m <= 8 ? kPathTC8 : kPathTC16;
}



// The flag combinations a call accepts: not both forced paths; FP8
// activations only from raw rows, and not on the dp4a path.
int check_flags(const GemmProblem* g, int n, unsigned flags) {
    if ((flags & BITMTP_FLAG_FORCE_TC) && (flags & BITMTP_FLAG_FORCE_DP)) return BITMTP_ERR_INVALID;
    if (flags & BITMTP_FLAG_FP8) {
        if (flags & BITMTP_FLAG_FORCE_DP) return BITMTP_ERR_INVALID;
        for (int i = 0; i < n; ++i)
            if (g[i].M > 0 && g[i].act_kind == BITMTP_Q8) return BITMTP_ERR_INVALID;
    }
    return BITMTP_OK;
}

int run_gemms(const GemmProblem* probs, int n, void* workspace, size_t ws_bytes, unsigned flags,
              cudaStream_t stream) {
    bool any = false;
    for (int i = 0; i < n; ++i) any = any || (probs[i].M > 0 && probs[i].N > 0);
    if (!any) return BITMTP_OK;  // empty problems never touch the device
    if (!workspace) return BITMTP_ERR_INVALID;
    if (!aligned16(workspace)) return BITMTP_ERR_ALIGN;
    size_t need = kWsAct;
    for (int i = 0; i < n; ++i)
        if (probs[i].M > 0 && probs[i].N > 0) need += act_region_bytes(probs[i].kt);
    if (ws_bytes < need) return BITMTP_ERR_SHAPE;
    DevInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != BITMTP_OK) return st;

    GemmParams prm;
    std::memset(&prm, 0, sizeof(prm));
    uint8_t* w = static_cast<uint8_t*>(workspace);
    size_t act_off = kWsAct;
    long long tiles = 0;
    int max_m = 1, np = 0;
    for (int i = 0; i < n; ++i) {
        if (probs[i].M == 0 || probs[i].N == 0) continue;
        GemmProblem g = probs[i];
        g.actb = w + act_off;
        g.rsp = reinterpret_cast<int*>(w + act_off + act_tiles_bytes(g.kt));
        g.asc = reinterpret_cast<float*>(w + act_off + act_tiles_bytes(g.kt) + act_rsp_bytes(g.kt));
        act_off += act_region_bytes(g.kt);
        g.tile_begin = tiles;
        tiles += static_cast<long long>(g.nt) * g.kt;
        max_m = std::max(max_m, g.M);
        prm.p[np++] = g;
    }
    int dp_rows = 1;
    const int path = choose_path(max_m, flags, &dp_rows);
    if (path < 0) return BITMTP_ERR_SHAPE;
    const long long cap = std::min(kMaxCtas, kCtasPerSm * dev->sms);
    prm.n_problems = np;
    prm.stages = gemm_stages(path, dp_rows);
    prm.total_tiles = tiles;
    // every CTA range is non-empty (nctas <= tiles) and, where the problem is
    // large enough, at least kMinTilesPerCta long
    prm.nctas = static_cast<int>(std::max(1ll, std::min(cap, (tiles + kMinTilesPerCta - 1) / kMinTilesPerCta)));
    prm.tiles_q = static_cast<int>(tiles / prm.nctas);
    prm.tiles_r = static_cast<int>(tiles % prm.nctas);
    prm.flags = reinterpret_cast<unsigned*>(w + kWsFlags);
    prm.slots = reinterpret_cast<int*>(w + kWsSlots);
    prm.err = dev->err;
    // a layer chain on the dp4a path: every live problem brings its rows'
    // absmax, so the GEMM quantises its own activation tiles (no preparation
    // launch); the workspace's first two words order the out.amax zeroing
    bool fused = path == kPathDP, any_amax_out = false;
    for (int i = 0; i < np; ++i) {
        fused = fused && prm.p[i].act_kind != BITMTP_Q8 && prm.p[i].amax_in != nullptr;
        any_amax_out = any_amax_out || prm.p[i].amax_out != nullptr;
    }
    prm.fused = fused ? 1 : 0;
    prm.sync_words = (fused && any_amax_out) ? reinterpret_cast<unsigned*>(w) : nullptr;
    const bool test_withhold = (flags & BITMTP_FLAG_TEST_WITHHOLD) != 0;
    prm.withhold = test_withhold ? 0 : -1;
    prm.wait_ns = test_withhold ? kTestWaitNs : kWaitNs;
    return cuda_status(launch_gemm(prm, path, dp_rows, (flags & BITMTP_FLAG_PDL) != 0, stream));
}

// ------------------------------------------------- no-allocation variant --
// Built-in scratch of bitmtp_linear_gemm_noalloc, laid out like a caller's
// workspace.  Host code must not pass the symbol itself to a kernel: on the
// host it names a stand-in, not device memory.  Its device address is looked
// up once per device (with that device current) and kept here.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BITMTP_NOALLOC_SCRATCH_BYTES];
static_assert(kWsAct + act_region_bytes(BITMTP_MAX_K / kTileK) <= BITMTP_NOALLOC_SCRATCH_BYTES,
              "built-in scratch smaller than the workspace of the largest single problem");

std::atomic<void*> g_noalloc_addr[64];

int noalloc_scratch(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return BITMTP_ERR_UNSUPPORTED;
    }
    void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        // two threads racing here both obtain the same address
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return BITMTP_ERR_CUDA;
        }
        g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return BITMTP_OK;
}

}  // namespace
}  // namespace bitmtp

using namespace bitmtp;

extern "C" {

size_t bitmtp_linear_packed_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1 || N > BITMTP_MAX_N || K > BITMTP_MAX_K) return 0;
    return static_cast<size_t>(ceil_div(N, kTileN)) * static_cast<size_t>(ceil_div(K, kTileK)) * kTileBytes + 16;
}

int bitmtp_linear_pack(const int8_t* T, int64_t N, int64_t K, int64_t ldt, void* pk, size_t pk_bytes,
                       void* stream) {
    if (N < 1 || K < 1 || N > BITMTP_MAX_N || K > BITMTP_MAX_K) return BITMTP_ERR_SHAPE;
    if (!T || !pk || ldt < K) return BITMTP_ERR_INVALID;
    if (!aligned16(pk)) return BITMTP_ERR_ALIGN;
    const size_t need = bitmtp_linear_packed_bytes(N, K);
    if (pk_bytes < need) return BITMTP_ERR_SHAPE;
    DevInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != BITMTP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int NT = static_cast<int>(ceil_div(N, kTileN));
    const int KT = static_cast<int>(ceil_div(K, kTileK));
    uint8_t* base = static_cast<uint8_t*>(pk);
    uint32_t* trailer = reinterpret_cast<uint32_t*>(base + need - 16);
    const uint32_t head[4] = {kTrailerMagic, static_cast<uint32_t>(N), static_cast<uint32_t>(K), 0u};
    st = cuda_status(cudaMemcpyAsync(trailer, head, sizeof(head), cudaMemcpyHostToDevice, s));
    if (st != BITMTP_OK) return st;
    pack_kernel<Int8Source><<<dim3(KT, NT), 256, 0, s>>>(Int8Source{T, ldt}, static_cast<int>(N),
                                                         static_cast<int>(K), KT,
                                                         reinterpret_cast<uint32_t*>(base), trailer + 3);
    st = cuda_status(cudaGetLastError());
    if (st != BITMTP_OK) return st;
    uint32_t invalid = 0;
    st = cuda_status(cudaMemcpyAsync(&invalid, trailer + 3, 4, cudaMemcpyDeviceToHost, s));
    if (st != BITMTP_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != BITMTP_OK) return st;
    return invalid ? BITMTP_ERR_NOT_TERNARY : BITMTP_OK;
}

size_t bitmtp_linear_ternarize_workspace_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1 || N > BITMTP_MAX_N || K > BITMTP_MAX_K) return 0;
    return bitmtp_linear_ternarize_workspace_bytes_grouped(1);
}

size_t bitmtp_linear_ternarize_workspace_bytes_grouped(int n_desc) {
    if (n_desc < 1 || n_desc > BITMTP_MAX_GROUP) return 0;
    // the bins of each matrix, then one non-finite flag per matrix
    return static_cast<size_t>(n_desc) * kHistBins * sizeof(unsigned long long) + 256;
}

int bitmtp_linear_ternarize_pack_grouped(const bitmtp_ternarize_desc* d, int n_desc, void* workspace,
                                         size_t ws_bytes, void* stream) {
    if (!d || n_desc < 1 || n_desc > BITMTP_MAX_GROUP) return BITMTP_ERR_INVALID;
    if (!workspace) return BITMTP_ERR_INVALID;
    if (!aligned16(workspace)) return BITMTP_ERR_ALIGN;
    if (ws_bytes < bitmtp_linear_ternarize_workspace_bytes_grouped(n_desc)) return BITMTP_ERR_SHAPE;
    for (int i = 0; i < n_desc; ++i) {  // every argument check before any CUDA call
        const bitmtp_ternarize_desc& g = d[i];
        if (g.N < 1 || g.K < 1 || g.N > BITMTP_MAX_N || g.K > BITMTP_MAX_K) return BITMTP_ERR_SHAPE;
        if (!g.W || !g.pk || !g.w_scale || g.ldw < g.K) return BITMTP_ERR_INVALID;
        if (!aligned16(g.pk)) return BITMTP_ERR_ALIGN;
        if (g.pk_bytes < bitmtp_linear_packed_bytes(g.N, g.K)) return BITMTP_ERR_SHAPE;
    }
    DevInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != BITMTP_OK) return st;
    TernParams P;
    std::memset(&P, 0, sizeof(P));
    P.n = n_desc;
    P.bins = static_cast<unsigned long long*>(workspace);
    P.nonfinite = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) +
                                              static_cast<size_t>(n_desc) * kHistBins * sizeof(unsigned long long));
    long long blocks = 0, tiles = 0, total = 0;
    for (int i = 0; i < n_desc; ++i) total += d[i].N * d[i].K;
    for (int i = 0; i < n_desc; ++i) {
        const bitmtp_ternarize_desc& g = d[i];
        const size_t need = bitmtp_linear_packed_bytes(g.N, g.K);
        TernMat& m = P.m[i];
        m.W = g.W;
        m.ldw = g.ldw;
        m.N = static_cast<int>(g.N);
        m.K = static_cast<int>(g.K);
        m.KT = static_cast<int>(ceil_div(g.K, kTileK));
        m.vec = aligned16(g.W) && (g.ldw % 4) == 0;
        m.flat = aligned16(g.W) && g.ldw == g.K;
        m.blk_begin = static_cast<int>(blocks);
        m.blocks = hist_blocks(g.N, g.K, total, m.flat != 0, dev->sms, dev->hist_per_sm);
        m.tile_begin = static_cast<int>(tiles);
        m.pk = static_cast<uint32_t*>(g.pk);
        m.trailer = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(g.pk) + need - 16);
        m.w_scale = g.w_scale;
        blocks += m.blocks;
        tiles += ceil_div(g.N, kTileN) * m.KT;
        if (blocks > INT32_MAX || tiles > INT32_MAX) return BITMTP_ERR_SHAPE;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = cuda_status(cudaMemsetAsync(workspace, 0, bitmtp_linear_ternarize_workspace_bytes_grouped(n_desc), s));
    if (st != BITMTP_OK) return st;
    absmean_hist_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(P);
    st = cuda_status(cudaGetLastError());
    if (st != BITMTP_OK) return st;
    absmean_finish_kernel<<<n_desc, kHistBins, 0, s>>>(P);
    st = cuda_status(cudaGetLastError());
    if (st != BITMTP_OK) return st;
    tern_pack_kernel<<<static_cast<unsigned>(tiles), 256, 0, s>>>(P);
    st = cuda_status(cudaGetLastError());
    if (st != BITMTP_OK) return st;
    uint32_t bad[BITMTP_MAX_GROUP] = {0};
    st = cuda_status(cudaMemcpyAsync(bad, P.nonfinite, sizeof(uint32_t) * n_desc, cudaMemcpyDeviceToHost, s));
    if (st != BITMTP_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != BITMTP_OK) return st;
    for (int i = 0; i < n_desc; ++i)
        if (bad[i]) return BITMTP_ERR_NOT_FINITE;
    return BITMTP_OK;
}

int bitmtp_linear_ternarize_pack(const float* W, int64_t N, int64_t K, int64_t ldw, void* pk, size_t pk_bytes,
                                 float* w_scale, void* workspace, size_t ws_bytes, void* stream) {
    if (N < 1 || K < 1 || N > BITMTP_MAX_N || K > BITMTP_MAX_K) return BITMTP_ERR_SHAPE;
    if (!W || !pk || !w_scale || !workspace || ldw < K) return BITMTP_ERR_INVALID;
    if (!aligned16(pk) || !aligned16(workspace)) return BITMTP_ERR_ALIGN;
    if (pk_bytes < bitmtp_linear_packed_bytes(N, K) || ws_bytes < bitmtp_linear_ternarize_workspace_bytes(N, K))
        return BITMTP_ERR_SHAPE;
    const bitmtp_ternarize_desc d = {W, N, K, ldw, pk, pk_bytes, w_scale};
    return bitmtp_linear_ternarize_pack_grouped(&d, 1, workspace, ws_bytes, stream);
}

int bitmtp_linear_quant_act(const void* x, int x_kind, int64_t M, int64_t K, int64_t ldx, int8_t* q,
                            int64_t ldq, float* a_scale, int32_t* rowsum, void* stream) {
    if (M < 0 || M > (1 << 20) || K < 1 || K > BITMTP_MAX_K) return BITMTP_ERR_SHAPE;
    if (x_kind != BITMTP_F32 && x_kind != BITMTP_BF16) return BITMTP_ERR_INVALID;
    if (M == 0) return BITMTP_OK;
    if (!x || !q || !a_scale || ldx < K || ldq < K) return BITMTP_ERR_INVALID;
    DevInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != BITMTP_OK) return st;
    quant_act_kernel<<<static_cast<unsigned>(M), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        x, x_kind, static_cast<int>(K), ldx, q, ldq, a_scale, rowsum);
    return cuda_status(cudaGetLastError());
}

size_t bitmtp_linear_workspace_bytes(int64_t N, int64_t K, int64_t M) {
    if (M < 1 || M > BITMTP_MAX_M || N < 1 || N > BITMTP_MAX_N || K < 1 || K > BITMTP_MAX_K) return 0;
    return kWsAct + act_region_bytes(static_cast<int>(ceil_div(K, kTileK)));
}

size_t bitmtp_linear_workspace_bytes_grouped(const bitmtp_gemm_desc* d, int n_desc) {
    if (n_desc < 1 || n_desc > BITMTP_MAX_GROUP || !d) return 0;
    for (int i = 0; i < n_desc; ++i) {
        const int64_t N = d[i].N, K = d[i].K, M = d[i].M;
        if (M < 0 || M > BITMTP_MAX_M || N < 0 || N > BITMTP_MAX_N || K < 1 || K > BITMTP_MAX_K) return 0;
    }
    size_t need = kWsAct;
    for (int i = 0; i < n_desc; ++i) need += act_region_bytes(static_cast<int>(ceil_div(d[i].K, kTileK)));
    return need;
}

int bitmtp_linear_gemm(const void* pk, float w_scale, int64_t N, int64_t K, int64_t M, const bitmtp_act* act,
                       const bitmtp_out* out, void* workspace, size_t workspace_bytes, unsigned flags,
                       void* stream) {
    GemmProblem g;
    std::memset(&g, 0, sizeof(g));
    int st = check_problem(pk, w_scale, N, K, M, act, out, &g);
    if (st != BITMTP_OK) return st;
    st = check_flags(&g, 1, flags);
    if (st != BITMTP_OK) return st;
    if (g.M == 0) return BITMTP_OK;
    return run_gemms(&g, 1, workspace, workspace_bytes, flags, static_cast<cudaStream_t>(stream));
}

int bitmtp_linear_gemm_grouped(const bitmtp_gemm_desc* d, int n_desc, void* workspace, size_t workspace_bytes,
                               unsigned flags, void* stream) {
    if (n_desc < 0 || n_desc > BITMTP_MAX_GROUP) return BITMTP_ERR_SHAPE;
    if (n_desc > 0 && !d) return BITMTP_ERR_INVALID;
    if ((flags & BITMTP_FLAG_FORCE_TC) && (flags & BITMTP_FLAG_FORCE_DP)) return BITMTP_ERR_INVALID;
    GemmProblem g[BITMTP_MAX_GROUP];
    std::memset(g, 0, sizeof(g));
    for (int i = 0; i < n_desc; ++i) {
        int st = check_problem(d[i].pk, d[i].w_scale, d[i].N, d[i].K, d[i].M, &d[i].act, &d[i].out, &g[i]);
        if (st != BITMTP_OK) return st;
    }
    const int fst = check_flags(g, n_desc, flags);
    if (fst != BITMTP_OK) return fst;
    if (n_desc == 0) return BITMTP_OK;
    return run_gemms(g, n_desc, workspace, workspace_bytes, flags, static_cast<cudaStream_t>(stream));
}

int bitmtp_linear_gemm_noalloc(const void* pk, float w_scale, int64_t N, int64_t K, int64_t M,
                               const bitmtp_act* act, const bitmtp_out* out, unsigned flags, void* stream) {
    GemmProblem g;
    std::memset(&g, 0, sizeof(g));
    int st = check_problem(pk, w_scale, N, K, M, act, out, &g);
    if (st != BITMTP_OK) return st;
    st = check_flags(&g, 1, flags);
    if (st != BITMTP_OK) return st;
    if (g.M == 0) return BITMTP_OK;
    const size_t need = bitmtp_linear_workspace_bytes(N, K, M);
    if (need == 0 || need > BITMTP_NOALLOC_SCRATCH_BYTES) return BITMTP_ERR_SHAPE;
    int dp_rows = 1;
    if (choose_path(g.M, flags, &dp_rows) < 0) return BITMTP_ERR_SHAPE;  // before anything is enqueued
    DevInfo* dev = nullptr;
    st = current_device(&dev);
    if (st != BITMTP_OK) return st;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != BITMTP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The sync words and flags must start at zero.  The array starts zeroed
    // and every launch leaves them at zero, except one that gave up a bounded
    // wait: once bitmtp_linear_device_error has reported that, the next call
    // clears them.
    if (dev->dirty.exchange(0, std::memory_order_acq_rel) != 0) {
        st = cuda_status(cudaMemsetAsync(scratch, 0, kWsSlots, s));
        if (st != BITMTP_OK) {
            dev->dirty.store(1, std::memory_order_release);
            return st;
        }
    }
    return run_gemms(&g, 1, scratch, BITMTP_NOALLOC_SCRATCH_BYTES, flags, s);
}

int bitmtp_linear_device_error(void* stream) {
    DevInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != BITMTP_OK) return st;
    st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    if (st != BITMTP_OK) return st;
    int v = 0;
    st = cuda_status(cudaMemcpy(&v, dev->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (st != BITMTP_OK) return st;
    if (v != 0) {
        dev->dirty.store(1, std::memory_order_release);
        const int zero = 0;
        st = cuda_status(cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice));
        if (st != BITMTP_OK) return st;
    }
    return v;
}

const char* bitmtp_linear_status_string(int status) {
    switch (status) {
        case BITMTP_OK: return "BITMTP_OK";
        case BITMTP_ERR_INVALID: return "BITMTP_ERR_INVALID: invalid argument";
        case BITMTP_ERR_ALIGN: return "BITMTP_ERR_ALIGN: packed weights must be 16-byte aligned";
        case BITMTP_ERR_SHAPE: return "BITMTP_ERR_SHAPE: dimension out of the supported range";
        case BITMTP_ERR_NOT_TERNARY: return "BITMTP_ERR_NOT_TERNARY: weight entry outside {-1,0,+1}";
        case BITMTP_ERR_UNSUPPORTED: return "BITMTP_ERR_UNSUPPORTED: no sm_103 device is current";
        case BITMTP_ERR_CUDA: return "BITMTP_ERR_CUDA: a CUDA runtime call failed";
        case BITMTP_ERR_DEVICE: return "BITMTP_ERR_DEVICE: a kernel gave up a bounded wait";
        case BITMTP_ERR_NOT_FINITE: return "BITMTP_ERR_NOT_FINITE: a weight is NaN or infinite";
        default: return "BITMTP: unknown status";
    }
}

int bitmtp_linear_version(void) { return 0x000100; }

}  // extern "C"
