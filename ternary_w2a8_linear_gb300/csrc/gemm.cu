// gemm.cu -- the W2A8 ternary linear on sm_103a: an activation-operand
// preparation kernel followed by a persistent, warp-specialised stream-K GEMM.
//
// Two launches per call, chained by programmatic dependent launch (PDL):
//
//   act_prep_kernel   one CTA per (problem, activation row): the row's absmax
//                     and int8 codes (the quantiser of the standalone kernel,
//                     the same fp32 operations), written once into the
//                     workspace as the GEMM's activation operand -- one tile
//                     per k tile, in the layout the compute path reads --
//                     with prefix sums over k tiles of the row's codes and the
//                     row's dequant scale.
//
//   w2a8_streamk_kernel  the flattened (problem, row tile, k tile) space is
//                     split into equal contiguous ranges, one per CTA
//                     (stream-K), so every SM streams the same number of
//                     weight bytes whatever the mix of shapes.  Each CTA:
//     warp 4      bulk copies (TMA engine) into a ring of chunks of four
//                 tiles: weight tiles first -- they do not depend on the
//                 preparation kernel, so they are requested before the PDL
//                 wait -- and, after it, the matching activation tiles; each
//                 contiguous run is one copy (the engine's cost is per copy);
//     warps 0-3   one output row per thread: the compute path (below), then
//                 the epilogue -- a whole row tile is dequantised and written
//                 straight away; a row tile split between CTAs is finished by
//                 the last contributor, which sums the others' int32 partials
//                 from the workspace;
//     warp 5      (tensor path) issues tcgen05.mma.
//
// Compute paths (the same 2-bit code words feed both):
//   tensor (kPathTC16 / kPathTC8): each thread turns its code words into fp16
//     bit patterns with one mask per register -- the 2-bit code u lands in the
//     fp16 subnormal range, value u * 4^J * 2^-24 -- and writes them to tensor
//     memory as the A operand (tcgen05.st, seven buffers in flight); one thread
//     issues tcgen05.mma kind::f16 (M=128, N=16, K=16) against the activation
//     tile in shared memory, whose fp16 entries are q * 2^(9-2J).  Every
//     product is u*q*2^-15 and every partial sum an integer multiple of 2^-15
//     below 2^9, so the fp32 accumulator is exact in any order.  kPathTC8 keeps
//     8 activation rows (the second row group aliases the first through a zero
//     stride).
//   dp4a (kPathDP): four byte masks per code word, four int32 accumulators
//     per row (scales 4^s, recombined with exact shifts).
// With u = T + 1, sum_k T*q = sum_k u*q - sum_k q; the second sum comes from
// the preparation kernel's prefix sums.
//
// The operation is the packed W2A8 linear of "BitMTP: When Multi-Token
// Prediction Meets Low-Bit Large Language Models" (AI summary: Main Findings,
// first bullet -- 2-bit weights, 8-bit activations; Methodology in Plain
// English -- width-specialised packed low-bit operators, role-dependent output
// projections).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace bitmtp {
namespace {

constexpr int kChunk = 4;            // k tiles per ring chunk (16 KiB of weights)
constexpr int kMaxRing = 6;          // chunks in the ring (upper bound)
constexpr int kCtrlBytes = 1024;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccCol = 0;      // D: 16 fp32 columns, one per activation row
constexpr uint32_t kACol = 32;       // A: kABufs buffers of 32 columns (64 k each)
constexpr int kABufs = 7;
constexpr uint32_t kIdesc = idesc_f16_f32(128, 16);
constexpr int kSmemTarget = 100 * 1024;
constexpr int kPrepThreads = 256;

enum : int {
    kErrWaitW = 0x101,
    kErrWaitB = 0x102,
    kErrWaitAFull = 0x103,
    kErrWaitAEmpty = 0x104,
    kErrWaitD = 0x105,
    kErrWaitEmpty = 0x106,
};

struct Ctrl {
    uint64_t wfull[kMaxRing];     // weight tiles of the chunk landed
    uint64_t bfull[kMaxRing];     // activation tiles of the chunk landed
    uint64_t empty[kMaxRing];     // chunk slot free again (MMA commit / dp4a consumers)
    uint64_t a_full[kABufs];
    uint64_t a_empty[kABufs];
    uint64_t dfull;
    uint32_t tmem_base;
    int failed;
    int flag[2];
    float asc[BITMTP_MAX_GROUP][16];  // dequant scale per (problem - p0, row)
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

__host__ __device__ constexpr int btile_bytes(int path, int dp_rows) {
    return path == kPathTC16 ? 4096 : path == kPathTC8 ? 2048 : dp_rows * 128;
}
__host__ __device__ constexpr int btile_lbo(int path) { return path == kPathTC16 ? 256 : 128; }
__host__ __device__ constexpr int btile_sbo(int path) { return path == kPathTC16 ? 128 : 0; }
// Activation rows an operand tile holds (rows from M on are zero).
__host__ __device__ constexpr int btile_rows(int path, int dp_rows) {
    return path == kPathTC16 ? 16 : path == kPathTC8 ? 8 : dp_rows;
}

// fp16 pre-scale shift of the activation for A column c (J = 0,1,2,3,4,0,1,2).
__device__ __forceinline__ int bscale_shift(int c) { return 9 - 2 * ((c < 5) ? c : (c - 5)); }

__device__ __forceinline__ void fail(Ctrl* c, int* err, int code) {
    *reinterpret_cast<volatile int*>(&c->failed) = 1;
    atomicCAS(err, 0, code);
}

// One code word -> eight fp16x2 registers (A columns c = 0..7; half e of
// column c is k = 2c + e of the word).
__device__ __forceinline__ void unpack_word_f16(uint32_t w, uint32_t* r) {
    r[0] = w & 0x00030003u;
    r[1] = w & 0x000C000Cu;
    r[2] = w & 0x00300030u;
    r[3] = w & 0x00C000C0u;
    r[4] = w & 0x03000300u;
    const uint32_t t = w >> 10;
    r[5] = t & 0x00030003u;
    r[6] = t & 0x000C000Cu;
    r[7] = t & 0x00300030u;
}

__device__ __forceinline__ int find_problem_by_tile(const GemmParams& P, long long t) {
    int pi = 0;
#pragma unroll 1
    for (int i = 1; i < P.n_problems; ++i)
        if (t >= P.p[i].tile_begin) pi = i;
    return pi;
}
__device__ __forceinline__ long long range_start(int b, long long T, int n) {
    return (static_cast<long long>(b) * T) / n;
}
// CTA whose range holds flattened tile t (every range is non-empty: n <= T).
__device__ __forceinline__ int range_owner(long long t, long long T, int n) {
    return static_cast<int>(((t + 1) * n - 1) / T);
}

// Flattened-tile walker: (problem, row tile, k tile) advancing with k fastest.
struct TileIter {
    int pi, rt, kt;
    __device__ void init(const GemmParams& P, long long t) {
        pi = find_problem_by_tile(P, t);
        const long long local = t - P.p[pi].tile_begin;
        rt = static_cast<int>(local / P.p[pi].kt);
        kt = static_cast<int>(local % P.p[pi].kt);
    }
    __device__ void next(const GemmParams& P) {
        if (++kt == P.p[pi].kt) {
            kt = 0;
            if (++rt == P.p[pi].nt) {
                rt = 0;
                ++pi;
            }
        }
    }
};

// Bulk-copy the weight tiles of tiles [first, first + count) of this CTA's
// range into consecutive ring slots, one copy per run that is contiguous in
// global memory (within one problem); all copies complete on `bar`.
__device__ void issue_weights(const GemmParams& P, long long first, int count, uint8_t* dst, uint32_t bar,
                              uint64_t pol) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(count * kTileBytes));
    TileIter it;
    it.init(P, first);
    const uint8_t* run_src = nullptr;
    int run_len = 0, run_pi = -1;
    uint8_t* run_dst = dst;
    for (int k = 0; k < count; ++k) {
        const GemmProblem& pr = P.p[it.pi];
        const uint8_t* src = pr.pk + (static_cast<size_t>(it.rt) * pr.kt + it.kt) * kTileBytes;
        if (run_len == 0 || it.pi != run_pi) {
            if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * kTileBytes, bar, pol);
            run_dst = dst + k * kTileBytes;
            run_src = src;
            run_len = 0;
            run_pi = it.pi;
        }
        ++run_len;
        it.next(P);
    }
    if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * kTileBytes, bar, pol);
}

// The same for the activation tiles (BT bytes each) of those tiles: a run
// ends where the k index wraps to the next row tile or the problem changes.
__device__ void issue_acts(const GemmParams& P, long long first, int count, int BT, uint8_t* dst, uint32_t bar,
                           uint64_t pol) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(count * BT));
    TileIter it;
    it.init(P, first);
    const uint8_t* run_src = nullptr;
    int run_len = 0;
    uint8_t* run_dst = dst;
    for (int k = 0; k < count; ++k) {
        const uint8_t* src = P.p[it.pi].actb + static_cast<size_t>(it.kt) * BT;
        if (run_len == 0 || src != run_src + static_cast<size_t>(run_len) * BT) {
            if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * BT, bar, pol);
            run_dst = dst + k * BT;
            run_src = src;
            run_len = 0;
        }
        ++run_len;
        it.next(P);
    }
    if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * BT, bar, pol);
}

// Load 8 consecutive activations k0..k0+7 of one row (zero beyond K).
__device__ __forceinline__ void load8(const GemmProblem& pr, const char* row, bool vec_ok, int k0,
                                      float (&v)[8]) {
    if (pr.act_kind == BITMTP_BF16) {
        if (vec_ok && k0 + 8 <= pr.K) {
            const uint4 u = *reinterpret_cast<const uint4*>(row + 2ll * k0);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const uint16_t* r = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = (k0 + i < pr.K) ? __uint_as_float(static_cast<uint32_t>(r[k0 + i]) << 16) : 0.f;
        }
    } else if (pr.act_kind == BITMTP_F32) {
        if (vec_ok && k0 + 8 <= pr.K) {
            const float4 a = *reinterpret_cast<const float4*>(row + 4ll * k0);
            const float4 b = *reinterpret_cast<const float4*>(row + 4ll * k0 + 16);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
            const float* r = reinterpret_cast<const float*>(row);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (k0 + i < pr.K) ? r[k0 + i] : 0.f;
        }
    } else {  // int8 codes
        const int8_t* r = reinterpret_cast<const int8_t*>(row);
        if (vec_ok && k0 + 8 <= pr.K) {
            const uint2 u = *reinterpret_cast<const uint2*>(r + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = static_cast<float>(static_cast<int8_t>(u.x >> (8 * i)));
                v[4 + i] = static_cast<float>(static_cast<int8_t>(u.y >> (8 * i)));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (k0 + i < pr.K) ? static_cast<float>(r[k0 + i]) : 0.f;
        }
    }
}

__device__ __forceinline__ const char* act_row(const GemmProblem& pr, int m) {
    const int esize = pr.act_kind == BITMTP_F32 ? 4 : (pr.act_kind == BITMTP_BF16 ? 2 : 1);
    return static_cast<const char*>(pr.x) + static_cast<long long>(m) * pr.ldx * esize;
}

// ---------------------------------------------------- activation operand --
// One CTA per (problem, row m < btile_rows).  Writes row m of every
// activation tile of the problem (zeros for m >= M and beyond K), the prefix
// sums rsp[m][0..kt] of the row's codes over k tiles, and asc[m].
template <int PATH, int DPR>
__global__ void __launch_bounds__(kPrepThreads)
act_prep_kernel(const __grid_constant__ GemmParams P) {
    constexpr int kRows = btile_rows(PATH, DPR);
    constexpr int BT = btile_bytes(PATH, DPR);
    __shared__ float red[kPrepThreads / 32];
    __shared__ int tsum[BITMTP_MAX_K / kTileK];
    pdl_launch_dependents();  // the GEMM may start streaming weights now

    const int pi = blockIdx.x / kRows;
    const int m = blockIdx.x - pi * kRows;
    const GemmProblem& pr = P.p[pi];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool live = m < pr.M;
    const bool raw = pr.act_kind != BITMTP_Q8;
    const char* row = live ? act_row(pr, m) : nullptr;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const int ngroups = pr.kt * 16;  // 8-element groups, the zero tail of the last tile included

    // The activations may come from the previous kernel on the stream, and the
    // previous GEMM on this workspace may still be reading it.
    pdl_wait();

    float amax = 0.f;
    if (live && raw) {
        for (int g0 = 0; g0 < ngroups; g0 += kPrepThreads * 4) {
            float v[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int g = g0 + j * kPrepThreads + tid;
                if (g < ngroups) {
                    load8(pr, row, vec_ok, g * 8, v[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[j][i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kPrepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float s = quant_scale(amax);

    // Each group of 16 consecutive threads covers one k tile: ngroups is a
    // multiple of 16, so the shuffles below always see whole groups.
    for (int g0 = 0; g0 < ngroups; g0 += kPrepThreads) {
        const int g = g0 + tid;
        const bool gv = g < ngroups;
        float v[8];
        if (live && gv) {
            load8(pr, row, vec_ok, g * 8, v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        int qv[8];
        int rsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qv[i] = !live ? 0 : raw ? ((amax > 0.f) ? quantize(v[i], s) : 0) : static_cast<int>(v[i]);
            rsum += qv[i];
        }
        const int kt = g >> 4, gg = g & 15;
        uint8_t* tile = pr.actb + static_cast<size_t>(kt) * BT;
        if constexpr (PATH != kPathDP) {
            if (gv) {
                uint32_t packed[4];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const int sh = bscale_shift((gg & 1) * 4 + (i >> 1));
                    const __half h0 = __int2half_rn(qv[i] * (1 << sh));
                    const __half h1 = __int2half_rn(qv[i + 1] * (1 << sh));
                    packed[i >> 1] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                                     (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
                }
                *reinterpret_cast<uint4*>(tile + gg * btile_lbo(PATH) + (m >> 3) * btile_sbo(PATH) + (m & 7) * 16) =
                    make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
        } else {
            // A 16-k unit is two 8-groups (lanes 2i, 2i+1): the even lane
            // interleaves its partner's codes with its own.
            const uint32_t lo = (static_cast<uint32_t>(qv[0]) & 0xFFu) | ((static_cast<uint32_t>(qv[1]) & 0xFFu) << 8) |
                                ((static_cast<uint32_t>(qv[2]) & 0xFFu) << 16) | (static_cast<uint32_t>(qv[3]) << 24);
            const uint32_t hi = (static_cast<uint32_t>(qv[4]) & 0xFFu) | ((static_cast<uint32_t>(qv[5]) & 0xFFu) << 8) |
                                ((static_cast<uint32_t>(qv[6]) & 0xFFu) << 16) | (static_cast<uint32_t>(qv[7]) << 24);
            const uint32_t plo = __shfl_xor_sync(0xffffffffu, lo, 1);
            const uint32_t phi = __shfl_xor_sync(0xffffffffu, hi, 1);
            if (gv && (gg & 1) == 0) {
                uint32_t b[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    b[i] = (lo >> (8 * i)) & 0xFFu;
                    b[4 + i] = (hi >> (8 * i)) & 0xFFu;
                    b[8 + i] = (plo >> (8 * i)) & 0xFFu;
                    b[12 + i] = (phi >> (8 * i)) & 0xFFu;
                }
                uint32_t reg[4];
#pragma unroll
                for (int si = 0; si < 4; ++si)
                    reg[si] = b[2 * si] | (b[8 + 2 * si] << 8) | (b[2 * si + 1] << 16) | (b[9 + 2 * si] << 24);
                *reinterpret_cast<uint4*>(tile + (gg >> 1) * (DPR * 16) + m * 16) =
                    make_uint4(reg[0], reg[1], reg[2], reg[3]);
            }
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
        if (gv && (tid & 15) == 0) tsum[kt] = rsum;
    }
    __syncthreads();

    // rsp[m][0] = 0, rsp[m][t + 1] = codes of k tiles 0..t summed
    if (warp == 0) {
        const int KT = pr.kt;
        int* rsp = pr.rsp + m * (KT + 1);
        const int per = (KT + 31) / 32;
        const int t0 = lane * per, t1 = min(KT, t0 + per);
        int loc = 0;
        for (int t = t0; t < t1; ++t) loc += tsum[t];
        int inc = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        int run = inc - loc;
        if (lane == 0) rsp[0] = 0;
        for (int t = t0; t < t1; ++t) {
            run += tsum[t];
            rsp[t + 1] = run;
        }
        if (lane == 0) pr.asc[m] = raw ? dequant_scale(amax) : (live ? pr.a_scale_in[m] : 0.f);
    }
    // the GEMM reads the tiles through the async proxy (bulk copies)
    fence_proxy_async_global();
}

// ------------------------------------------------------------ epilogue --
__device__ __forceinline__ void store_out(const GemmProblem& pr, int m, int n, int acc, float a_scale) {
    const float v = __fmul_rn(__fmul_rn(static_cast<float>(acc), a_scale), pr.w_scale);
    const long long o = static_cast<long long>(m) * pr.ldy + n;
    if (pr.out_dtype == BITMTP_F32) {
        static_cast<float*>(pr.y)[o] = v;
    } else {
        static_cast<__nv_bfloat16*>(pr.y)[o] = __float2bfloat16_rn(v);
    }
    if (pr.acc) pr.acc[static_cast<long long>(m) * pr.lda + n] = acc;
}

// A split row tile this CTA contributed to, finished after the main loop.
struct Pending {
    int pi, rt, b_first, b_last;
    long long t_first;
};

// Finish one segment (k tiles [ka, kb) of row tile rt of problem pi).
// acc[m] is the exact partial sum_k T*q for the thread's row.  A whole row
// tile is written out at once; a split one is stored to this CTA's slot in
// the workspace (slot 0 if it is the first segment of the range, else 1) and
// recorded in `pend`.
__device__ void segment_epilogue(const GemmParams& P, const Ctrl* c, int p0, int pi, int rt, int ka, int kb,
                                 bool first_segment, const int (&acc)[16], int tid, bool alive, Pending* pend,
                                 int& npend) {
    const GemmProblem& pr = P.p[pi];
    const int M = pr.M;
    const int n = rt * kTileN + tid;
    if (ka == 0 && kb == pr.kt) {
        if (alive && n < pr.N) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < M) store_out(pr, m, n, acc[m], c->asc[pi - p0][m]);
        }
        return;
    }
    int* slot = P.slots + (static_cast<size_t>(blockIdx.x) * 2 + (first_segment ? 0 : 1)) * 16 * kTileN;
#pragma unroll
    for (int m = 0; m < 16; ++m)
        if (alive && m < M) slot[m * kTileN + tid] = acc[m];
    const long long T = P.total_tiles;
    const long long t_first = pr.tile_begin + static_cast<long long>(rt) * pr.kt;
    Pending& pe = pend[npend++];
    pe.pi = pi;
    pe.rt = rt;
    pe.t_first = t_first;
    pe.b_first = range_owner(t_first, T, P.nctas);
    pe.b_last = range_owner(t_first + pr.kt - 1, T, P.nctas);
}

// After the main loop: one fence, one counter increment per split row tile;
// the last contributor of a tile sums every contributor's slot (loads of four
// contributors in flight at a time), writes the output and leaves the counter
// at zero.  A split row tile is identified by the CTA holding its last k tile
// (a CTA is the last contributor of at most one split row tile).  Warps 0-3.
__device__ void finish_pending(const GemmParams& P, Ctrl* c, int p0, const Pending* pend, int npend, int tid,
                               bool alive) {
    if (npend == 0) return;  // uniform across the four warps
    __threadfence();
    named_bar_sync(1, 128);
    if (tid == 0) {
        for (int k = 0; k < npend; ++k) {
            const unsigned old = atomicAdd(P.counters + pend[k].b_last, 1u);
            c->flag[k] = (old == static_cast<unsigned>(pend[k].b_last - pend[k].b_first)) ? 1 : 0;
        }
    }
    named_bar_sync(1, 128);
    const int last0 = c->flag[0], last1 = npend > 1 ? c->flag[1] : 0;
    if (last0 | last1) __threadfence();
    const long long T = P.total_tiles;
    for (int k = 0; k < npend; ++k) {
        if (!(k == 0 ? last0 : last1)) continue;
        const GemmProblem& pr = P.p[pend[k].pi];
        const int M = pr.M;
        int tot[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) tot[m] = 0;
        for (int ob0 = pend[k].b_first; ob0 <= pend[k].b_last; ob0 += 4) {
            int v[4][16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ob = ob0 + j;
#pragma unroll
                for (int m = 0; m < 16; ++m) v[j][m] = 0;
                if (ob > pend[k].b_last) continue;
                const int sl = (range_start(ob, T, P.nctas) >= pend[k].t_first) ? 0 : 1;
                const int* os = P.slots + (static_cast<size_t>(ob) * 2 + sl) * 16 * kTileN;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    if (m < M) v[j][m] = __ldcg(os + m * kTileN + tid);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int m = 0; m < 16; ++m) tot[m] += v[j][m];
        }
        const int n = pend[k].rt * kTileN + tid;
        if (alive && n < pr.N) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < M) store_out(pr, m, n, tot[m], c->asc[pend[k].pi - p0][m]);
        }
        if (tid == 0) P.counters[pend[k].b_last] = 0u;
    }
    named_bar_sync(1, 128);
}

// Codes of rows 0..15 summed over k tiles [ka, kb) of problem pr (zero for
// rows >= M); read from the preparation kernel's prefix sums.
__device__ __forceinline__ void segment_code_sums(const GemmProblem& pr, int ka, int kb, int (&rq)[16]) {
    const int* rsp = pr.rsp;
    const int stride = pr.kt + 1;
#pragma unroll
    for (int m = 0; m < 16; ++m)
        rq[m] = (m < pr.M) ? __ldcg(rsp + m * stride + kb) - __ldcg(rsp + m * stride + ka) : 0;
}

template <int PATH, int DPR>
__global__ void __launch_bounds__(kGemmThreads, kCtasPerSm)
w2a8_streamk_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr bool kTC = PATH != kPathDP;
    constexpr int BT = btile_bytes(PATH, DPR);
    Ctrl* c = reinterpret_cast<Ctrl*>(smem);
    const int R = P.stages;                                  // chunks in the ring
    uint8_t* Wr = smem + kCtrlBytes;                         // [R][kChunk][4096]
    uint8_t* Br = Wr + static_cast<size_t>(R) * kChunk * kTileBytes;  // [R][kChunk][BT]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b = blockIdx.x;
    const long long T = P.total_tiles;
    const long long t_begin = range_start(b, T, P.nctas);
    const int nloc = static_cast<int>(range_start(b + 1, T, P.nctas) - t_begin);
    const int nchunks = (nloc + kChunk - 1) / kChunk;
    const int p0 = find_problem_by_tile(P, t_begin);
    const int p1 = find_problem_by_tile(P, t_begin + nloc - 1);

    // ------------------------------------------------------------ set-up --
    if (tid == 0) {
        for (int q = 0; q < R; ++q) {
            mbar_init(smem_u32(&c->wfull[q]), 1);
            mbar_init(smem_u32(&c->bfull[q]), 1);
            mbar_init(smem_u32(&c->empty[q]), kTC ? 1 : 4);
        }
        for (int a = 0; a < kABufs; ++a) {
            mbar_init(smem_u32(&c->a_full[a]), 4);
            mbar_init(smem_u32(&c->a_empty[a]), 1);
        }
        mbar_init(smem_u32(&c->dfull), 1);
        c->failed = 0;
        fence_mbar_init();
    }
    if constexpr (kTC) {
        if (warp == 0) {
            tmem_alloc(smem_u32(&c->tmem_base), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (kTC) tc_fence_after();
    const uint32_t tmem = kTC ? c->tmem_base : 0u;
    pdl_launch_dependents();

    const int npre = nchunks < R ? nchunks : R;
    int w_issued = 0, b_issued = 0;  // chunks whose copies were requested (warp 4, lane 0)

    // -------------------------------------------------------- main loop --
    if (warp == 4) {
        if (lane == 0) {
            // weights first: they do not depend on the kernels before this one
            const uint64_t pol = policy_evict_first();
            for (int j = 0; j < npre; ++j)
                issue_weights(P, t_begin + static_cast<long long>(j) * kChunk, min(kChunk, nloc - j * kChunk),
                              Wr + static_cast<size_t>(j) * kChunk * kTileBytes, smem_u32(&c->wfull[j]), pol);
            w_issued = npre;
            pdl_wait();  // the activation tiles are written by the preparation kernel
            const uint64_t pol_b = policy_evict_last();
            for (int j = 0; j < npre; ++j)
                issue_acts(P, t_begin + static_cast<long long>(j) * kChunk, min(kChunk, nloc - j * kChunk), BT,
                           Br + static_cast<size_t>(j) * kChunk * BT, smem_u32(&c->bfull[j]), pol_b);
            b_issued = npre;
            // refill ring slots as they are released
            for (int j = npre; j < nchunks; ++j) {
                const int q = j % R;
                if (!mbar_wait_bounded(smem_u32(&c->empty[q]), ((j / R) - 1) & 1)) {
                    fail(c, P.err, kErrWaitEmpty);
                    break;
                }
                const long long first = t_begin + static_cast<long long>(j) * kChunk;
                const int cnt = min(kChunk, nloc - j * kChunk);
                issue_weights(P, first, cnt, Wr + static_cast<size_t>(q) * kChunk * kTileBytes,
                              smem_u32(&c->wfull[q]), pol);
                w_issued = j + 1;
                issue_acts(P, first, cnt, BT, Br + static_cast<size_t>(q) * kChunk * BT, smem_u32(&c->bfull[q]),
                           pol_b);
                b_issued = j + 1;
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if constexpr (kTC) {
            if (lane == 0 && nloc > 0) {
                TileIter it;
                it.init(P, t_begin);
                const uint32_t bbase = smem_u32(Br);
                bool seg_first = true;
                bool ok = true;
                for (int i = 0; i < nloc && ok; ++i) {
                    const int j = i / kChunk, q = j % R;
                    const int s = q * kChunk + (i % kChunk);
                    const bool seg_last = (i == nloc - 1) || (it.kt == P.p[it.pi].kt - 1);
                    if ((i % kChunk) == 0 && !mbar_wait_bounded(smem_u32(&c->bfull[q]), (j / R) & 1)) {
                        fail(c, P.err, kErrWaitB);
                        break;
                    }
                    for (int h = 0; h < 2; ++h) {
                        const int u = 2 * i + h;
                        const int a = u % kABufs;
                        if (!mbar_wait_bounded(smem_u32(&c->a_full[a]), (u / kABufs) & 1)) {
                            fail(c, P.err, kErrWaitAFull);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int ch = h * 4 + jj;  // 16-k chunk within the k tile
                            const uint64_t bdesc = smem_desc_noswizzle(
                                bbase + s * BT + ch * 2 * btile_lbo(PATH), btile_lbo(PATH), btile_sbo(PATH));
                            mma_f16_ts(tmem + kAccCol, tmem + kACol + a * 32 + jj * 8, bdesc, kIdesc,
                                       (seg_first && h == 0 && jj == 0) ? 0u : 1u);
                        }
                        mma_commit(smem_u32(&c->a_empty[a]));
                    }
                    if (!ok) break;
                    if ((i % kChunk) == kChunk - 1 || i == nloc - 1) mma_commit(smem_u32(&c->empty[q]));
                    if (seg_last) mma_commit(smem_u32(&c->dfull));
                    seg_first = seg_last;
                    it.next(P);
                }
            }
        }
        __syncwarp();
    } else {
        // warps 0-3: one output row per thread.  A failed (timed-out) wait only
        // clears `alive`; every named barrier is still executed by all four warps.
        pdl_wait();  // outputs and workspace: the preparation kernel has finished
        for (int z = tid; z < (p1 - p0 + 1) * 16; z += 128) {
            const GemmProblem& pr = P.p[p0 + z / 16];
            c->asc[z / 16][z % 16] = (z % 16 < pr.M) ? __ldcg(pr.asc + z % 16) : 0.f;
        }
        named_bar_sync(1, 128);
        TileIter it;
        it.pi = it.rt = it.kt = 0;
        if (nloc > 0) it.init(P, t_begin);
        int ka = it.kt, seg_idx = 0, seg_first_i = 0;
        Pending pend[2];
        int npend = 0;
        int rq[16];
        if (nloc > 0) segment_code_sums(P.p[it.pi], ka, min(P.p[it.pi].kt, ka + nloc), rq);
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        int dacc[4][DPR];
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
            for (int m = 0; m < DPR; ++m) dacc[s4][m] = 0;
        bool alive = true;
        for (int i = 0; i < nloc; ++i) {
            const int j = i / kChunk, q = j % R;
            const int s = q * kChunk + (i % kChunk);
            const bool chunk_first = (i % kChunk) == 0;
            const bool chunk_last = (i % kChunk) == kChunk - 1 || i == nloc - 1;
            const bool seg_last = (i == nloc - 1) || (it.kt == P.p[it.pi].kt - 1);
            if (alive && chunk_first) {
                alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->wfull[q]), (j / R) & 1));
                if (!alive && lane == 0) fail(c, P.err, kErrWaitW);
                if constexpr (!kTC) {
                    if (alive) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->bfull[q]), (j / R) & 1));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitB);
                    }
                }
            }
            const uint8_t* wst = Wr + static_cast<size_t>(s) * kTileBytes;
            if constexpr (kTC) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int u = 2 * i + h;
                    const int a = u % kABufs;
                    if (alive && u >= kABufs) {
                        alive = __all_sync(0xffffffffu,
                                           mbar_wait_bounded(smem_u32(&c->a_empty[a]), ((u / kABufs) - 1) & 1));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitAEmpty);
                        tc_fence_after();
                    }
                    if (alive) {
                        const uint4 wv = *reinterpret_cast<const uint4*>(wst + h * 2048 + tid * 16);
                        uint32_t r[32];
                        unpack_word_f16(wv.x, r + 0);
                        unpack_word_f16(wv.y, r + 8);
                        unpack_word_f16(wv.z, r + 16);
                        unpack_word_f16(wv.w, r + 24);
                        tmem_st32(tmem + lane_base + kACol + a * 32, r);
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&c->a_full[a]));
                    }
                }
            } else {
                if (alive) {
                    const uint8_t* bst = Br + static_cast<size_t>(s) * BT;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 wv = *reinterpret_cast<const uint4*>(wst + h * 2048 + tid * 16);
                        const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int ch = h * 4 + jj;
                            const uint32_t w = wd[jj];
                            const uint32_t m0 = w & 0x03030303u, m1 = w & 0x0C0C0C0Cu;
                            const uint32_t m2 = w & 0x30303030u, m3 = w & 0xC0C0C0C0u;
#pragma unroll
                            for (int m = 0; m < DPR; ++m) {
                                const int4 qv = *reinterpret_cast<const int4*>(bst + ch * (DPR * 16) + m * 16);
                                dacc[0][m] = dp4a_us(m0, qv.x, dacc[0][m]);
                                dacc[1][m] = dp4a_us(m1, qv.y, dacc[1][m]);
                                dacc[2][m] = dp4a_us(m2, qv.z, dacc[2][m]);
                                dacc[3][m] = dp4a_us(m3, qv.w, dacc[3][m]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0 && chunk_last) mbar_arrive(smem_u32(&c->empty[q]));
                }
            }
            if (seg_last) {
                int acc[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) acc[m] = 0;
                if constexpr (kTC) {
                    if (alive) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->dfull), seg_idx & 1));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitD);
                    }
                    if (alive) {
                        tc_fence_after();
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + kAccCol, v);
                        tc_wait_ld();
                        tc_fence_before();
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            acc[m] = __float2int_rn(__uint_as_float(v[m]) * 32768.f) - rq[m];
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < DPR; ++m) {
                        acc[m] = dacc[0][m] + (dacc[1][m] >> 2) + (dacc[2][m] >> 4) + (dacc[3][m] >> 6) - rq[m];
                        dacc[0][m] = dacc[1][m] = dacc[2][m] = dacc[3][m] = 0;
                    }
                }
                segment_epilogue(P, c, p0, it.pi, it.rt, ka, it.kt + 1, seg_first_i == 0, acc, tid, alive, pend,
                                 npend);
                ++seg_idx;
                seg_first_i = i + 1;
                ka = 0;
            }
            it.next(P);
            if (seg_last && i + 1 < nloc)  // the next segment starts at k tile 0 of the next row tile
                segment_code_sums(P.p[it.pi], 0, min(P.p[it.pi].kt, nloc - (i + 1)), rq);
        }
        finish_pending(P, c, p0, pend, npend, tid, alive);
    }

    // ------------------------------------------------------- tear-down --
    __syncthreads();
    if (warp == 4 && lane == 0 && c->failed) {
        // never release shared memory with a bulk copy still in flight: wait
        // (bounded) for the last requested phase of every slot
        for (int q = 0; q < R; ++q) {
            if (q < w_issued)
                (void)mbar_wait_bounded(smem_u32(&c->wfull[q]), ((w_issued - 1 - q) / R) & 1, 100000000ull);
            if (q < b_issued)
                (void)mbar_wait_bounded(smem_u32(&c->bfull[q]), ((b_issued - 1 - q) / R) & 1, 100000000ull);
        }
    }
    if constexpr (kTC) {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
    }
}

cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

template <int PATH, int DPR>
cudaError_t launch_one(const GemmParams& prm, bool pdl, cudaStream_t stream) {
    auto kern = &w2a8_streamk_kernel<PATH, DPR>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gemm_smem_bytes(PATH, DPR, kMaxRing)));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaLaunchAttribute attr[1] = {pdl_attr()};

    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(static_cast<unsigned>(prm.n_problems * btile_rows(PATH, DPR)), 1, 1);
    pc.blockDim = dim3(kPrepThreads, 1, 1);
    pc.dynamicSmemBytes = 0;
    pc.stream = stream;
    pc.attrs = attr;
    pc.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&pc, &act_prep_kernel<PATH, DPR>, prm);
    if (e != cudaSuccess) return e;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(prm.nctas), 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_smem_bytes(PATH, DPR, prm.stages);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // overlaps the preparation kernel: only weights are read before its wait
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

int gemm_stages(int path, int dp_rows) {
    const int per_chunk = kChunk * (kTileBytes + btile_bytes(path, dp_rows));
    int r = (kSmemTarget - kCtrlBytes) / per_chunk;
    if (r > kMaxRing) r = kMaxRing;
    if (r < 2) r = 2;
    return r;
}

size_t gemm_smem_bytes(int path, int dp_rows, int stages) {
    return static_cast<size_t>(kCtrlBytes) +
           static_cast<size_t>(stages) * kChunk * (kTileBytes + btile_bytes(path, dp_rows));
}

cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, bool pdl, cudaStream_t stream) {
    if (path == kPathTC16) return launch_one<kPathTC16, 1>(prm, pdl, stream);
    if (path == kPathTC8) return launch_one<kPathTC8, 1>(prm, pdl, stream);
    if (dp_rows <= 1) return launch_one<kPathDP, 1>(prm, pdl, stream);
    if (dp_rows <= 2) return launch_one<kPathDP, 2>(prm, pdl, stream);
    return launch_one<kPathDP, 4>(prm, pdl, stream);
}

}  // namespace bitmtp
