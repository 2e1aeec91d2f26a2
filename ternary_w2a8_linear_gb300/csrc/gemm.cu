// gemm.cu -- the W2A8 ternary linear on sm_103a: a persistent stream-K kernel.
//
// One launch computes one or several independent linears ("problems") with
// the same compute path:
//
//  phase 0  every CTA starts streaming its first packed-weight tiles into a
//           shared-memory ring with bulk copies (TMA engine) of up to four
//           contiguous 4 KiB tiles each -- the engine's cost is per copy, so
//           16 KiB copies stream at HBM speed where 4 KiB ones do not;
//           weights do not depend on the previous kernel on the stream;
//  phase 1  activation rows are quantised (per-row absmax, fp32 round half to
//           even, the same code as the standalone quantiser) one row per CTA
//           task, written straight into the activation operand tiles the
//           compute path consumes, with per-k-tile row sums of the codes;
//  barrier  one grid-wide barrier (all CTAs are co-resident by construction);
//  phase 2  the flattened (problem, row tile, k tile) space is split into
//           equal contiguous ranges, one per CTA (stream-K), so every SM
//           streams the same number of weight bytes whatever the mix of
//           shapes.  A row tile whose k tiles span several CTAs is finished by
//           the last of them to arrive, after each added its partial into an
//           accumulator in the workspace; the dequant epilogue is fused.
//
// Compute paths (the same 2-bit code words feed both):
//   tensor (kPathTC16 / kPathTC8): each of 128 threads owns one output row
//     (one TMEM lane), turns its code words into fp16 bit patterns with one
//     mask per register -- the 2-bit code u lands in the fp16 subnormal range,
//     value u * 4^J * 2^-24 -- and writes them to tensor memory as the A
//     operand (tcgen05.st); one thread issues tcgen05.mma kind::f16 (M=128,
//     N=16, K=16) against the activation tile in shared memory, whose fp16
//     entries are q * 2^(9-2J).  Every product is u*q*2^-15 and every partial
//     sum an integer multiple of 2^-15 below 2^9, so the fp32 accumulator is
//     exact in any order.  kPathTC8 keeps 8 activation rows (the second row
//     group aliases the first through a zero stride).
//   dp4a (kPathDP): four byte masks per code word, four int32 accumulators
//     per row (scales 4^s, recombined with exact shifts).
// With u = T + 1, sum_k T*q = sum_k u*q - sum_k q; the row sums come from the
// quantisation phase.
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

constexpr int kMaxStages = 24;   // tile slots in the shared-memory ring
constexpr int kChunk = 4;        // tile slots per bulk-copy chunk (16 KiB of weights)
constexpr int kMaxChunks = kMaxStages / kChunk;
constexpr int kCtrlBytes = 1024;
constexpr int kScratchBytes = 2048;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kAccCol = 0;      // D: 16 fp32 columns, one per activation row
constexpr uint32_t kACol = 32;       // A: three buffers of 32 columns (64 k each)
constexpr int kABufs = 3;
constexpr uint32_t kIdesc = idesc_f16_f32(128, 16);
constexpr int kSmemTarget = 100 * 1024;  // two CTAs per SM, deep weight ring

enum : int {
    kErrWaitW = 0x101,
    kErrWaitB = 0x102,
    kErrWaitAFull = 0x103,
    kErrWaitAEmpty = 0x104,
    kErrWaitD = 0x105,
    kErrWaitEmpty = 0x106,
    kErrGridBarrier = 0x107,
};

struct Ctrl {
    uint64_t wfull[kMaxChunks];
    uint64_t bfull[kMaxChunks];
    uint64_t empty[kMaxChunks];
    uint64_t a_full[kABufs];
    uint64_t a_empty[kABufs];
    uint64_t dfull;
    uint32_t tmem_base;
    int failed;
    int last;
    float red_f[4];
    int red_i[4];
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

__host__ __device__ constexpr int btile_lbo(int path) { return path == kPathTC16 ? 256 : 128; }
__host__ __device__ constexpr int btile_sbo(int path) { return path == kPathTC16 ? 128 : 0; }

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

__device__ __forceinline__ int find_problem_by_task(const GemmParams& P, int task) {
    int pi = 0;
#pragma unroll 1
    for (int i = 1; i < P.n_problems; ++i)
        if (task >= P.p[i].task_begin) pi = i;
    return pi;
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
// CTA whose range holds flattened tile t.
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

// Bulk-copy the weight tiles (or the activation tiles) of tiles
// [first, first + count) of this CTA's range into consecutive ring slots,
// merging runs that are contiguous in global memory (weights: within one
// problem; activation tiles: within one row tile) into single copies; all
// copies complete on `bar`, which expects their total bytes.
template <bool kW>
__device__ void issue_chunk(const GemmParams& P, long long first, int count, uint8_t* dst, int slot_bytes,
                            uint32_t bar, uint64_t pol) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(count * slot_bytes));
    TileIter it;
    it.init(P, first);
    const uint8_t* run_src = nullptr;
    int run_len = 0;
    uint8_t* run_dst = dst;
    int prev_pi = -1, prev_rt = -1;
    for (int k = 0; k < count; ++k) {
        const GemmProblem& pr = P.p[it.pi];
        const uint8_t* src = kW ? pr.pk + (static_cast<size_t>(it.rt) * pr.kt + it.kt) * kTileBytes
                                : P.btiles + (static_cast<size_t>(pr.bt_begin) + it.kt) * slot_bytes;
        const bool contiguous = run_len > 0 && it.pi == prev_pi && (kW || it.rt == prev_rt);
        if (!contiguous) {
            if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * slot_bytes, bar, pol);
            run_dst = dst + k * slot_bytes;
            run_src = src;
            run_len = 0;
        }
        ++run_len;
        prev_pi = it.pi;
        prev_rt = it.rt;
        it.next(P);
    }
    if (run_len > 0) bulk_g2s(smem_u32(run_dst), run_src, run_len * slot_bytes, bar, pol);
}

// Block-wide (128 threads, named barrier 1) max of non-negative floats.
__device__ __forceinline__ float block128_max(float v, Ctrl* c, int tid) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((tid & 31) == 0) c->red_f[tid >> 5] = v;
    named_bar_sync(1, 128);
    const float r = fmaxf(fmaxf(c->red_f[0], c->red_f[1]), fmaxf(c->red_f[2], c->red_f[3]));
    named_bar_sync(1, 128);
    return r;
}

// Exclusive prefix sum over 128 threads (named barrier 1); returns the
// exclusive sum and writes the block total to *total.
__device__ __forceinline__ int block128_exscan(int v, Ctrl* c, int tid, int* total) {
    const int lane = tid & 31;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) c->red_i[tid >> 5] = incl;
    named_bar_sync(1, 128);
    int base = 0;
    for (int w = 0; w < (tid >> 5); ++w) base += c->red_i[w];
    *total = c->red_i[0] + c->red_i[1] + c->red_i[2] + c->red_i[3];
    named_bar_sync(1, 128);
    return base + incl - v;
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
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (k0 + i < pr.K) ? static_cast<float>(r[k0 + i]) : 0.f;
    }
}

// ------------------------------------------------ phase 1: one activation row --
// One CTA task = one activation row: absmax over K (all loads of a batch in
// flight), then the codes written into the operand tiles, with per-k-tile row
// sums and their prefix over k tiles.
template <int PATH, int DPR>
__device__ void quant_row_task(const GemmParams& P, int task, Ctrl* c, int* tsum, int tid) {
    const int pi = find_problem_by_task(P, task);
    const GemmProblem& pr = P.p[pi];
    const int m = task - pr.task_begin;
    const int KT = pr.kt;
    const int esize = pr.act_kind == BITMTP_F32 ? 4 : (pr.act_kind == BITMTP_BF16 ? 2 : 1);
    const char* row = static_cast<const char*>(pr.x) + static_cast<long long>(m) * pr.ldx * esize;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const bool raw = pr.act_kind != BITMTP_Q8;

    for (int t = tid; t < KT; t += 128) tsum[t] = 0;
    float s = 0.f;
    if (raw) {
        const int ng = (pr.K + 7) >> 3;
        float a = 0.f;
        for (int g0 = tid; g0 < ng; g0 += 512) {
            float v[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int g = g0 + j * 128;
                if (g < ng) {
                    load8(pr, row, vec_ok, g * 8, v[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[j][i]));
        }
        const float amax = block128_max(a, c, tid);  // also orders the tsum zeroing
        s = quant_scale(amax);
        if (tid == 0) P.ascale[pr.task_begin + m] = dequant_scale(amax);
    } else {
        if (tid == 0) P.ascale[pr.task_begin + m] = pr.a_scale_in[m];
        named_bar_sync(1, 128);
    }

    uint8_t* bt = P.btiles + static_cast<size_t>(pr.bt_begin) * P.btile_bytes;
    if constexpr (PATH != kPathDP) {
        // 8-k groups, 16 per k tile
        const int ngroups = KT * 16;
        for (int g0 = tid; g0 < ngroups; g0 += 256) {
            float v[2][8];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int g = g0 + j * 128;
                if (g < ngroups) {
                    load8(pr, row, vec_ok, g * 8, v[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int g = g0 + j * 128;
                if (g >= ngroups) continue;
                int rs = 0;
                uint32_t packed[4];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const int q0 = raw ? quantize(v[j][i], s) : static_cast<int>(v[j][i]);
                    const int q1 = raw ? quantize(v[j][i + 1], s) : static_cast<int>(v[j][i + 1]);
                    rs += q0 + q1;
                    const int sh = bscale_shift((g & 1) * 4 + (i >> 1));
                    const __half h0 = __int2half_rn(q0 * (1 << sh));
                    const __half h1 = __int2half_rn(q1 * (1 << sh));
                    packed[i >> 1] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                                     (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
                }
                const int tile = g >> 4, kg = g & 15;
                uint8_t* dst = bt + static_cast<size_t>(tile) * P.btile_bytes + kg * btile_lbo(PATH) +
                               (m >> 3) * btile_sbo(PATH) + (m & 7) * 16;
                *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                if (rs != 0) atomicAdd(&tsum[tile], rs);
            }
        }
    } else {
        // 16-k chunks, 8 per k tile
        const int nchunks = KT * 8;
        for (int g = tid; g < nchunks; g += 128) {
            float v[16];
            load8(pr, row, vec_ok, g * 16, *reinterpret_cast<float(*)[8]>(v));
            load8(pr, row, vec_ok, g * 16 + 8, *reinterpret_cast<float(*)[8]>(v + 8));
            int q[16];
            int rs = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                q[i] = raw ? quantize(v[i], s) : static_cast<int>(v[i]);
                rs += q[i];
            }
            uint32_t reg[4];
#pragma unroll
            for (int sidx = 0; sidx < 4; ++sidx) {
                reg[sidx] = (static_cast<uint32_t>(q[2 * sidx]) & 0xFFu) |
                            ((static_cast<uint32_t>(q[8 + 2 * sidx]) & 0xFFu) << 8) |
                            ((static_cast<uint32_t>(q[2 * sidx + 1]) & 0xFFu) << 16) |
                            ((static_cast<uint32_t>(q[9 + 2 * sidx]) & 0xFFu) << 24);
            }
            const int tile = g >> 3, ch = g & 7;
            uint8_t* dst = bt + static_cast<size_t>(tile) * P.btile_bytes + ch * (DPR * 16) + m * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(reg[0], reg[1], reg[2], reg[3]);
            if (rs != 0) atomicAdd(&tsum[tile], rs);
        }
    }
    named_bar_sync(1, 128);
    // prefix[kt] = sum of the row's codes over k tiles [0, kt), kt = 0..KT
    int* pre = P.prefix + pr.pre_begin;
    const int a0 = (2 * tid < KT) ? tsum[2 * tid] : 0;
    const int a1 = (2 * tid + 1 < KT) ? tsum[2 * tid + 1] : 0;
    int total = 0;
    const int ex = block128_exscan(a0 + a1, c, tid, &total);
    if (2 * tid < KT) pre[(2 * tid) * 16 + m] = ex;
    if (2 * tid + 1 < KT) pre[(2 * tid + 1) * 16 + m] = ex + a0;
    if (tid == 0) pre[KT * 16 + m] = total;
    named_bar_sync(1, 128);
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
};

// Finish one segment (k tiles [ka, kb) of row tile rt of problem pi) held by
// this CTA.  part[m] = sum_k u*q for the thread's row over the segment.  A
// whole row tile is written out at once.  For a split row tile the partial is
// added into the row tile's accumulator in the workspace (fp32 vector
// atomics; every value is an integer below 2^24, so every sum is exact in any
// order) without waiting, and the tile is recorded in `pend` to be finished
// after the main loop.  A split row tile is identified by the CTA holding its
// last k tile: a CTA is the last contributor of at most one split row tile.
__device__ void segment_epilogue(const GemmParams& P, int pi, int rt, int ka, int kb, const int (&part)[16],
                                 int tid, bool alive, Pending* pend, int& npend) {
    const GemmProblem& pr = P.p[pi];
    const int M = pr.M;
    const int* pre = P.prefix + pr.pre_begin;
    const int n = rt * kTileN + tid;
    int acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m)
        acc[m] = (m < M) ? part[m] - (pre[kb * 16 + m] - pre[ka * 16 + m]) : 0;

    if (ka == 0 && kb == pr.kt) {
        if (alive && n < pr.N) {
            const float* asc = P.ascale + pr.task_begin;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < M) store_out(pr, m, n, acc[m], asc[m]);
        }
        return;
    }
    const long long T = P.total_tiles;
    const long long t_first = pr.tile_begin + static_cast<long long>(rt) * pr.kt;
    const int b_last = range_owner(t_first + pr.kt - 1, T, P.nctas);
    float4* accum = reinterpret_cast<float4*>(P.accum) + (static_cast<size_t>(b_last) * kTileN + tid) * 4;
    if (alive) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (4 * g < M)
                atomicAdd(accum + g, make_float4(static_cast<float>(acc[4 * g]), static_cast<float>(acc[4 * g + 1]),
                                                 static_cast<float>(acc[4 * g + 2]),
                                                 static_cast<float>(acc[4 * g + 3])));
    }
    pend[npend].pi = pi;
    pend[npend].rt = rt;
    pend[npend].b_first = range_owner(t_first, T, P.nctas);
    pend[npend].b_last = b_last;
    ++npend;
}

// After the main loop: publish this CTA's contributions to its split row
// tiles (one fence, one counter increment each); the last contributor of a
// tile reads the total, writes the output and leaves accumulator and counter
// at zero.  Warps 0-3 only (named barrier 1).
__device__ void finish_pending(const GemmParams& P, Ctrl* c, const Pending* pend, int npend, int tid, bool alive) {
    if (npend == 0) return;  // uniform across the four warps
    __threadfence();
    named_bar_sync(1, 128);
    if (tid == 0) {
        for (int k = 0; k < npend; ++k) {
            const unsigned old = atomicAdd(P.counters + pend[k].b_last, 1u);
            c->red_i[k] = (old == static_cast<unsigned>(pend[k].b_last - pend[k].b_first)) ? 1 : 0;
        }
    }
    named_bar_sync(1, 128);
    const int last0 = c->red_i[0], last1 = npend > 1 ? c->red_i[1] : 0;
    if (last0 | last1) __threadfence();
    for (int k = 0; k < npend; ++k) {
        if (!(k == 0 ? last0 : last1)) continue;
        const GemmProblem& pr = P.p[pend[k].pi];
        const int M = pr.M;
        const int n = pend[k].rt * kTileN + tid;
        float4* accum = reinterpret_cast<float4*>(P.accum) + (static_cast<size_t>(pend[k].b_last) * kTileN + tid) * 4;
        float tot[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (4 * g < M) {
                const float4 v = __ldcg(accum + g);
                tot[4 * g] = v.x; tot[4 * g + 1] = v.y; tot[4 * g + 2] = v.z; tot[4 * g + 3] = v.w;
                __stcg(accum + g, make_float4(0.f, 0.f, 0.f, 0.f));
            } else {
                tot[4 * g] = tot[4 * g + 1] = tot[4 * g + 2] = tot[4 * g + 3] = 0.f;
            }
        }
        if (alive && n < pr.N) {
            const float* asc = P.ascale + pr.task_begin;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < M) store_out(pr, m, n, static_cast<int>(tot[m]), asc[m]);
        }
        if (tid == 0) P.counters[pend[k].b_last] = 0u;
    }
    named_bar_sync(1, 128);
}

// Grid-wide barrier: each CTA adds 1 except CTA 0, which adds 2^31 - (n-1), so
// the counter crosses a multiple of 2^31 -- its top bit flips -- exactly when
// the last CTA arrives, provided its low 31 bits start at zero; they come back
// to zero after every barrier.  Called by one thread per CTA.
__device__ bool grid_barrier(unsigned* bar, int nblocks) {
    __threadfence();
    const unsigned inc = (blockIdx.x == 0) ? (0x80000000u - static_cast<unsigned>(nblocks - 1)) : 1u;
    const unsigned old = atomicAdd(bar, inc);
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
        if (((old ^ ld_acquire_gpu(bar)) & 0x80000000u) != 0) break;
        if ((it & 63u) == 63u && global_ns() - t0 > 2000000000ull) return false;
    }
    __threadfence();
    return true;
}

template <int PATH, int DPR>
__global__ void __launch_bounds__(kGemmThreads, kCtasPerSm)
w2a8_streamk_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Ctrl* c = reinterpret_cast<Ctrl*>(smem);
    int* tsum = reinterpret_cast<int*>(smem + kCtrlBytes);
    uint8_t* Wr = smem + kCtrlBytes + kScratchBytes;
    const int S = P.stages;
    uint8_t* Br = Wr + static_cast<size_t>(S) * kTileBytes;
    const int BT = P.btile_bytes;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b = blockIdx.x;
    const long long T = P.total_tiles;
    const long long t_begin = range_start(b, T, P.nctas);
    const int nloc = static_cast<int>(range_start(b + 1, T, P.nctas) - t_begin);
    constexpr bool kTC = PATH != kPathDP;

    // ------------------------------------------------------------ set-up --
    if (tid == 0) {
        for (int q = 0; q < S / kChunk; ++q) {
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

    // ------------------------------- phase 0: start the weight stream --
    const int R = S / kChunk;                         // chunks in the ring
    const int nchunks = (nloc + kChunk - 1) / kChunk;
    const int npre = nchunks < R ? nchunks : R;
    uint64_t pol = 0;
    if (warp == 4 && lane == 0) {
        pol = policy_evict_first();
        for (int j = 0; j < npre; ++j) {
            const int cnt = min(kChunk, nloc - j * kChunk);
            issue_chunk<true>(P, t_begin + j * kChunk, cnt, Wr + static_cast<size_t>(j) * kChunk * kTileBytes,
                              kTileBytes, smem_u32(&c->wfull[j]), pol);
        }
    }
    __syncwarp();
    pdl_launch_dependents();

    // --------------------------------- phase 1: quantise activation rows --
    if (warp < 4) {
        pdl_wait();  // activations may be written by the previous kernel on the stream
            for (int task = b; task < P.total_tasks; task += P.nctas)
            quant_row_task<PATH, DPR>(P, task, c, tsum, tid);
        fence_proxy_async_global();  // operand tiles are read back by bulk copies
        __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
        if (!grid_barrier(P.gridbar, P.nctas)) fail(c, P.err, kErrGridBarrier);
    }
    __syncthreads();

    // ------------------------------------------------ phase 2: stream-K --
    if (warp == 4) {
        if (lane == 0 && nloc > 0) {
            fence_proxy_async_global();
            for (int j = 0; j < nchunks; ++j) {
                const int q = j % R;
                const int cnt = min(kChunk, nloc - j * kChunk);
                const long long first = t_begin + static_cast<long long>(j) * kChunk;
                if (j >= R) {
                    if (!mbar_wait_bounded(smem_u32(&c->empty[q]), ((j / R) - 1) & 1)) {
                        fail(c, P.err, kErrWaitEmpty);
                        break;
                    }
                    issue_chunk<true>(P, first, cnt, Wr + static_cast<size_t>(q) * kChunk * kTileBytes, kTileBytes,
                                      smem_u32(&c->wfull[q]), pol);
                }
                issue_chunk<false>(P, first, cnt, Br + static_cast<size_t>(q) * kChunk * BT, BT,
                                   smem_u32(&c->bfull[q]), pol);
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
                    const int s = i % S;
                    const int q = (i / kChunk) % R;
                    const bool seg_last = (i == nloc - 1) || (it.kt == P.p[it.pi].kt - 1);
                    if ((i % kChunk) == 0 && !mbar_wait_bounded(smem_u32(&c->bfull[q]), ((i / kChunk) / R) & 1)) {
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
                            const int chunk = h * 4 + jj;  // 16-k chunk within the k tile
                            const uint64_t bdesc = smem_desc_noswizzle(
                                bbase + s * BT + chunk * 2 * btile_lbo(PATH), btile_lbo(PATH), btile_sbo(PATH));
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
        TileIter it;
        it.pi = it.rt = it.kt = 0;
        if (nloc > 0) it.init(P, t_begin);
        int part[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) part[m] = 0;
        int ka = it.kt, seg_idx = 0;
        Pending pend[2];
        int npend = 0;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        int dacc[4][DPR];
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
            for (int m = 0; m < DPR; ++m) dacc[s4][m] = 0;
        bool alive = true;
        for (int i = 0; i < nloc; ++i) {
            const int s = i % S;
            const int q = (i / kChunk) % R;
            const bool chunk_first = (i % kChunk) == 0;
            const bool chunk_last = (i % kChunk) == kChunk - 1 || i == nloc - 1;
            const bool seg_last = (i == nloc - 1) || (it.kt == P.p[it.pi].kt - 1);
            if (alive && chunk_first) {
                alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->wfull[q]), ((i / kChunk) / R) & 1));
                if (!alive && lane == 0) fail(c, P.err, kErrWaitW);
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
                if (alive && chunk_first) {
                    alive = __all_sync(0xffffffffu,
                                       mbar_wait_bounded(smem_u32(&c->bfull[q]), ((i / kChunk) / R) & 1));
                    if (!alive && lane == 0) fail(c, P.err, kErrWaitB);
                }
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
                        for (int m = 0; m < 16; ++m) part[m] = __float2int_rn(__uint_as_float(v[m]) * 32768.f);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < DPR; ++m) {
                        part[m] = dacc[0][m] + (dacc[1][m] >> 2) + (dacc[2][m] >> 4) + (dacc[3][m] >> 6);
                        dacc[0][m] = dacc[1][m] = dacc[2][m] = dacc[3][m] = 0;
                    }
                }
                segment_epilogue(P, it.pi, it.rt, ka, it.kt + 1, part, tid, alive, pend, npend);
                ++seg_idx;
                ka = 0;
            }
            it.next(P);
        }
        finish_pending(P, c, pend, npend, tid, alive);
    }

    // ------------------------------------------------------- tear-down --
    __syncthreads();
    if (warp == 4 && lane == 0 && c->failed) {
        // never release shared memory with a bulk copy still in flight
        for (int q = 0; q < npre; ++q) (void)mbar_wait_bounded(smem_u32(&c->wfull[q]), 0, 100000000ull);
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

template <int PATH, int DPR>
cudaError_t launch_one(const GemmParams& prm, bool pdl, cudaStream_t stream) {
    auto kern = &w2a8_streamk_kernel<PATH, DPR>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gemm_smem_bytes(PATH, DPR, kMaxStages)));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(prm.nctas), 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_smem_bytes(PATH, DPR, prm.stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

int gemm_stages(int path, int dp_rows) {
    const int bt = path == kPathTC16 ? 4096 : path == kPathTC8 ? 2048 : dp_rows * 128;
    int s = (kSmemTarget - kCtrlBytes - kScratchBytes) / (kTileBytes + bt);
    if (s > kMaxStages) s = kMaxStages;
    s -= s % kChunk;
    if (s < 2 * kChunk) s = 2 * kChunk;
    return s;
}

size_t gemm_smem_bytes(int path, int dp_rows, int stages) {
    const int bt = path == kPathTC16 ? 4096 : path == kPathTC8 ? 2048 : dp_rows * 128;
    return static_cast<size_t>(kCtrlBytes) + kScratchBytes + static_cast<size_t>(stages) * (kTileBytes + bt);
}

cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, bool pdl, cudaStream_t stream) {
    if (path == kPathTC16) return launch_one<kPathTC16, 1>(prm, pdl, stream);
    if (path == kPathTC8) return launch_one<kPathTC8, 1>(prm, pdl, stream);
    if (dp_rows <= 1) return launch_one<kPathDP, 1>(prm, pdl, stream);
    if (dp_rows <= 2) return launch_one<kPathDP, 2>(prm, pdl, stream);
    return launch_one<kPathDP, 4>(prm, pdl, stream);
}

}  // namespace bitmtp
