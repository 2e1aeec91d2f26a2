// gemm.cu -- the W2A8 ternary linear on sm_103a: an activation-operand
// preparation kernel followed by a persistent, warp-specialised stream-K GEMM.
//
// Two launches per call, chained by programmatic dependent launch (PDL)
// (one in the layer-chain mode of the dp4a path, below):
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
//                     weight bytes whatever the mix of shapes.  A range is a
//                     run of "segments" (the k tiles of one row tile it
//                     covers), worked from the range's end back to its start:
//                     its last segment, the head of a row tile the next CTA
//                     finishes ("contributor"), comes first, and its partial
//                     sums go to the CTA's slot in the workspace, published
//                     by a flag early on; its first segment, the tail of a row
//                     tile that earlier CTAs began ("owner"), comes last, when
//                     the contributors' flags are normally set: it adds their
//                     slots and writes the output.  Whole row tiles in between
//                     are written directly.  Only owners wait for other CTAs,
//                     and contributors never wait, so nothing can deadlock;
//                     every wait is bounded.  Each CTA:
//     warp 4      bulk copies (TMA engine) into a ring of chunks of four
//                 tiles: weight tiles first -- they do not depend on the
//                 preparation kernel, so they are requested before the PDL
//                 wait -- and, after it, the matching activation tiles; each
//                 contiguous run is one copy (the engine's cost is per copy);
//                 and the flag that publishes a contributor's partial sums;
//     warps 0-3   one output row per thread: the compute path (below), then
//                 the segment epilogues;
//     warp 5      (tensor path) issues tcgen05.mma.
//
// Compute paths (the same 2-bit code words feed both):
//   tensor (kPathTC16 / kPathTC8): each thread turns its code words into e4m3
//     bytes with one shift and one mask per register -- the 2-bit code u is
//     the mantissa of an e4m3 subnormal, value u * 2^-9 -- and writes them to
//     tensor memory as the A operand (tcgen05.st, six k-tile buffers in
//     flight).  The activation operand splits every code exactly as
//     q = 16*h + l (h in [-8, 7], l in [0, 15], both exact in e4m3) into two
//     operand rows, so one tcgen05.mma kind::f8f6f4 (M=128, K=32, N = twice the
//     activation rows: 32 or 16) yields both halves.  Products are integers
//     times 2^-9 and every sum stays below 2^24 of those units, so the fp32
//     accumulator is exact; the epilogue forms 2^9 * (16*D_h + D_l).  The
//     elected lane of a converged warp issues the MMAs under a predicate, two
//     k tiles (eight MMAs, straight-line code) per wait: a branch or a wait
//     between tcgen05.mma issues costs more than the MMAs themselves.  Two
//     accumulators alternate between consecutive row-tile segments, so a
//     segment's epilogue runs while the next segment's MMAs go on.
//   dp4a (kPathDP): four byte masks per code word, four int32 accumulators
//     per row (scales 4^s, recombined with exact shifts).
// With u = T + 1, sum_k T*q = sum_k u*q - sum_k q; the second sum comes from
// the preparation kernel's prefix sums.
//
// Layer-chain mode (dp4a path, every problem's row absmax handed over by the
// call that wrote the rows): no preparation kernel.  The consumer warps
// quantise the first ring chunk's activation tiles themselves and warp 5 the
// later ones, with per-tile code sums in shared memory; CTA 0 zeroes the
// output absmax and releases every CTA's epilogues through a workspace word,
// which the last CTA to finish resets.  A kernel instantiation of its own.  Both paths store the activation
// operand in units of 16 k: per operand row 16 bytes, byte 4s + b holding
// k = {2s, 2s+8, 2s+1, 2s+9}[b] of the unit -- the order in which one shift
// and mask per register lays out the code word.
//
// The operation is the packed W2A8 linear of "BitMTP: When Multi-Token
// Prediction Meets Low-Bit Large Language Models" (AI summary: Main Findings,
// first bullet -- 2-bit weights, 8-bit activations; Methodology in Plain
// English -- width-specialised packed low-bit operators, role-dependent output
// projections).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstddef>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace bitmtp {
namespace {

constexpr int kChunk = 4;            // k tiles per ring chunk (16 KiB of weights)
constexpr int kMaxRing = 6;          // chunks in the ring (upper bound)
constexpr int kCtrlBytes = 2304;
constexpr int kBarEpi = 1;           // named barrier: the four consumer warps
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccCol = 0;      // D: two accumulators (alternate segments), columns 0 .. 2 * d_cols
constexpr uint32_t kATileCols = 32;  // A: one k tile (128 k, one e4m3 byte each) per buffer
constexpr int kMaxATiles = 7;
constexpr int kDeferTiles = 5;       // a segment's epilogue runs this many tiles into the next one
constexpr int kMmaBatch = 2;         // k tiles per MMA-issuer wait
constexpr int kBatchBars = 8;        // MMA batch completion barriers (> A buffers)
constexpr int kSmemTarget = 102 * 1024;
constexpr int kPrepThreads = 512;
constexpr int kPrepUnits = 2;      // 16-element units of one row per thread and pass

enum : int {
    kErrWaitW = 0x101,
    kErrWaitB = 0x102,
    kErrWaitAFull = 0x103,
    kErrWaitAEmpty = 0x104,
    kErrWaitD = 0x105,
    kErrWaitEmpty = 0x106,
    kErrWaitFlag = 0x107,
    kErrWaitSlot = 0x108,
    kErrWaitZero = 0x109,
};

struct Ctrl {
    uint64_t wfull[kMaxRing];     // weight tiles of the chunk landed
    uint64_t bfull[kMaxRing];     // activation tiles of the chunk landed
    uint64_t empty[kMaxRing];     // chunk slot free again (both MMA warps' commits / dp4a consumers)
    uint64_t a_full[kBatchBars];  // A tiles of MMA batch b written: a_full[b % kBatchBars] (four writer warps)
    uint64_t mma_done[kBatchBars]; // MMA batch b complete: barrier b % kBatchBars
    uint64_t dfull[2][4];         // MMA warp 5 + i finished segment s: dfull[i][s & 3]
    uint64_t slot_done;           // contributor partial sums stored (four consumer warps)
    uint64_t drained[2];          // after a failed wait: every MMA MMA warp 5 + i issued is complete
    uint64_t zero_ready;          // fused dp4a mode: the output absmax is zeroed for this launch
    uint32_t tmem_base;
    int failed;
    int owner_ok;
    float asc[BITMTP_MAX_GROUP][16];  // dequant scale per (problem - p0, row)
    GemmProblem prob[BITMTP_MAX_GROUP];  // copy of the problem table
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

// Activation rows an operand tile holds (rows from M on are zero).
__host__ __device__ constexpr int btile_rows(int path, int dp_rows) {
    return (path == kPathTC16 || path == kPathF8) ? 16 : path == kPathTC8 ? 8 : dp_rows;
}
// Operand rows: the int8 tensor paths keep two (h and l) per activation row.
__host__ __device__ constexpr int btile_brows(int path, int dp_rows) {
    return (path == kPathDP || path == kPathF8) ? btile_rows(path, dp_rows) : 2 * btile_rows(path, dp_rows);
}
// Bytes of one k tile of the activation operand: 8 units of 16 k, each
// holding 16 bytes per operand row.
__host__ __device__ constexpr int btile_bytes(int path, int dp_rows) { return btile_brows(path, dp_rows) * 128; }
// Tensor-memory layout of the tensor paths: each accumulator is one fp32
// column per B row (the MMA's N); the last 8 columns hold the constant A
// operand -2^-9 (one MMA's 32 k); the A buffers fill the rest of the 256
// allocated columns (five at 16 rows, six at 8 and for FP8).
constexpr uint32_t kNegCols = 8;
__host__ __device__ constexpr uint32_t tmem_d_cols(int path, int dp_rows) {
    return static_cast<uint32_t>(btile_brows(path, dp_rows));
}
__host__ __device__ constexpr uint32_t tmem_a_col(int path, int dp_rows) { return 2 * tmem_d_cols(path, dp_rows); }
__host__ __device__ constexpr uint32_t tmem_neg_col(int path) { return path == kPathDP ? kTmemCols : kTmemCols - kNegCols; }
__host__ __device__ constexpr int tmem_a_tiles(int path, int dp_rows) {
    return path == kPathDP ? 1 : static_cast<int>((tmem_neg_col(path) - tmem_a_col(path, dp_rows)) / kATileCols);
}

__device__ __forceinline__ void fail(Ctrl* c, int* err, int code) {
    *reinterpret_cast<volatile int*>(&c->failed) = 1;
    atomicCAS(err, 0, code);
}

// One code word (16 k) -> four registers of e4m3 bytes u * 2^-9: register s,
// byte b holds k = {2s, 2s+8, 2s+1, 2s+9}[b] of the word.
__device__ __forceinline__ void unpack_word_e4m3(uint32_t w, uint32_t* r) {
    r[0] = w & 0x03030303u;
    r[1] = (w >> 2) & 0x03030303u;
    r[2] = (w >> 4) & 0x03030303u;
    r[3] = (w >> 6) & 0x03030303u;
}

// One tile row's 32 bytes (eight words) -> 32 registers of e4m3 bytes u * 2^-9.
__device__ __forceinline__ void unpack_row_e4m3(const uint4& a0, const uint4& a1, uint32_t (&r)[32]) {
    const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) unpack_word_e4m3(w[i], r + 4 * i);
}

// Two floats -> their E4M3 bytes, a in bits 0-7, b in bits 8-15 (hardware
// conversion: round to nearest even, saturating at +-448).  The int8 paths
// pass integer values |v| <= 15, which are exact in E4M3.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Problem holding flattened tile t.  pp: the problem table (a shared-memory
// copy: indexing the kernel parameter with a runtime index costs a slow
// dependent load per field).
__device__ __forceinline__ int find_problem_by_tile(const GemmProblem* pp, int np, long long t) {
    int pi = 0;
#pragma unroll 1
    for (int i = 1; i < np; ++i)
        if (t >= pp[i].tile_begin) pi = i;
    return pi;
}
// Stream-K split of the flattened tiles: CTA b holds q tiles, plus one if
// b < r (q = T / nctas, r = T % nctas, worked out on the host; T < 2^31).
__device__ __forceinline__ int range_start(int b, int q, int r) { return b * q + min(b, r); }
// CTA whose range holds flattened tile t.
__device__ __forceinline__ int range_owner(int t, int q, int r) {
    const int big = r * (q + 1);  // tiles of the first r CTAs
    return t < big ? t / (q + 1) : r + (t - big) / q;
}

// k tiles [ka, kb) of row tile rt of problem pi; flattened index of k tile ka.
struct Seg {
    int pi, rt, ka, kb;
    long long t0;
};

// The segment that holds flattened tile t_end - 1, clipped below at t_begin.
__device__ __forceinline__ void seg_ending_at(const GemmProblem* pp, int np, long long t_begin, long long t_end,
                                              Seg& s) {
    const long long t = t_end - 1;
    const int pi = find_problem_by_tile(pp, np, t);
    const GemmProblem& pr = pp[pi];
    const int local = static_cast<int>(t - pr.tile_begin);  // < nt * kt < 2^31
    const int rt = local / pr.kt;
    const long long r0 = pr.tile_begin + static_cast<long long>(rt) * pr.kt;
    const long long s0 = r0 > t_begin ? r0 : t_begin;
    s.pi = pi;
    s.rt = rt;
    s.ka = static_cast<int>(s0 - r0);
    s.kb = static_cast<int>(t_end - r0);
    s.t0 = s0;
}

// The tiles of a CTA's range in processing order: segments from the range's
// end to its start, k ascending inside each.
struct ProcIter {
    Seg s;
    int k;
    __device__ void init(const GemmProblem* pp, int np, long long t_begin, long long t_end) {
        seg_ending_at(pp, np, t_begin, t_end, s);
        k = s.ka;
    }
    __device__ void next(const GemmProblem* pp, int np, long long t_begin) {
        if (++k < s.kb) return;
        if (s.t0 > t_begin) {
            seg_ending_at(pp, np, t_begin, s.t0, s);
            k = s.ka;
        }
    }
};

// Position of local tile i (processing order) in the chunk ring and in the kNA
// A buffers, advanced one tile at a time (no division by the runtime ring size
// on the way to an MMA issue or a barrier wait).
template <int kNA>
struct RingPos {
    int cp;          // i % kChunk
    int q;           // (i / kChunk) % R: ring slot of the chunk
    uint32_t qph;    // ((i / kChunk) / R) & 1: phase of that slot's barriers
    int ab;          // i % kNA: A buffer
    int i;
    __device__ void reset() { cp = q = ab = i = 0; qph = 0u; }
    __device__ void next(int R) {
        ++i;
        if (++cp == kChunk) {
            cp = 0;
            if (++q == R) {
                q = 0;
                qph ^= 1u;
            }
        }
        if (++ab == kNA) ab = 0;
    }
    __device__ int slot() const { return q * kChunk + cp; }  // tile slot in the ring
};

// Bulk-copy the weight tiles of the next `count` tiles of `it` (processing
// order) into consecutive ring slots, one copy per run that is contiguous in
// global memory (the k tiles of one segment); all copies complete on `bar`.
// Run by a whole converged warp; only the lane with `on` set issues.
__device__ void issue_weights(const GemmProblem* pp, int np, long long t_begin, ProcIter& it, int count,
                              uint8_t* dst, uint32_t bar, uint64_t pol, uint32_t on) {
    mbar_arrive_expect_tx_if(on, bar, static_cast<uint32_t>(count * kTileBytes));
    int k = 0;
    while (k < count) {
        const GemmProblem& pr = pp[it.s.pi];
        const int run = min(count - k, it.s.kb - it.k);
        if (run <= 0) break;  // never: count never exceeds the tiles left
        const uint8_t* src = pr.pk + (static_cast<size_t>(it.s.rt) * pr.kt + it.k) * kTileBytes;
        bulk_g2s_if(on, smem_u32(dst + static_cast<size_t>(k) * kTileBytes), src,
                    static_cast<uint32_t>(run * kTileBytes), bar, pol);
        k += run;
        it.k += run - 1;
        it.next(pp, np, t_begin);
    }
}

// The same for the activation tiles (BT bytes each) of those tiles, from the
// preparation kernel's operand in the workspace (one tile per k tile of the
// problem): a run ends where the k index or the problem changes.
__device__ void issue_acts(const GemmProblem* pp, int np, long long t_begin, ProcIter& it, int count, int BT,
                           uint8_t* dst, uint32_t bar, uint64_t pol, uint32_t on) {
    mbar_arrive_expect_tx_if(on, bar, static_cast<uint32_t>(count * BT));
    int k = 0;
    while (k < count) {
        const int run = min(count - k, it.s.kb - it.k);
        if (run <= 0) break;  // never: count never exceeds the tiles left
        const uint8_t* src = pp[it.s.pi].actb + static_cast<size_t>(it.k) * BT;
        bulk_g2s_if(on, smem_u32(dst + static_cast<size_t>(k) * BT), src, static_cast<uint32_t>(run * BT), bar, pol);
        k += run;
        it.k += run - 1;
        it.next(pp, np, t_begin);
    }
}

// Element k of one activation row as fp32 (exact for all three kinds).
__device__ __forceinline__ float load_elem(int kind, const char* row, int k) {
    if (kind == BITMTP_F32) return reinterpret_cast<const float*>(row)[k];
    if (kind == BITMTP_BF16) return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[k]) << 16);
    return static_cast<float>(reinterpret_cast<const int8_t*>(row)[k]);
}

// The unit k0..k0+15 element by element (zero beyond K): the row's tail or a
// row that is not 16-byte aligned.  Kept out of line: rarely run, and its 48
// predicated loads would otherwise sit in every copy of the hot path.
__device__ __noinline__ void load16_tail(int kind, const char* row, int K, int k0, float* v) {
#pragma unroll 4
    for (int i = 0; i < 16; ++i) v[i] = (k0 + i < K) ? load_elem(kind, row, k0 + i) : 0.f;
}

// Load the 16-element unit k0..k0+15 of one row (zero beyond K): vector loads
// when the row is 16-byte aligned and the unit lies inside it, else element
// by element.
__device__ __forceinline__ void load16(const GemmProblem& pr, const char* row, bool vec_ok, int k0,
                                       float (&v)[16]) {
    if (vec_ok && k0 + 16 <= pr.K) {
        if (pr.act_kind == BITMTP_BF16) {
            const uint4* q = reinterpret_cast<const uint4*>(row + 2ll * k0);
            const uint4 a = q[0], b = q[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else if (pr.act_kind == BITMTP_F32) {
            const float4* q = reinterpret_cast<const float4*>(row + 4ll * k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 a = q[i];
                v[4 * i] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
            }
        } else {  // int8 codes
            const uint4 a = *reinterpret_cast<const uint4*>(row + k0);
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = static_cast<float>(static_cast<int8_t>(w[i / 4] >> (8 * (i % 4))));
        }
    } else {
        float t[16];
        load16_tail(pr.act_kind, row, pr.K, k0, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = t[i];
    }
}

__device__ __forceinline__ const char* act_row(const GemmProblem& pr, int m) {
    const int esize = pr.act_kind == BITMTP_F32 ? 4 : (pr.act_kind == BITMTP_BF16 ? 2 : 1);
    return static_cast<const char*>(pr.x) + static_cast<long long>(m) * pr.ldx * esize;
}

// ---------------------------------------------------- activation operand --
// One CTA per (problem, row m < btile_rows).  Writes row m of every
// activation tile of the problem (zeros for m >= M and beyond K), on the
// dp4a path the prefix sums rsp[m][0..kt] of the row's codes over k tiles,
// and asc[m].  Each
// thread owns whole 16-k units; rows of up to kPass units (K <= 16384) stay in
// registers between the absmax and the quantisation (one pass over the row),
// longer rows are read twice.  512 threads, at most 64 registers each.
template <int PATH, int DPR>
__global__ void __launch_bounds__(kPrepThreads, 2)  // <= 64 registers
act_prep_kernel(const __grid_constant__ GemmParams P) {
    constexpr int kRows = btile_rows(PATH, DPR);
    constexpr int kBRows = btile_brows(PATH, DPR);
    constexpr int BT = btile_bytes(PATH, DPR);
    constexpr int kPass = kPrepThreads * kPrepUnits;  // 16-element units per pass
    constexpr bool kF8 = PATH == kPathF8;             // E4M3 values instead of int8 codes
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
    const int nunits = pr.kt * 8;  // 16-element units, the zero tail of the last tile included
    const int npass = (nunits + kPass - 1) / kPass;

    // The activations may come from the previous kernel on the stream, and the
    // previous GEMM on this workspace may still be reading it.
    pdl_wait();
    // this call's epilogues combine the output rows' absmax into amax_out
    if (tid == 0 && pr.amax_out && m < pr.M) pr.amax_out[m] = 0.f;
    // a layer chain hands over the rows' absmax: no absmax pass
    const bool have_amax = raw && pr.amax_in != nullptr;

    float v[kPrepUnits][16];
    float amax = 0.f, s = 0.f;
    if (have_amax) {
        amax = live ? __ldcg(pr.amax_in + m) : 0.f;
        s = kF8 ? fp8_quant_scale(amax) : quant_scale(amax);
    }
    // Passes 0..npass-1 find the row's absmax; the quantisation then takes
    // the last pass first, from the values still in registers, and reads the
    // row again only for the earlier ones.  One loop, so that the loads are
    // compiled once.
    for (int it = have_amax ? npass : 0; it < 2 * npass; ++it) {
        const bool quant = it >= npass;
        const int ps = !quant ? it : (it == npass ? npass - 1 : it - npass - 1);
        if (!quant || ps != npass - 1 || have_amax) {
#pragma unroll
            for (int j = 0; j < kPrepUnits; ++j) {
                const int u = ps * kPass + j * kPrepThreads + tid;
                if (live && u < nunits) {
                    load16(pr, row, vec_ok, u * 16, v[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[j][i] = 0.f;
                }
            }
        }
        if (!quant) {
            if (raw) {
#pragma unroll
                for (int j = 0; j < kPrepUnits; ++j)
#pragma unroll
                    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[j][i]));
            }
            if (it == npass - 1) {  // uniform over the block
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                if (lane == 0) red[warp] = amax;
                __syncthreads();
                amax = red[0];
#pragma unroll
                for (int w = 1; w < kPrepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
                s = kF8 ? fp8_quant_scale(amax) : quant_scale(amax);
            }
            continue;
        }
        // Eight consecutive threads cover one k tile; units per pass and units
        // of the row are multiples of 8, so the 8-lane sums below see whole
        // tiles (the dp4a path's code sums; the tensor paths correct for the
        // weight offset with an MMA instead).
#pragma unroll
        for (int j = 0; j < kPrepUnits; ++j) {
            if (ps * kPass + j * kPrepThreads >= nunits) break;  // uniform over the block
            const int u = ps * kPass + j * kPrepThreads + tid;
            const bool uv = u < nunits;
            if constexpr (kF8) {
                // operand row m: E4M3(RN32(x * s)), rounded by the conversion
                // (an all-zero row has s = 0); register si holds k = {2si,
                // 2si+8, 2si+1, 2si+9} as below
                uint8_t* unit = pr.actb + static_cast<size_t>(u >> 3) * BT + (u & 7) * (kBRows * 16);
                uint32_t er[4];
#pragma unroll
                for (int si = 0; si < 4; ++si) {
                    const int k0 = 2 * si, k1 = 2 * si + 8, k2 = 2 * si + 1, k3 = 2 * si + 9;
                    er[si] = e4m3x2(__fmul_rn(v[j][k0], s), __fmul_rn(v[j][k1], s)) |
                             (e4m3x2(__fmul_rn(v[j][k2], s), __fmul_rn(v[j][k3], s)) << 16);
                }
                if (uv) *reinterpret_cast<uint4*>(unit + m * 16) = make_uint4(er[0], er[1], er[2], er[3]);
                continue;
            }
            // codes as exact small floats: clamp(rint(RN(x * s))) gives the same
            // values as the integer quantiser (quant.cuh), without conversions
            float qf[16];
            float fsum = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                qf[i] = raw ? ((amax > 0.f) ? fminf(fmaxf(rintf(__fmul_rn(v[j][i], s)), -127.f), 127.f) : 0.f)
                            : v[j][i];
                fsum += qf[i];
            }
            int rsum = static_cast<int>(fsum);  // |sum| <= 2032: exact
            const int kt = u >> 3;
            uint8_t* unit = pr.actb + static_cast<size_t>(kt) * BT + (u & 7) * (kBRows * 16);
            // register si of a unit row holds k = {2si, 2si+8, 2si+1, 2si+9}
            if constexpr (PATH == kPathDP) {
                uint32_t reg[4];
#pragma unroll
                for (int si = 0; si < 4; ++si) {
                    const uint32_t b0 = static_cast<uint32_t>(static_cast<int>(qf[2 * si])) & 0xFFu;
                    const uint32_t b1 = static_cast<uint32_t>(static_cast<int>(qf[2 * si + 8])) & 0xFFu;
                    const uint32_t b2 = static_cast<uint32_t>(static_cast<int>(qf[2 * si + 1])) & 0xFFu;
                    const uint32_t b3 = static_cast<uint32_t>(static_cast<int>(qf[2 * si + 9]));
                    reg[si] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
                }
                if (uv) *reinterpret_cast<uint4*>(unit + m * 16) = make_uint4(reg[0], reg[1], reg[2], reg[3]);
            } else {
                // operand row m: high parts h = floor(q / 16); row m + kRows: low
                // parts l = q - 16 h; both exact small floats, e4m3 bytes
                float h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) h[i] = floorf(qf[i] * 0.0625f);
                uint32_t hr[4], lr[4];
#pragma unroll
                for (int si = 0; si < 4; ++si) {
                    const int k0 = 2 * si, k1 = 2 * si + 8, k2 = 2 * si + 1, k3 = 2 * si + 9;
                    hr[si] = e4m3x2(h[k0], h[k1]) | (e4m3x2(h[k2], h[k3]) << 16);
                    lr[si] = e4m3x2(fmaf(h[k0], -16.f, qf[k0]), fmaf(h[k1], -16.f, qf[k1])) |
                             (e4m3x2(fmaf(h[k2], -16.f, qf[k2]), fmaf(h[k3], -16.f, qf[k3])) << 16);
                }
                if (uv) {
                    *reinterpret_cast<uint4*>(unit + m * 16) = make_uint4(hr[0], hr[1], hr[2], hr[3]);
                    *reinterpret_cast<uint4*>(unit + (m + kRows) * 16) = make_uint4(lr[0], lr[1], lr[2], lr[3]);
                }
            }
            if constexpr (PATH == kPathDP) {
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
                if (uv && (tid & 7) == 0) tsum[kt] = rsum;
            }
        }
    }
    __syncthreads();

    // rsp[m][0] = 0, rsp[m][t + 1] = codes of k tiles 0..t summed (dp4a
    // path only)
    if (PATH != kPathDP) {
        if (tid == 0)
            pr.asc[m] = kF8 ? fp8_dequant_scale(amax)
                            : (raw ? dequant_scale(amax) : (live ? pr.a_scale_in[m] : 0.f));
    } else if (warp == 0) {
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

// ------------------------------------------------ fused activation tiles --
// Layer-chain mode of the dp4a path (every problem brings its rows' absmax):
// the GEMM writes the activation tiles of its ring itself, from the raw rows,
// with the quantiser and byte order of the preparation kernel, instead of the
// producer copying a preparation kernel's output.  Chunk j holds the tiles
// whose weights the producer's chunk j brings (processing order).  Unit g of
// a chunk (0 <= g < 32 * DPR) is 16-k unit g % 8 of operand row (g / 8) % DPR
// of chunk tile g / (8 * DPR); the eight consecutive units of one (tile, row)
// sum its codes into Rs[tile slot][row] for the consumers' u = T + 1
// correction.  The consumer warps quantise chunk 0 (one unit per thread:
// they would only wait for it), warp 5 the later chunks, one unit per lane
// and pass, ahead of the consumers.

// Codes of one unit into `dst` (16 bytes; register si holds k = {2si, 2si+8,
// 2si+1, 2si+9}); returns their sum.  q = clamp(rint(RN(x * s)), -127, 127)
// in integers, the same values as the preparation kernel's float steps.
__device__ __forceinline__ int quant_unit(const float (&v)[16], float sc, uint8_t* dst, bool store) {
    int q[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) q[e] = max(-127, min(127, __float2int_rn(__fmul_rn(v[e], sc))));
    uint32_t reg[4];
    int sum = 0;
#pragma unroll
    for (int si = 0; si < 4; ++si) {
        reg[si] = (static_cast<uint32_t>(q[2 * si]) & 0xFFu) | ((static_cast<uint32_t>(q[2 * si + 8]) & 0xFFu) << 8) |
                  ((static_cast<uint32_t>(q[2 * si + 1]) & 0xFFu) << 16) | (static_cast<uint32_t>(q[2 * si + 9]) << 24);
        sum = __dp4a(static_cast<int>(reg[si]), 0x01010101, sum);
    }
    if (store) *reinterpret_cast<uint4*>(dst) = make_uint4(reg[0], reg[1], reg[2], reg[3]);
    return sum;
}

// Chunk 0 by the consumer warps: thread tid < 32 * DPR quantises unit tid.
template <int DPR>
__device__ __noinline__ void fused_chunk0(const GemmProblem* pp, int np, long long t_begin, long long t_end,
                                             uint8_t* tiles, int* rs, int tid) {
    constexpr int BT = btile_bytes(kPathDP, DPR);
    const int nloc = static_cast<int>(t_end - t_begin);
    const int cnt = min(kChunk, nloc);
    const int ti = tid / (8 * DPR), m = (tid >> 3) % DPR;
    ProcIter it;
    it.init(pp, np, t_begin, t_end);
    for (int z = 0; z < ti && z + 1 < cnt; ++z) it.next(pp, np, t_begin);
    const GemmProblem& pr = pp[it.s.pi];
    const bool live = ti < cnt && m < pr.M;
    float v[16];
    float amax = 0.f;
    if (live) {
        amax = __ldcg(pr.amax_in + m);
        load16(pr, act_row(pr, m), pr.vec_ok != 0, it.k * kTileK + (tid & 7) * 16, v);
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
    }
    int rsum = quant_unit(v, quant_scale(amax), tiles + static_cast<size_t>(ti) * BT + (tid & 7) * (DPR * 16) + m * 16,
                          ti < cnt);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
    if (ti < cnt && (tid & 7) == 0) rs[ti * 4 + m] = rsum;
}

// Chunks 1.. by warp 5.  Per chunk all of a lane's loads are issued first,
// unconditionally (one round trip to L2 per chunk): units that are not whole
// aligned vectors read a harmless aligned dummy and are reloaded element by
// element afterwards (the rare tail).  The quantisation then runs as a rolled
// loop (the unit's registers shifted down each pass): this code runs once
// per chunk and warp, and its size, not its arithmetic, sets its speed.
// kWide: some problem of the launch has fp32 rows (four 16-byte loads per
// unit instead of two).  One call covers the kPer units i0 .. i0 + kPer - 1
// of the lane.
template <int DPR, bool kWide, int kPer>
__device__ __forceinline__ void fused_chunk(const GemmProblem* pp, const int (&tp)[kChunk], const int (&tk)[kChunk],
                                            int cnt, int m, int lane, int i0, const uint4* dummy, uint8_t* tiles,
                                            int* rs) {
    constexpr int BT = btile_bytes(kPathDP, DPR);
    constexpr int kLd = kWide ? 4 : 2;
    uint4 raw[kPer][kLd];
    int pis[kPer], k0s[kPer];
    bool vec[kPer], live[kPer];
    // the row's absmax for the chunk's first problem (every CTA reads the same
    // few words: one load per chunk, not per unit)
    const GemmProblem& p0 = pp[tp[0]];
    const float am0 = __ldcg(m < p0.M ? p0.amax_in + m : reinterpret_cast<const float*>(dummy));
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int ti = ((i0 + i) * 32 + lane) / (8 * DPR);
        int pi = 0, kk = 0;
#pragma unroll
        for (int z = 0; z < kChunk; ++z)
            if (z == ti) {
                pi = tp[z];
                kk = tk[z];
            }
        const GemmProblem& pr = pp[pi];
        pis[i] = pi;
        k0s[i] = kk * kTileK + (lane & 7) * 16;
        live[i] = ti < cnt && m < pr.M;
        vec[i] = live[i] && pr.vec_ok != 0 && k0s[i] + 16 <= pr.K;
        const bool f32 = pr.act_kind == BITMTP_F32;
        const uint4* src = vec[i] ? reinterpret_cast<const uint4*>(act_row(pr, m) + (f32 ? 4ll : 2ll) * k0s[i])
                                  : dummy;
        raw[i][0] = __ldcg(src);
        raw[i][1] = __ldcg(src + 1);
        if constexpr (kWide) {
            const uint4* src2 = (vec[i] && f32) ? src + 2 : src;
            raw[i][2] = __ldcg(src2);
            raw[i][3] = __ldcg(src2 + 1);
        }
    }
#pragma unroll 1
    for (int i = 0; i < kPer; ++i) {
        const int ti = ((i0 + i) * 32 + lane) / (8 * DPR);
        const GemmProblem& pr = pp[pis[0]];
        const bool f32 = pr.act_kind == BITMTP_F32;
        float v[16];
        if constexpr (kWide) {
            if (f32) {
                const uint32_t w[16] = {raw[0][0].x, raw[0][0].y, raw[0][0].z, raw[0][0].w,
                                        raw[0][1].x, raw[0][1].y, raw[0][1].z, raw[0][1].w,
                                        raw[0][2].x, raw[0][2].y, raw[0][2].z, raw[0][2].w,
                                        raw[0][3].x, raw[0][3].y, raw[0][3].z, raw[0][3].w};
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(w[e]);
            }
        }
        if (!f32) {
            const uint32_t w[8] = {raw[0][0].x, raw[0][0].y, raw[0][0].z, raw[0][0].w,
                                   raw[0][1].x, raw[0][1].y, raw[0][1].z, raw[0][1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[2 * e] = __uint_as_float(w[e] << 16);
                v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
        if (!vec[0]) {
            float t[16];
            if (live[0]) {
                load16_tail(pr.act_kind, act_row(pr, m), pr.K, k0s[0], t);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) t[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = t[e];
        }
        float amax = am0;
        if (pis[0] != tp[0]) amax = __ldcg(pr.amax_in + m);  // a problem boundary inside the chunk
        if (!live[0]) amax = 0.f;
        int rsum = quant_unit(v, quant_scale(amax),
                              tiles + static_cast<size_t>(ti) * BT + (lane & 7) * (DPR * 16) + m * 16, ti < cnt);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
        if (ti < cnt && (lane & 7) == 0) rs[ti * 4 + m] = rsum;
        // the next unit into position 0
#pragma unroll
        for (int k = 0; k + 1 < kPer; ++k) {
#pragma unroll
            for (int l = 0; l < kLd; ++l) raw[k][l] = raw[k + 1][l];
            pis[k] = pis[k + 1];
            k0s[k] = k0s[k + 1];
            vec[k] = vec[k + 1];
            live[k] = live[k + 1];
        }
    }
}

template <int DPR>
__device__ void fused_act_tiles(const GemmParams& P, Ctrl* c, const GemmProblem* pp, int np, long long t_begin,
                                long long t_end, int R, uint8_t* Br, int* Rs, int lane) {
    constexpr int BT = btile_bytes(kPathDP, DPR);
    const int nloc = static_cast<int>(t_end - t_begin);
    const int nchunks = (nloc + kChunk - 1) / kChunk;
    if (nchunks < 2) return;  // chunk 0 is the consumer warps'
    const int m = (lane >> 3) % DPR;  // the lane's operand row, the same for all its units
    bool wide = false;
    for (int i = 0; i < np; ++i) wide = wide || pp[i].act_kind == BITMTP_F32;
    // an aligned address that is always valid to read (this CTA's own
    // partial-sum slot): the target of loads whose results are not used
    const uint4* dummy = reinterpret_cast<const uint4*>(P.slots) + static_cast<size_t>(blockIdx.x) * 4 * kTileN;
    ProcIter it;
    it.init(pp, np, t_begin, t_end);
    for (int z = 0; z < kChunk; ++z) it.next(pp, np, t_begin);  // past chunk 0 (whole: nchunks >= 2)
    pdl_wait();  // the rows and their absmax come from the kernel before this one
    for (int j = 1; j < nchunks; ++j) {
        const int q = j % R;
        if (j >= R &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->empty[q]), ((j / R) - 1) & 1, P.wait_ns))) {
            if (lane == 0) fail(c, P.err, kErrWaitEmpty);
            return;
        }
        const int cnt = min(kChunk, nloc - j * kChunk);
        int tp[kChunk], tk[kChunk];  // problem and k tile of each chunk tile
#pragma unroll
        for (int z = 0; z < kChunk; ++z) {
            tp[z] = it.s.pi;
            tk[z] = it.k;
            if (z < cnt) it.next(pp, np, t_begin);
        }
        uint8_t* tiles = Br + static_cast<size_t>(q) * kChunk * BT;
        int* rs = Rs + q * kChunk * 4;
        constexpr int kPer = DPR;  // units per lane and chunk (32 * DPR / 32)
        if (wide) {  // fp32 rows: half of the units per batch of loads (registers)
            constexpr int kHalf = kPer > 1 ? kPer / 2 : 1;
            for (int i0 = 0; i0 < kPer; i0 += kHalf)
                fused_chunk<DPR, true, kHalf>(pp, tp, tk, cnt, m, lane, i0, dummy, tiles, rs);
        } else {
            fused_chunk<DPR, false, kPer>(pp, tp, tk, cnt, m, lane, 0, dummy, tiles, rs);
        }
        __syncwarp();
        mbar_arrive_if(lane == 0, smem_u32(&c->bfull[q]));  // release: the tiles and sums above
    }
}

// ------------------------------------------------------------ epilogue --
// Store y[m][n] (and acc); returns |y[m][n]| as stored.
// The output fields of one problem, read once per segment into registers:
// the problem record lives in shared memory behind a generic pointer, and
// every generic store to y would otherwise force the compiler to read the
// record again before the next one.
struct OutRef {
    void* y;
    int32_t* acc;
    long long ldy, lda;
    float w_scale;
    bool f32;
};
__device__ __forceinline__ OutRef out_ref(const GemmProblem& pr) {
    OutRef o;
    o.y = pr.y;
    o.acc = pr.acc;
    o.ldy = pr.ldy;
    o.lda = pr.lda;
    o.w_scale = pr.w_scale;
    o.f32 = pr.out_dtype == BITMTP_F32;
    return o;
}

// Store y[m][n] (and acc); returns |y[m][n]| as stored.  kF: acc holds an
// fp32 accumulator's bit pattern (FP8 path), else an exact integer sum.
template <bool kF>
__device__ __forceinline__ float store_out(const OutRef& o, int m, int n, int acc, float a_scale) {
    const float a = kF ? __int_as_float(acc) : static_cast<float>(acc);
    const float v = __fmul_rn(__fmul_rn(a, a_scale), o.w_scale);
    const long long off = static_cast<long long>(m) * o.ldy + n;
    float stored = v;
    if (o.f32) {
        static_cast<float*>(o.y)[off] = v;
    } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        static_cast<__nv_bfloat16*>(o.y)[off] = h;
        stored = __bfloat162float(h);
    }
    if (o.acc) o.acc[static_cast<long long>(m) * o.lda + n] = acc;
    return fabsf(stored);
}

// Partial-sum slot of CTA b: four groups of four rows, one int4 per column in
// each, columns consecutive (a warp's stores and loads cover 512 contiguous
// bytes; a narrow block touches only the groups its rows occupy).
__device__ __forceinline__ int4* slot_ptr(const GemmParams& P, int b, int g, int col) {
    return reinterpret_cast<int4*>(P.slots) + (static_cast<size_t>(b) * 4 + g) * kTileN + col;
}

// Bounded wait for another CTA's flag (acquire at GPU scope).
__device__ __forceinline__ bool wait_flag(const unsigned* f, unsigned long long limit_ns) {
    if (ld_acquire_gpu(f) != 0u) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (ld_acquire_gpu(f) != 0u) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// The same wait with a pause between polls, for a word that every CTA of
// the launch polls at once: back-to-back polls from every SM would queue at
// the word's L2 slice ahead of the loads the other warps need.
__device__ __forceinline__ bool wait_flag_backoff(const unsigned* f, unsigned long long limit_ns) {
    if (ld_acquire_gpu(f) != 0u) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        __nanosleep(100);
        if (ld_acquire_gpu(f) != 0u) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Segment roles: the whole row tile, the tail that finishes a row tile begun
// by earlier CTAs (owner), or a part that another CTA finishes (contributor).
enum SegRole : int { kWhole = 0, kOwner = 1, kContrib = 2 };

__device__ __forceinline__ int seg_role(const Seg& s, const GemmProblem& pr) {
    if (s.kb < pr.kt) return kContrib;
    return s.ka == 0 ? kWhole : kOwner;
}

// Partial sums of one output: integers, or fp32 bit patterns (kF).
template <bool kF>
__device__ __forceinline__ int acc_add(int a, int b) {
    return kF ? __float_as_int(__fadd_rn(__int_as_float(a), __int_as_float(b))) : a + b;
}

// Finish one segment.  acc[m]: the exact sum_k T*q of the segment for the
// thread's output column (row tile column tid) and block row m (kF: the fp32
// sum_k T*e of the FP8 path, as bit patterns; contributors' partial sums are
// then added in CTA order).  kRows: the
// compute path's rows per tile, a compile-time bound on M that keeps the
// unrolled row loops (and the code) short.  owner_first: the first CTA of the
// owner segment's row tile.  Every consumer thread calls it with the same
// segment (the named barriers below need all four warps).
template <int kRows, bool kF>
__device__ void segment_epilogue(const GemmParams& P, Ctrl* c, int p_lo, const Seg& s, int owner_first,
                                 int (&acc)[16], int tid, bool& alive) {
    const GemmProblem& pr = c->prob[s.pi];
    const int M = pr.M;
    const int n = s.rt * kTileN + tid;
    const int role = seg_role(s, pr);
    const int b = blockIdx.x;
    constexpr int kGroups = (kRows + 3) / 4;
    if (role == kContrib) {
        // the partial sums of this CTA's slot; warp 4 publishes the flag
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
            if (alive && 4 * g < M)
                *slot_ptr(P, b, g, tid) = make_int4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(smem_u32(&c->slot_done));
        return;
    }
    if (role == kOwner) {
        // thread i waits for contributor owner_first + i (all at once)
        if (tid == 0) c->owner_ok = 1;
        named_bar_sync(kBarEpi, 128);
        for (int cc = owner_first + tid; cc < b; cc += 128) {
            const bool ok = alive && wait_flag(P.flags + static_cast<size_t>(cc) * kFlagStride, P.wait_ns);
            if (ok) {
                P.flags[static_cast<size_t>(cc) * kFlagStride] = 0u;  // consumed (no CTA of this launch sets it again)
            } else {
                c->owner_ok = 0;
                if (alive) fail(c, P.err, kErrWaitFlag);
            }
        }
        named_bar_sync(kBarEpi, 128);
        alive = alive && c->owner_ok;
        if (alive) {
            // a long row tile split over many short CTA ranges has many
            // contributors: on the dp4a path (one group of rows, integer sums)
            // their slots are read kBatch at a time, every load of a batch in
            // flight together (absent ones read as zero)
            constexpr int kBatch = 8;
            int cc = owner_first;
            if constexpr (kGroups == 1 && !kF) {
                for (; cc < b; cc += kBatch) {
                    int4 v[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u)
                        v[u] = (cc + u < b) ? __ldcg(slot_ptr(P, cc + u, 0, tid)) : make_int4(0, 0, 0, 0);
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        acc[0] += v[u].x;
                        acc[1] += v[u].y;
                        acc[2] += v[u].z;
                        acc[3] += v[u].w;
                    }
                }
            }
            // the tensor paths, in CTA order: two contributors per step at 16
            // rows, one at 8 (the faster form of each, measured)
            constexpr int kStep = kGroups == 4 ? 2 : 1;
            for (; cc < b; cc += kStep) {
                int4 v[kStep][kGroups];
#pragma unroll
                for (int u = 0; u < kStep; ++u)
#pragma unroll
                    for (int g = 0; g < kGroups; ++g)
                        v[u][g] = (cc + u < b && 4 * g < M) ? __ldcg(slot_ptr(P, cc + u, g, tid))
                                                            : make_int4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < kStep; ++u) {
                    if (cc + u < b) {
#pragma unroll
                        for (int g = 0; g < kGroups; ++g) {
                            if (4 * g < M) {
                                acc[4 * g] = acc_add<kF>(acc[4 * g], v[u][g].x);
                                acc[4 * g + 1] = acc_add<kF>(acc[4 * g + 1], v[u][g].y);
                                acc[4 * g + 2] = acc_add<kF>(acc[4 * g + 2], v[u][g].z);
                                acc[4 * g + 3] = acc_add<kF>(acc[4 * g + 3], v[u][g].w);
                            }
                        }
                    }
                }
            }
        }
    }
    float am[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) am[m] = 0.f;
    const OutRef o = out_ref(pr);
    float* const amax_out = pr.amax_out;
    if (alive && n < pr.N) {
        // the rows' scales, all read before the first store
        float asv[kRows];
#pragma unroll
        for (int m = 0; m < kRows; ++m) asv[m] = c->asc[s.pi - p_lo][m];
#pragma unroll
        for (int m = 0; m < kRows; ++m)
            if (m < M) am[m] = store_out<kF>(o, m, n, acc[m], asv[m]);
    }
    if (amax_out) {
        // first phase of the output rows' absmax: this warp's 32 columns, one
        // atomic per row (non-negative floats order like their bit patterns)
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            if (m < M) {
                float v = am[m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                if ((tid & 31) == 0 && v > 0.f)
                    atomicMax(reinterpret_cast<unsigned*>(amax_out + m), __float_as_uint(v));
            }
        }
    }
}

// The preparation kernel's prefix sums at k tiles ka and kb: lane m < 16
// loads row m at ka, lane 16 + m row m at kb (zero for rows >= M).  One load
// per lane, issued at the start of a segment; code_sum() reads the
// difference at its end.
__device__ __forceinline__ int load_code_sum_lane(const GemmProblem& pr, int ka, int kb, int lane) {
    const int m = lane & 15;
    return (m < pr.M) ? __ldcg(pr.rsp + m * (pr.kt + 1) + ((lane & 16) ? kb : ka)) : 0;
}
// Codes of row m summed over the segment (every lane must take part).
__device__ __forceinline__ int code_sum(int v, int m) {
    return __shfl_sync(0xffffffffu, v, 16 + m) - __shfl_sync(0xffffffffu, v, m);
}

template <int PATH, int DPR, bool kFused>
__global__ void __maxnreg__(gemm_max_regs(PATH))
w2a8_streamk_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr bool kTC = PATH != kPathDP;
    constexpr bool kF8 = PATH == kPathF8;  // fp32 accumulators (bit patterns in the int arrays)
    // fused activation tiles (the dp4a path only): a kernel of its own, so
    // the other kernels carry none of its code
    static_assert(!kFused || PATH == kPathDP, "fused mode is a dp4a-path mode");
    constexpr bool fused = kFused;
    unsigned* const sync_words = kFused ? P.sync_words : nullptr;
    constexpr int BT = btile_bytes(PATH, DPR);
    constexpr int kOutRows = btile_rows(PATH, DPR);  // M <= kOutRows (the host's path choice)
    constexpr uint32_t kDCols = tmem_d_cols(PATH, DPR);
    constexpr uint32_t kACol = tmem_a_col(PATH, DPR);
    constexpr int kATiles = tmem_a_tiles(PATH, DPR);
    constexpr uint32_t kNegCol = tmem_neg_col(PATH);
    static_assert(!kTC || (kATiles <= kMaxATiles && kATiles < kBatchBars && kDCols <= 32 &&
                           kACol + kATiles * kATileCols <= kNegCol), "tensor-memory layout");
    using RP = RingPos<kATiles>;
    Ctrl* c = reinterpret_cast<Ctrl*>(smem);
    const int R = P.stages;                                  // chunks in the ring
    uint8_t* Wr = smem + kCtrlBytes;                         // [R][kChunk][4096]
    uint8_t* Br = Wr + static_cast<size_t>(R) * kChunk * kTileBytes;  // [R][kChunk][BT]
    int* Rs = reinterpret_cast<int*>(Br + static_cast<size_t>(R) * kChunk * BT);  // dp4a fused: [R * kChunk][4]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b = blockIdx.x;
    const long long t_begin = range_start(b, P.tiles_q, P.tiles_r);
    const long long t_end = range_start(b + 1, P.tiles_q, P.tiles_r);
    const int nloc = static_cast<int>(t_end - t_begin);
    const int nchunks = (nloc + kChunk - 1) / kChunk;
    const int np = P.n_problems;

    // ------------------------------------------------------------ set-up --
    // the problem table, copied once into shared memory (word by word)
    static_assert(sizeof(GemmProblem) % 4 == 0, "problem record not word-sized");
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&P.p[0]);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&c->prob[0]);
        const int words = np * static_cast<int>(sizeof(GemmProblem) / 4);
        for (int z = tid; z < words; z += gemm_threads(PATH)) dst[z] = src[z];
    }
    const GemmProblem* pp = c->prob;
    // the mbarriers, one per thread (consecutive 8-byte words)
    static_assert(offsetof(Ctrl, slot_done) == offsetof(Ctrl, wfull) + 8 * (3 * kMaxRing + kBatchBars + kBatchBars + 8),
                  "mbarriers not consecutive");
    static_assert(offsetof(Ctrl, drained) == offsetof(Ctrl, slot_done) + 8, "mbarriers not consecutive");
    static_assert(offsetof(Ctrl, zero_ready) == offsetof(Ctrl, drained) + 16, "mbarriers not consecutive");
    if (tid < 3 * kMaxRing + kBatchBars + kBatchBars + 12) {
        uint32_t count = 1;                                            // wfull, bfull, mma_done, dfull, drained, zero_ready
        if (tid >= 2 * kMaxRing && tid < 3 * kMaxRing) count = kTC ? 2 : 4;          // empty
        else if (tid >= 3 * kMaxRing && tid < 3 * kMaxRing + kBatchBars) count = 4;  // a_full
        else if (tid == 3 * kMaxRing + kBatchBars + kBatchBars + 8) count = 4;          // slot_done
        mbar_init(smem_u32(&c->wfull[0]) + 8 * tid, count);
        fence_mbar_init();
    }
    if (tid == 0) {
        c->failed = 0;
        c->owner_ok = 0;
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
    const int p0 = find_problem_by_tile(pp, np, t_begin);
    const int p1 = find_problem_by_tile(pp, np, t_end - 1);

    const int npre = nchunks < R ? nchunks : R;
    int w_issued[kMaxRing], b_issued[kMaxRing];  // warp 4: chunk index + 1 of the last requests per slot
#pragma unroll
    for (int q = 0; q < kMaxRing; ++q) w_issued[q] = b_issued[q] = 0;

    // -------------------------------------------------------- main loop --
    if (warp == 4) {
        // The whole warp runs the producer loop; the elected lane issues.  A
        // CTA whose range ends inside a row tile also publishes that
        // segment's partial sums (processed first) once the consumer warps
        // have stored them: checked between refills, else waited for at the
        // end.
        const uint32_t leader = elect_one();
        Seg sl;
        seg_ending_at(pp, np, t_begin, t_end, sl);
        bool pending = seg_role(sl, pp[sl.pi]) == kContrib;
        auto publish = [&]() {
            if (leader && !c->failed) {
                __threadfence();  // the slot's stores before the flag
                *reinterpret_cast<volatile unsigned*>(P.flags + static_cast<size_t>(b) * kFlagStride) = 1u;
            }
            pending = false;
        };
        // weights first: they do not depend on the kernels before this one
        const uint64_t pol = policy_evict_first();
        ProcIter itw, ita;  // processing order
        itw.init(pp, np, t_begin, t_end);
        ita = itw;
        for (int j = 0; j < npre; ++j) {
            const bool withheld = P.withhold == j && b == 0;  // test only: never requested
            issue_weights(pp, np, t_begin, itw, min(kChunk, nloc - j * kChunk),
                          Wr + static_cast<size_t>(j) * kChunk * kTileBytes, smem_u32(&c->wfull[j]), pol,
                          withheld ? 0u : leader);
            if (!withheld) w_issued[j] = j + 1;
        }
        pdl_wait();  // the activation tiles are written by the preparation kernel
        const bool copy_acts = !fused;  // fused: the consumer warps and warp 5 write them
        const uint64_t pol_b = policy_evict_last();
        if (copy_acts) {
            for (int j = 0; j < npre; ++j) {
                issue_acts(pp, np, t_begin, ita, min(kChunk, nloc - j * kChunk), BT,
                           Br + static_cast<size_t>(j) * kChunk * BT, smem_u32(&c->bfull[j]), pol_b, leader);
                b_issued[j] = j + 1;
            }
        } else if (sync_words != nullptr) {
            // this launch's epilogues combine the output rows' absmax into
            // amax_out: CTA 0 zeroes it and sets sync word 0; every CTA waits
            // for the word here, long before its first epilogue, and passes
            // it on to its consumer warps by zero_ready
            if (b == 0) {
                for (int i = 0; i < np; ++i)
                    if (pp[i].amax_out != nullptr && lane < pp[i].M) pp[i].amax_out[lane] = 0.f;
                __syncwarp();
                if (leader) {
                    __threadfence();
                    *reinterpret_cast<volatile unsigned*>(sync_words) = 1u;
                }
            }
            if (leader) {
                if (!wait_flag_backoff(sync_words, P.wait_ns)) fail(c, P.err, kErrWaitZero);
                mbar_arrive(smem_u32(&c->zero_ready));
            }
            __syncwarp();
        }
        // refill ring slots as they are released
        for (int j = npre; j < nchunks; ++j) {
            const int q = j % R;
            // one answer for the whole warp: the lanes must agree on `pending`
            if (pending && __shfl_sync(0xffffffffu, mbar_test_wait(smem_u32(&c->slot_done), 0) ? 1u : 0u, 0))
                publish();
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->empty[q]), ((j / R) - 1) & 1, P.wait_ns))) {
                if (leader) fail(c, P.err, kErrWaitEmpty);
                break;
            }
            const int cnt = min(kChunk, nloc - j * kChunk);
            issue_weights(pp, np, t_begin, itw, cnt, Wr + static_cast<size_t>(q) * kChunk * kTileBytes,
                          smem_u32(&c->wfull[q]), pol, leader);
            w_issued[q] = j + 1;
            if (copy_acts) {
                issue_acts(pp, np, t_begin, ita, cnt, BT, Br + static_cast<size_t>(q) * kChunk * BT,
                           smem_u32(&c->bfull[q]), pol_b, leader);
                b_issued[q] = j + 1;
            }
        }
        if (pending) {
            if (__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->slot_done), 0, P.wait_ns))) {
                publish();
            } else if (leader) {
                fail(c, P.err, kErrWaitSlot);
            }
        }
        __syncwarp();
    } else if (warp >= 5) {
        // Tensor paths (the dp4a block's warp 5 idles).  Two MMA
        // warps: warp 5 issues the even MMA batches, warp 6 the odd ones (one
        // issuing warp cannot keep up: each tcgen05.mma holds it for tens of
        // ns).  Both accumulate into the segment's D buffer, which the consumer
        // warps zero before the segment's first A tile, so every MMA adds
        // (the order does not matter: every partial sum is a multiple of
        // 2^-9 below 2^15 in magnitude, so fp32 holds it exactly).  A batch
        // is up to kMmaBatch tiles of one segment; its issuer waits for the
        // activation tiles of every chunk it is the first to touch, then for
        // the batch's A tiles (a_full of the batch), issues the batch's MMAs as
        // straight-line code and commits mma_done.  Chunk slots and finished
        // segments need both warps: each commits `empty` at every chunk end
        // and its own dfull[.][s & 3] at every segment end s it passes (a
        // commit tracks only the committing thread's own MMAs).  A warp with
        // no batch in a short segment passes it at once, so it can run up to
        // two segments ahead of the epilogue's wait: four barriers per warp
        // keep its phases apart.  The whole warp runs the loop; the
        // elected lane issues through guard predicates.
        if constexpr (kTC) {
            static_assert(kMmaBatch == 2, "the issue loop below handles batches of one or two tiles");
            const int par = warp - 5;
            const uint32_t leader = elect_one();
            constexpr int kBR = btile_brows(PATH, DPR);
            constexpr uint32_t kIdesc = idesc_f16_f32(128, kBR);
            constexpr uint32_t kUnit = kBR * 16;                  // bytes of one 16-k unit
            const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(Br), kUnit, 128);
            constexpr uint64_t kStepDesc = (2 * kUnit) >> 4;      // 32 k further, in descriptor units
            constexpr uint64_t kTileDesc = static_cast<uint64_t>(BT) >> 4;
            RP rp;
            rp.reset();
            int nbatch = 0, seg = 0, my_chunk = -1;
            bool ok = true;
            long long cur_end = t_end;
            while (rp.i < nloc && ok) {
                Seg sg;
                seg_ending_at(pp, np, t_begin, cur_end, sg);
                cur_end = sg.t0;
                const int len = sg.kb - sg.ka;
                const uint32_t dcol = tmem + kAccCol + (seg & 1) * kDCols;
                for (int e = 0; e < len && ok;) {
                    const int nb = min(kMmaBatch, len - e);
                    RP r1 = rp;  // the batch's last tile
                    if (nb > 1) r1.next(R);
                    if ((nbatch & 1) == par) {
                        const int c0 = rp.i / kChunk, c1 = r1.i / kChunk;
                        if (c0 > my_chunk) {
                            ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->bfull[rp.q]), rp.qph, P.wait_ns));
                            my_chunk = c0;
                        }
                        if (ok && c1 > my_chunk) {
                            ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->bfull[r1.q]), r1.qph, P.wait_ns));
                            my_chunk = c1;
                        }
                        if (!ok) {
                            if (leader) fail(c, P.err, kErrWaitB);
                            break;
                        }
                        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->a_full[nbatch % kBatchBars]),
                                                                       (nbatch / kBatchBars) & 1, P.wait_ns));
                        if (!ok) {
                            if (leader) fail(c, P.err, kErrWaitAFull);
                            break;
                        }
                        tc_fence_after();
                        // k step j of a tile: A columns 8j, B units 2j and 2j + 1
                        const uint64_t b0 = bdesc0 + static_cast<uint64_t>(rp.slot()) * kTileDesc;
                        const uint32_t a0 = tmem + kACol + rp.ab * kATileCols;
                        mma_f8_ts_acc_if(leader, dcol, a0, b0, kIdesc);
                        mma_f8_ts_acc_if(leader, dcol, a0 + 8, b0 + kStepDesc, kIdesc);
                        mma_f8_ts_acc_if(leader, dcol, a0 + 16, b0 + 2 * kStepDesc, kIdesc);
                        mma_f8_ts_acc_if(leader, dcol, a0 + 24, b0 + 3 * kStepDesc, kIdesc);
                        {
                            // the correction: sum_k u*b*2^-9 - sum_k b*2^-9 =
                            // 2^-9 * sum_k T*b for every operand row b
                            const uint32_t an = tmem + kNegCol;
                            mma_f8_ts_acc_if(leader, dcol, an, b0, kIdesc);
                            mma_f8_ts_acc_if(leader, dcol, an, b0 + kStepDesc, kIdesc);
                            mma_f8_ts_acc_if(leader, dcol, an, b0 + 2 * kStepDesc, kIdesc);
                            mma_f8_ts_acc_if(leader, dcol, an, b0 + 3 * kStepDesc, kIdesc);
                        }
                        const uint32_t on1 = nb > 1 ? leader : 0u;
                        const uint64_t b1 = bdesc0 + static_cast<uint64_t>(r1.slot()) * kTileDesc;
                        const uint32_t a1 = tmem + kACol + r1.ab * kATileCols;
                        mma_f8_ts_acc_if(on1, dcol, a1, b1, kIdesc);
                        mma_f8_ts_acc_if(on1, dcol, a1 + 8, b1 + kStepDesc, kIdesc);
                        mma_f8_ts_acc_if(on1, dcol, a1 + 16, b1 + 2 * kStepDesc, kIdesc);
                        mma_f8_ts_acc_if(on1, dcol, a1 + 24, b1 + 3 * kStepDesc, kIdesc);
                        {
                            const uint32_t an = tmem + kNegCol;
                            mma_f8_ts_acc_if(on1, dcol, an, b1, kIdesc);
                            mma_f8_ts_acc_if(on1, dcol, an, b1 + kStepDesc, kIdesc);
                            mma_f8_ts_acc_if(on1, dcol, an, b1 + 2 * kStepDesc, kIdesc);
                            mma_f8_ts_acc_if(on1, dcol, an, b1 + 3 * kStepDesc, kIdesc);
                        }
                        mma_commit_if(leader, smem_u32(&c->mma_done[nbatch % kBatchBars]));
                    }
                    // chunk ends inside the batch: this warp's MMAs so far read them
                    if (rp.cp == kChunk - 1 || rp.i == nloc - 1) mma_commit_if(leader, smem_u32(&c->empty[rp.q]));
                    if (nb > 1 && (r1.cp == kChunk - 1 || r1.i == nloc - 1)) mma_commit_if(leader, smem_u32(&c->empty[r1.q]));
                    ++nbatch;
                    rp = r1;
                    rp.next(R);
                    e += nb;
                }
                if (!ok) break;
                mma_commit_if(leader, smem_u32(&c->dfull[par][seg & 3]));
                ++seg;
            }
            if (!ok) {
                // tensor memory is freed at exit: first let every MMA this warp
                // issued complete (bounded)
                mma_commit_if(leader, smem_u32(&c->drained[par]));
                (void)mbar_wait_bounded(smem_u32(&c->drained[par]), 0, 100000000ull);
            }
        } else {
            if (fused) fused_act_tiles<DPR>(P, c, pp, np, t_begin, t_end, R, Br, Rs, lane);
        }
        __syncwarp();
    } else {
        // warps 0-3: one output row per thread, segment by segment.  A failed
        // (timed-out) wait only clears `alive`; every named barrier is still
        // executed by all four warps.
        // The owner segment (processed last) needs its row tile's first CTA:
        // worked out while the preparation kernel still runs.
        int owner_first = b;
        {
            Seg s0;
            seg_ending_at(pp, np, t_begin, t_begin + 1, s0);
            const GemmProblem& pa = pp[s0.pi];
            owner_first = range_owner(static_cast<int>(pa.tile_begin) + s0.rt * pa.kt, P.tiles_q, P.tiles_r);
        }
        pdl_wait();  // outputs and workspace: the preparation kernel has finished
        // dequant scales of problems p0..p1 (at most 8 x 16: one per thread),
        // first needed by the first epilogue, which stores and publishes them
        float asc_reg = 0.f;
        const bool asc_mine = tid < (p1 - p0 + 1) * 16;
        if (asc_mine) {
            const GemmProblem& pr = pp[p0 + tid / 16];
            if (tid % 16 < pr.M)
                asc_reg = __ldcg(fused ? pr.amax_in + tid % 16 : pr.asc + tid % 16);  // fused: the absmax
        }
        if constexpr (!kTC) {
            if (fused) {
                // chunk 0 of the ring, quantised here (warp 5 takes the later
                // ones); its bfull phase is then completed by hand, so the
                // loop below waits for it like for any other chunk
                if (tid < 32 * DPR) fused_chunk0<DPR>(pp, np, t_begin, t_end, Br, Rs, tid);
                named_bar_sync(kBarEpi, 128);
                if (tid == 0) mbar_arrive(smem_u32(&c->bfull[0]));
            }
        }
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        if constexpr (kTC) {
            // the constant A operand -2^-9 (e4m3 0x81) of the correction
            // MMAs; ordered before them by this warp's first A-tile arrival
            // (wait::st, fence, mbarrier)
            tmem_st8_fill(tmem + lane_base + kNegCol, 0x81818181u);
            tc_wait_st();
        }
        bool alive = true;
        int seg_idx = 0;
        RP rp;
        rp.reset();
        // MMA batch of each of the last kATiles tiles (the batch that must
        // complete before an A buffer is written again); batches never span
        // segments and hold up to kMmaBatch tiles, as in the MMA thread
        int hist[kATiles];
#pragma unroll
        for (int k = 0; k < kATiles; ++k) hist[k] = 0;
        int nbatch = 0;
        int waited = -1;  // the last MMA batch waited for
        bool first_epi = true;
        // Tensor paths: a segment's epilogue is deferred until kDeferTiles tiles
        // of the next segment are written (the accumulator is double-buffered),
        // so the MMA pipeline does not drain at row-tile boundaries.
        bool dv = false;
        Seg ds;
        ds.pi = ds.rt = ds.ka = ds.kb = 0;
        ds.t0 = 0;
        int d_seg = 0;
        auto epilogue = [&](const Seg& es, int (&acc)[16]) {
            if (first_epi) {  // publish the dequant scales once
                if (asc_mine) c->asc[tid / 16][tid % 16] = fused ? dequant_scale(asc_reg) : asc_reg;
                // fused: no atomic on amax_out before CTA 0 has zeroed it
                if (sync_words != nullptr && tid == 0 && alive &&
                    !mbar_wait_bounded(smem_u32(&c->zero_ready), 0, P.wait_ns))
                    fail(c, P.err, kErrWaitZero);
                named_bar_sync(kBarEpi, 128);
                if (sync_words != nullptr) alive = alive && !*reinterpret_cast<volatile int*>(&c->failed);
                first_epi = false;
            }
            segment_epilogue<kOutRows, kF8>(P, c, p0, es, owner_first, acc, tid, alive);
        };
        auto finish_deferred = [&]() {
            int acc[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = 0;
            if constexpr (kTC) {
                // both MMA warps have finished the segment
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (alive) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->dfull[w][d_seg & 3]),
                                                                          (d_seg >> 2) & 1, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitD);
                    }
                }
                if (alive) {
                    // D column m: high parts of row m; column m + kRows: low parts
                    constexpr int kRows = btile_rows(PATH, DPR);
                    const uint32_t dcol = tmem + lane_base + kAccCol + (d_seg & 1) * kDCols;
                    tc_fence_after();
                    uint32_t v[32];
                    tmem_ld16(dcol, *reinterpret_cast<uint32_t(*)[16]>(v));
                    if constexpr (kDCols == 32) tmem_ld16(dcol + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                    tc_wait_ld();
                    tc_fence_before();
                    if constexpr (kF8) {
                        // FP8: D column m is row m's fp32 sum of T * e * 2^-9
#pragma unroll
                        for (int m = 0; m < kRows; ++m) acc[m] = __float_as_int(__fmul_rn(__uint_as_float(v[m]), 512.f));
                    } else {
#pragma unroll
                        for (int m = 0; m < kRows; ++m) {
                            // D holds 2^-9 * sum_k T*h and 2^-9 * sum_k T*l, exact
                            const float d = __fadd_rn(__fmul_rn(__uint_as_float(v[m]), 16.f),
                                                      __uint_as_float(v[m + kRows]));
                            acc[m] = __float2int_rn(__fmul_rn(d, 512.f));
                        }
                    }
                }
            }
            epilogue(ds, acc);
            dv = false;
        };
        long long cur_end = t_end;
        while (rp.i < nloc) {
            Seg sg;
            seg_ending_at(pp, np, t_begin, cur_end, sg);
            cur_end = sg.t0;
            const GemmProblem& pr = pp[sg.pi];
            const int ka = sg.ka;
            const int len = sg.kb - sg.ka;
            const int rsl = (kTC || fused) ? 0 : load_code_sum_lane(pr, ka, ka + len, lane);
            int rs[DPR];  // fused: the segment's code sums, from Rs
#pragma unroll
            for (int m = 0; m < DPR; ++m) rs[m] = 0;
            int dacc[4][DPR];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
                for (int m = 0; m < DPR; ++m) dacc[s4][m] = 0;
            if constexpr (kTC) {
                // one MMA batch (up to two tiles) per iteration: both tiles'
                // shared loads in flight together, one wait for the stores,
                // one arrival for the batch
                static_assert(kMmaBatch == 2, "the writer loop below handles batches of one or two tiles");
                for (int e = 0; e < len;) {
                    const int nb = min(kMmaBatch, len - e);
                    if (dv && e <= kDeferTiles && kDeferTiles < e + nb) finish_deferred();
                    RP r1 = rp;  // the batch's last tile
                    if (nb > 1) r1.next(R);
                    if (alive && rp.cp == 0) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->wfull[rp.q]), rp.qph, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitW);
                    }
                    if (alive && nb > 1 && r1.cp == 0) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->wfull[r1.q]), r1.qph, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitW);
                    }
                    // the batches that last read the two A buffers (kATiles
                    // tiles back); the second usually equals the first
                    const int bn = nbatch + e / kMmaBatch;
                    const int prev0 = hist[0];
#pragma unroll
                    for (int k = 0; k + 1 < kATiles; ++k) hist[k] = hist[k + 1];
                    hist[kATiles - 1] = bn;
                    int prev1 = prev0;
                    if (nb > 1) {
                        prev1 = hist[0];
#pragma unroll
                        for (int k = 0; k + 1 < kATiles; ++k) hist[k] = hist[k + 1];
                        hist[kATiles - 1] = bn;
                    }
                    if (alive && rp.i >= kATiles && prev0 != waited) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->mma_done[prev0 % kBatchBars]),
                                                                          (prev0 / kBatchBars) & 1, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitAEmpty);
                        tc_fence_after();
                        waited = prev0;
                    }
                    if (alive && nb > 1 && r1.i >= kATiles && prev1 != waited) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->mma_done[prev1 % kBatchBars]),
                                                                          (prev1 / kBatchBars) & 1, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitAEmpty);
                        tc_fence_after();
                        waited = prev1;
                    }
                    if (alive) {
                        // the segment's accumulator starts at zero (both MMA
                        // warps only add); its previous use was read out by
                        // the epilogue of the segment two back
                        if (e == 0) {
                            const uint32_t dz = tmem + lane_base + kAccCol + (seg_idx & 1) * kDCols;
                            if constexpr (kDCols == 32) tmem_st32_fill(dz, 0u);
                            else tmem_st16_fill(dz, 0u);
                        }
                        const uint8_t* wa = Wr + static_cast<size_t>(rp.slot()) * kTileBytes + tid * 16;
                        const uint8_t* wb = Wr + static_cast<size_t>(r1.slot()) * kTileBytes + tid * 16;
                        const uint4 a0 = *reinterpret_cast<const uint4*>(wa);
                        const uint4 a1 = *reinterpret_cast<const uint4*>(wa + 2048);
                        uint4 b0 = a0, b1 = a1;
                        if (nb > 1) {
                            b0 = *reinterpret_cast<const uint4*>(wb);
                            b1 = *reinterpret_cast<const uint4*>(wb + 2048);
                        }
                        uint32_t r[32];  // A columns 4w + s: word w (16 k), register s
                        unpack_row_e4m3(a0, a1, r);
                        tmem_st32(tmem + lane_base + kACol + rp.ab * kATileCols, r);
                        if (nb > 1) {
                            unpack_row_e4m3(b0, b1, r);
                            tmem_st32(tmem + lane_base + kACol + r1.ab * kATileCols, r);
                        }
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        mbar_arrive_if(lane == 0, smem_u32(&c->a_full[bn % kBatchBars]));
                    }
                    rp = r1;
                    rp.next(R);
                    e += nb;
                }
            } else {
                for (int e = 0; e < len; ++e, rp.next(R)) {
                    const int s = rp.slot();
                    if (alive && rp.cp == 0) {
                        alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->wfull[rp.q]), rp.qph, P.wait_ns));
                        if (!alive && lane == 0) fail(c, P.err, kErrWaitW);
                        if (alive) {
                            alive = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c->bfull[rp.q]), rp.qph, P.wait_ns));
                            if (!alive && lane == 0) fail(c, P.err, kErrWaitB);
                        }
                    }
                    if (alive) {
                        const uint8_t* wst = Wr + static_cast<size_t>(s) * kTileBytes;
                        const uint8_t* bst = Br + static_cast<size_t>(s) * BT;
                        if (fused) {
                            const int4 rv = *reinterpret_cast<const int4*>(Rs + s * 4);
                            const int rva[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                            for (int m = 0; m < DPR; ++m) rs[m] += rva[m];
                        }
                        const uint4 w0 = *reinterpret_cast<const uint4*>(wst + tid * 16);
                        const uint4 w1 = *reinterpret_cast<const uint4*>(wst + 2048 + tid * 16);
                        const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint32_t w = wd[ch];
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
                        __syncwarp();
                        mbar_arrive_if(lane == 0 && (rp.cp == kChunk - 1 || rp.i == nloc - 1),
                                       smem_u32(&c->empty[rp.q]));
                    }
                }
            }
            if constexpr (kTC) {
                if (dv) finish_deferred();  // the previous segment, if this one was short
                ds = sg;
                d_seg = seg_idx;
                dv = true;
            } else {
                int acc[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) acc[m] = 0;
#pragma unroll
                for (int m = 0; m < DPR; ++m)
                    acc[m] = dacc[0][m] + (dacc[1][m] >> 2) + (dacc[2][m] >> 4) + (dacc[3][m] >> 6) -
                             (fused ? rs[m] : code_sum(rsl, m));
                epilogue(sg, acc);
            }
            ++seg_idx;
            nbatch += (len + kMmaBatch - 1) / kMmaBatch;
        }
        if (dv) finish_deferred();
    }

    // ------------------------------------------------------- tear-down --
    __syncthreads();
    if (sync_words != nullptr && tid == 0) {
        // every epilogue of this CTA has passed its wait on sync word 0: the
        // last CTA to get here resets both words for the next launch
        if (atomicAdd(sync_words + 1, 1u) == static_cast<unsigned>(P.nctas) - 1u) {
            atomicExch(sync_words, 0u);
            atomicExch(sync_words + 1, 0u);
        }
    }
    if (warp == 4 && lane == 0 && c->failed) {
        // never release shared memory with a bulk copy still in flight: wait
        // (bounded) for the last requested phase of every slot
        for (int q = 0; q < R; ++q) {
            if (w_issued[q] > 0)
                (void)mbar_wait_bounded(smem_u32(&c->wfull[q]), ((w_issued[q] - 1) / R) & 1, 100000000ull);
            if (b_issued[q] > 0)
                (void)mbar_wait_bounded(smem_u32(&c->bfull[q]), ((b_issued[q] - 1) / R) & 1, 100000000ull);
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

template <int PATH, int DPR, bool kFused>
cudaError_t launch_one(const GemmParams& prm, bool pdl, cudaStream_t stream) {
    auto kern = &w2a8_streamk_kernel<PATH, DPR, kFused>;
    // the opt-in shared-memory size, once per device (first-use races only
    // repeat the same call)
    static std::atomic<unsigned long long> configured{0ull};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (dev >= 64 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gemm_smem_bytes(PATH, DPR, kMaxRing)));
        if (e != cudaSuccess) return e;
        if (dev < 64) configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchAttribute attr[1] = {pdl_attr()};

    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(static_cast<unsigned>(prm.n_problems * btile_rows(PATH, DPR)), 1, 1);
    pc.blockDim = dim3(kPrepThreads, 1, 1);
    pc.dynamicSmemBytes = 0;
    pc.stream = stream;
    pc.attrs = attr;
    pc.numAttrs = pdl ? 1 : 0;
    if (!kFused) {
        e = cudaLaunchKernelEx(&pc, &act_prep_kernel<PATH, DPR>, prm);
        if (e != cudaSuccess) return e;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(prm.nctas), 1, 1);
    cfg.blockDim = dim3(gemm_threads(PATH), 1, 1);
    cfg.dynamicSmemBytes = gemm_smem_bytes(PATH, DPR, prm.stages);
    cfg.stream = stream;
    cfg.attrs = attr;
    // overlaps the kernel before it (the preparation kernel, or in fused mode
    // the caller's previous kernel when the caller allows it): only weights
    // are read before its wait
    cfg.numAttrs = (kFused && !pdl) ? 0 : 1;
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
           static_cast<size_t>(stages) * kChunk * (kTileBytes + btile_bytes(path, dp_rows)) +
           (path == kPathDP ? static_cast<size_t>(stages) * kChunk * 16 : 0);  // fused mode's code sums
}

cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, bool pdl, cudaStream_t stream) {
    if (path == kPathTC16) return launch_one<kPathTC16, 1, false>(prm, pdl, stream);
    if (path == kPathTC8) return launch_one<kPathTC8, 1, false>(prm, pdl, stream);
    if (path == kPathF8) return launch_one<kPathF8, 1, false>(prm, pdl, stream);
    const bool f = prm.fused != 0;
    if (dp_rows <= 1) return f ? launch_one<kPathDP, 1, true>(prm, pdl, stream) : launch_one<kPathDP, 1, false>(prm, pdl, stream);
    if (dp_rows <= 2) return f ? launch_one<kPathDP, 2, true>(prm, pdl, stream) : launch_one<kPathDP, 2, false>(prm, pdl, stream);
    return f ? launch_one<kPathDP, 4, true>(prm, pdl, stream) : launch_one<kPathDP, 4, false>(prm, pdl, stream);
}

}  // namespace bitmtp
