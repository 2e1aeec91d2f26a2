// internal.h -- declarations shared by the library's translation units (host side).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/bitmtp_linear.h"

namespace bitmtp {

constexpr int kTileN = 128;       // out-features per row tile (= TMEM lanes)
constexpr int kTileK = 128;       // in-features per k tile
constexpr int kTileBytes = 4096;  // packed bytes per (row tile, k tile)
constexpr int kCtasPerSm = 2;     // persistent CTAs per SM

// Compute paths.  The activation operand ("B tile", one per k tile) is laid
// out for the path that consumes it.
enum ComputePath : int {
    kPathTC16 = 0,  // tcgen05, block width 9..16: B = 32 operand rows (h and l of 16 rows), 4096 B
    kPathTC8 = 1,   // tcgen05, block width 5..8:  B = 16 operand rows, 2048 B
    kPathDP = 2,    // dp4a, block width 1..4:     B = dp_rows rows of int8 codes, 128 B per row
    kPathF8 = 3,    // tcgen05, FP8 activations (any width 1..16): B = 16 rows of E4M3 values, 2048 B
};

// GEMM block: warps 0-3 compute + epilogue, 4 bulk copies; the tensor paths
// add warps 5 and 6, which issue the MMAs of alternate batches.
__host__ __device__ constexpr int gemm_threads(int path) { return path == kPathDP ? 192 : 224; }
// Register cap of a GEMM thread (no spills at these caps): two GEMM CTAs take
// 2 x 224 x 128 = 57,344 (tensor paths) or 2 x 192 x 120 = 46,080 (dp4a) of
// an SM's 65,536 registers.
__host__ __device__ constexpr int gemm_max_regs(int path) { return path == kPathDP ? 120 : 128; }

struct GemmProblem {
    const uint8_t* pk;
    const void* x;
    const float* a_scale_in;  // BITMTP_Q8 only
    void* y;
    int32_t* acc;             // optional
    long long ldx, ldy, lda;
    float w_scale;
    int N, K, M;
    int nt, kt;               // row tiles, k tiles
    int act_kind;             // BITMTP_F32 / BITMTP_BF16 / BITMTP_Q8
    int out_dtype;            // BITMTP_F32 / BITMTP_BF16
    int vec_ok;               // activation rows 16-byte aligned (base and row stride)
    long long tile_begin;     // first flattened (row tile, k tile) index of this problem
    // Activation operand in the workspace, written by the preparation kernel:
    uint8_t* actb;            // [kt] tiles in the compute path's layout
    int* rsp;                 // [16][kt + 1] prefix sums over k tiles of each row's codes
    float* asc;               // [16] per-row dequant scales (amax / 127)
    const float* amax_in;     // optional [M]: the rows' absmax, precomputed (layer chain)
    float* amax_out;          // optional [M]: receives max_n |y[m][n]| (zeroed by the preparation)
};

struct GemmParams {
    GemmProblem p[BITMTP_MAX_GROUP];
    int n_problems;
    int stages;               // chunks in the shared-memory ring
    int nctas;
    int withhold;             // test only: ring chunk CTA 0 never requests (-1: none)
    int fused;                // dp4a path, every row's absmax handed over: no preparation
                              // kernel; warp 5 quantises the activation tiles into the ring
    unsigned* sync_words;     // fused with an out.amax: [0] out.amax zeroed for this launch,
                              // [1] CTAs finished (both left at zero); else null
    int tiles_q, tiles_r;     // stream-K split: CTA b gets tiles_q tiles, plus one if b < tiles_r
    long long total_tiles;
    unsigned long long wait_ns;  // bound on every wait of the launch
    unsigned* flags;          // [kMaxCtas][kFlagStride] partial-sum-ready flags, word 0 of each (left at zero)
    int* slots;               // [kMaxCtas][4][128][4] int32 partial sums of split row tiles
    int* err;                 // device error word
};

constexpr int kMaxCtas = 320;         // persistent CTAs per launch (>= 2 per SM on GB300)
constexpr int kMinTilesPerCta = 4;    // fewer CTAs on small problems: fewer split row tiles

// Workspace: two sync words of the fused dp4a mode (bytes 0-7) and the
// partial-sum-ready flags (both must be zero when a launch starts; every
// launch leaves them at zero), one partial-sum slot per CTA, then one
// activation region per problem (sized by its k tiles).
constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
constexpr size_t kWsFlags = 256;
// One ready flag per 128-byte line: packed 32 to a line, every CTA's polls
// and stores went to a handful of L2 lines, and spreading them out made the
// 16-row calls 0.67 µs and the width-4 layer-chain calls 0.76 µs faster
// (measured).
constexpr int kFlagStride = 32;  // words
constexpr size_t kWsSlots = kWsFlags + static_cast<size_t>(kMaxCtas) * kFlagStride * 4;
constexpr size_t kWsAct = kWsSlots + static_cast<size_t>(kMaxCtas) * 16 * kTileN * 4;
// 4.5 KiB per k tile, not the 4 KiB the largest operand tile needs: with
// regions of exactly 4 KiB per tile a grouped call's problems started at
// offsets that made its width-4 dp4a calls ~3% slower (measured: where the
// L2 places the activation tiles that many CTAs read at once).
constexpr size_t act_tiles_bytes(int kt) { return align256(static_cast<size_t>(kt) * 4608); }
constexpr size_t act_rsp_bytes(int kt) { return align256(static_cast<size_t>(16) * (kt + 1) * 4); }
constexpr size_t act_region_bytes(int kt) { return act_tiles_bytes(kt) + act_rsp_bytes(kt) + 256; }

constexpr unsigned long long kWaitNs = 2000000000ull;      // 2 s: every wait of a normal launch
constexpr unsigned long long kTestWaitNs = 1000000ull;     // 1 ms: launches with BITMTP_FLAG_TEST_WITHHOLD

size_t gemm_smem_bytes(int path, int dp_rows, int stages);
int gemm_stages(int path, int dp_rows);

// Launch the activation preparation kernel, then the stream-K GEMM kernel
// (params validated and filled); in fused mode the GEMM kernel alone.  `pdl`
// lets the first of them overlap the kernel before it on the stream; the GEMM
// always overlaps the preparation kernel (it only streams weights before
// waiting for it).
cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, bool pdl, cudaStream_t stream);

}  // namespace bitmtp
