// internal.h -- declarations shared by the library's translation units (host side).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/bitmtp_linear.h"

namespace bitmtp {

constexpr int kTileN = 128;       // out-features per row tile (= TMEM lanes)
constexpr int kTileK = 128;       // in-features per k tile
constexpr int kTileBytes = 4096;  // packed bytes per (row tile, k tile)
constexpr int kGemmThreads = 192; // warps 0-3 compute, warp 4 bulk copies, warp 5 MMA issue
constexpr int kCtasPerSm = 2;     // persistent CTAs per SM

// Compute paths.  The activation operand ("B tile", one per k tile) is laid
// out for the path that consumes it.
enum ComputePath : int {
    kPathTC16 = 0,  // tcgen05, block width 9..16: B = 16 rows fp16, 4096 B
    kPathTC8 = 1,   // tcgen05, block width 3..8:  B = 8 rows fp16, 2048 B
    kPathDP = 2,    // dp4a, block width 1..4:     B = dp_rows rows int8, 128 B per row
};

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
    long long tile_begin;     // first flattened (row tile, k tile) index of this problem
    int task_begin;           // first activation-row task (rows_b per problem)
    int rt_begin;             // first row-tile counter
    int bt_begin;             // first B tile in the workspace
    int pre_begin;            // first row-sum prefix entry ((kt + 1) * 16 per problem)
};

struct GemmParams {
    GemmProblem p[BITMTP_MAX_GROUP];
    int n_problems;
    int rows_b;               // activation rows held per B tile
    int btile_bytes;
    int stages;               // shared-memory ring depth (k tiles)
    int total_tasks;          // activation rows to quantise (sum of M)
    int nctas;
    long long total_tiles;
    // workspace sections
    unsigned* gridbar;
    unsigned* counters;
    float* ascale;            // [total_tasks]
    int* prefix;              // row-sum prefixes
    float* accum;             // [kMaxCtas][128][16] split-row-tile accumulators
    uint8_t* btiles;          // activation operand tiles
    int* err;                 // device error word
};

// Workspace layout for a launch (sizes in bytes, sections 256-byte aligned).
struct WorkspaceLayout {
    size_t gridbar, counters, accum, ascale, prefix, btiles, total;
};
constexpr int kMaxCtas = 320;  // persistent CTAs per launch (>= 2 per SM on GB300)

size_t gemm_smem_bytes(int path, int dp_rows, int stages);
int gemm_stages(int path, int dp_rows);

// Launch the stream-K GEMM kernel (params validated and filled).
cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, bool pdl, cudaStream_t stream);

}  // namespace bitmtp
