// internal.h -- declarations shared by the library's translation units (host side).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/bitmtp_linear.h"

namespace bitmtp {

constexpr int kTileN = 128;       // out-features per row tile (= TMEM lanes)
constexpr int kTileK = 128;       // in-features per k tile
constexpr int kTileBytes = 4096;  // packed bytes per (row tile, k tile)
constexpr int kMaxKtPerCta = 16;  // k tiles resident in one CTA's shared memory
constexpr int kMaxCluster = 16;   // split-K factor (CTAs per cluster)
constexpr int kGemmThreads = 160; // 4 producer/epilogue warps + 1 control warp

enum ComputePath : int { kPathTC = 0, kPathDP = 1 };

struct GemmProblem {
    const uint8_t* pk;
    const void* x;
    const float* a_scale;   // Q8 only
    void* y;
    int32_t* acc;           // optional
    long long ldx, ldy, lda;
    float w_scale;
    int N, K, M;
    int nt, kt;             // row tiles, k tiles
    int act_kind;           // BITMTP_F32 / BITMTP_BF16 / BITMTP_Q8
    int out_dtype;          // BITMTP_F32 / BITMTP_BF16
    int cluster_begin;      // first cluster (row tile) index of this problem in the grid
};

struct GemmParams {
    GemmProblem p[BITMTP_MAX_GROUP];
    int n_problems;
    int csize;              // CTAs per cluster = split-K factor
    int nkt_max;            // max k tiles of any CTA (sizes shared memory)
    int* err;               // device error word
};

// Shared-memory bytes a GEMM CTA needs for nkt_max resident k tiles.
size_t gemm_smem_bytes(int path, int nkt_max);

// Launch the GEMM kernel for params (already validated).  dp_rows selects the
// dp4a accumulator width (1, 2 or 4) for kPathDP.
cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, int total_clusters,
                        bool pdl, cudaStream_t stream);

// Device error word of the current device (cudaGetSymbolAddress of a
// file-scope __device__ int), or nullptr on failure.
int* device_error_word();

}  // namespace bitmtp
