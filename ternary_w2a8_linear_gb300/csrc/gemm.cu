// gemm.cu -- the W2A8 ternary linear on sm_103a.
//
// One kernel template, two compute paths that share the weight stream, the
// activation prologue and the split-K epilogue:
//
//   kPathTC  tcgen05 tensor cores, any block width 1..16.  Each producer
//            thread owns one output row (one TMEM lane), unpacks its 2-bit
//            codes straight into fp16 bit patterns with one mask per register
//            (the codes land in the fp16 subnormal range, value u * 4^J * 2^-24),
//            writes them to tensor memory (tcgen05.st) as the A operand, and one
//            thread issues tcgen05.mma (M=128, N=16, K=16) against the
//            activation block held in shared memory as fp16 pre-scaled by
//            2^(9-2J) per k position.  Every product is u*q*2^-15 exactly and
//            every partial sum stays below 2^24 * 2^-15, so the fp32
//            accumulator holds the exact integer sum.
//   kPathDP  integer dp4a for narrow blocks (1..4 rows): the same code words,
//            four byte masks per word and four int32 accumulators per row.
//
// With u = T + 1, sum_k T*q = sum_k u*q - sum_k q; the CTA subtracts the row
// sums of its own k slice.
//
// Work split: a cluster of `csize` CTAs owns one 128-row tile of the output;
// CTA r of the cluster owns k tiles [r*KT/csize, (r+1)*KT/csize).  The whole
// k slice of packed weights is fetched up front with 4 KiB bulk copies (TMA),
// so every byte the CTA needs is in flight from the first cycle.  Split-K
// partials (exact int32) are summed through distributed shared memory; the
// raw-activation absmax is exchanged the same way, so quantisation is fused
// without a second kernel or any global scratch.
//
// The operation is the packed W2A8 linear of "BitMTP: When Multi-Token
// Prediction Meets Low-Bit Large Language Models" (AI summary: Main Findings,
// first bullet -- 2-bit weights, 8-bit activations; Methodology in Plain
// English -- width-specialised packed low-bit operators).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace bitmtp {
namespace {

constexpr int kCtrlBytes = 1024;
constexpr int kPartBytes = 16 * kTileN * 4;   // int32 partials [16 rows][128 out-features]
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kAccCol = 0;               // D: columns 0..15 (fp32, one per block row)
constexpr uint32_t kACol = 32;                // A: two buffers of 32 columns (64 k each)
constexpr uint32_t kIdesc = idesc_f16_f32(128, 16);
constexpr int kTcSmemFloor = 48 * 1024;       // caps residency at 4 CTAs/SM -> 4 x 128 TMEM columns

enum : int {
    kErrWaitFull = 0x101,
    kErrWaitAFull = 0x102,
    kErrWaitAEmpty = 0x103,
    kErrWaitDone = 0x104,
};

struct Ctrl {
    uint64_t full[kMaxKtPerCta];
    uint64_t a_full[2];
    uint64_t a_empty[2];
    uint64_t done;
    uint32_t tmem_base;
    int failed;
    float amax_part[16];
    float a_scale[16];
    float qscale[16];
    int rowsum_part[16];
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

// fp16 pre-scale of the activation for code column c (J = 0,1,2,3,4,0,1,2).
__device__ __forceinline__ int bscale_shift(int c) {
    return 9 - 2 * ((c < 5) ? c : (c - 5));
}

__device__ __forceinline__ void fail(Ctrl* c, int* err, int code) {
    *reinterpret_cast<volatile int*>(&c->failed) = 1;
    atomicCAS(err, 0, code);
}
__device__ __forceinline__ bool failed(Ctrl* c) {
    return *reinterpret_cast<volatile int*>(&c->failed) != 0;
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

__device__ __forceinline__ void store_out(const GemmProblem& pr, int m, int n, int acc,
                                          float a_scale) {
    const float v = __fmul_rn(__fmul_rn(static_cast<float>(acc), a_scale), pr.w_scale);
    const long long o = static_cast<long long>(m) * pr.ldy + n;
    if (pr.out_dtype == BITMTP_F32) {
        static_cast<float*>(pr.y)[o] = v;
    } else {
        static_cast<__nv_bfloat16*>(pr.y)[o] = __float2bfloat16_rn(v);
    }
    if (pr.acc) pr.acc[static_cast<long long>(m) * pr.lda + n] = acc;
}

template <int PATH, int DPR>
__global__ void __launch_bounds__(kGemmThreads, 1)
w2a8_gemm_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
    uint8_t* Ws = smem + kCtrlBytes;
    uint8_t* Bs = Ws + static_cast<size_t>(P.nkt_max) * kTileBytes;
    int* part = reinterpret_cast<int*>(Bs + static_cast<size_t>(P.nkt_max) * kTileBytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int csize = P.csize;
    const int rank = (csize > 1) ? static_cast<int>(cluster_ctarank()) : 0;
    const int cl = blockIdx.x / csize;

    int pi = 0;
#pragma unroll 1
    for (int i = 1; i < P.n_problems; ++i)
        if (cl >= P.p[i].cluster_begin) pi = i;
    const GemmProblem& pr = P.p[pi];

    const int rt = cl - pr.cluster_begin;
    const int KT = pr.kt;
    const int kt0 = static_cast<int>(static_cast<long long>(rank) * KT / csize);
    const int kt1 = static_cast<int>(static_cast<long long>(rank + 1) * KT / csize);
    const int nkt = kt1 - kt0;
    const int M = pr.M;
    const int kbase = kt0 * kTileK;                    // first k of this CTA's slice
    const int kend = min(kt1 * kTileK, pr.K);          // end of valid k in the slice
    const bool raw = pr.act_kind != BITMTP_Q8;

    // ------------------------------------------------------------ set-up --
    if (tid == 0) {
        for (int s = 0; s < nkt; ++s) mbar_init(smem_u32(&ctrl->full[s]), 1);
        mbar_init(smem_u32(&ctrl->a_full[0]), 4);
        mbar_init(smem_u32(&ctrl->a_full[1]), 4);
        mbar_init(smem_u32(&ctrl->a_empty[0]), 1);
        mbar_init(smem_u32(&ctrl->a_empty[1]), 1);
        mbar_init(smem_u32(&ctrl->done), 1);
        ctrl->failed = 0;
        fence_mbar_init();
    }
    if (tid < 16) {
        ctrl->rowsum_part[tid] = 0;
        ctrl->amax_part[tid] = 0.f;
    }
    if constexpr (PATH == kPathTC) {
        if (warp == 0) {
            tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (PATH == kPathTC) tc_fence_after();
    const uint32_t tmem = (PATH == kPathTC) ? ctrl->tmem_base : 0u;

    // The packed weights do not depend on earlier kernels: start streaming now.
    if (warp == 4 && lane == 0 && nkt > 0) {
        const uint64_t pol = policy_evict_first();
        const uint8_t* src = pr.pk + (static_cast<size_t>(rt) * KT + kt0) * kTileBytes;
        for (int s = 0; s < nkt; ++s) {
            const uint32_t bar = smem_u32(&ctrl->full[s]);
            mbar_arrive_expect_tx(bar, kTileBytes);
            bulk_g2s(smem_u32(Ws + s * kTileBytes), src + static_cast<size_t>(s) * kTileBytes,
                     kTileBytes, bar, pol);
        }
    }
    __syncwarp();
    pdl_launch_dependents();

    // ------------------------------------- activation prologue (warps 0-3) --
    if (warp < 4) {
        pdl_wait();  // activations may come from the previous kernel on the stream
        if (raw) {
            for (int m = warp; m < M; m += 4) {
                float a = 0.f;
                for (int k = kbase + lane; k < kend; k += 32)
                    a = fmaxf(a, fabsf(load_act(pr.x, pr.act_kind, static_cast<long long>(m) * pr.ldx + k)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                if (lane == 0) ctrl->amax_part[m] = a;
            }
        }
    }
    __syncwarp();
    if (raw && csize > 1) cluster_sync(); else __syncthreads();
    if (tid < 16) {
        const int m = tid;
        if (raw) {
            float a = ctrl->amax_part[m];
            for (int q = 0; q < csize; ++q)
                if (q != rank) a = fmaxf(a, ld_cluster_f32(mapa(smem_u32(&ctrl->amax_part[m]), q)));
            ctrl->qscale[m] = quant_scale(a);
            ctrl->a_scale[m] = dequant_scale(a);
        } else {
            ctrl->qscale[m] = 0.f;
            ctrl->a_scale[m] = (m < M) ? pr.a_scale[m] : 0.f;
        }
    }
    __syncthreads();

    if (warp < 4) {
        int rs = 0;
        const int slice_k = nkt * kTileK;
        if constexpr (PATH == kPathTC) {
            // B: [8-k group g][row group m/8][row m%8][8 fp16], core matrices of 8 x 16 B.
            const int units = (slice_k / 8) * 16;
            for (int u = tid; u < units; u += 128) {
                const int m = u & 15;
                const int g = u >> 4;
                const float s = ctrl->qscale[m];
                uint32_t packed[4];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    int qv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = kbase + g * 8 + i + e;
                        int v = 0;
                        if (m < M && k < kend) {
                            const long long idx = static_cast<long long>(m) * pr.ldx + k;
                            v = raw ? quantize(load_act(pr.x, pr.act_kind, idx), s)
                                    : static_cast<int>(static_cast<const int8_t*>(pr.x)[idx]);
                        }
                        qv[e] = v;
                        rs += v;
                    }
                    const int c = (g & 1) * 4 + (i >> 1);
                    const int sh = bscale_shift(c);
                    const __half h0 = __int2half_rn(qv[0] * (1 << sh));
                    const __half h1 = __int2half_rn(qv[1] * (1 << sh));
                    packed[i >> 1] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                                     (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
                }
                uint4* dst = reinterpret_cast<uint4*>(Bs + g * 256 + (m >> 3) * 128 + (m & 7) * 16);
                *dst = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
            fence_proxy_async_smem();
        } else {
            // B: [16-k chunk t][row m] 16 bytes = four int8x4 registers matching the
            // byte lanes of the masked code word: s -> {2s, 8+2s, 2s+1, 9+2s}.
            const int units = (slice_k / 16) * 16;
            for (int u = tid; u < units; u += 128) {
                const int m = u & 15;
                const int t = u >> 4;
                const float s = ctrl->qscale[m];
                int qv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k = kbase + t * 16 + i;
                    int v = 0;
                    if (m < M && k < kend) {
                        const long long idx = static_cast<long long>(m) * pr.ldx + k;
                        v = raw ? quantize(load_act(pr.x, pr.act_kind, idx), s)
                                : static_cast<int>(static_cast<const int8_t*>(pr.x)[idx]);
                    }
                    qv[i] = v;
                    rs += v;
                }
                uint32_t reg[4];
#pragma unroll
                for (int sidx = 0; sidx < 4; ++sidx) {
                    reg[sidx] = (static_cast<uint32_t>(qv[2 * sidx]) & 0xFFu) |
                                ((static_cast<uint32_t>(qv[8 + 2 * sidx]) & 0xFFu) << 8) |
                                ((static_cast<uint32_t>(qv[2 * sidx + 1]) & 0xFFu) << 16) |
                                ((static_cast<uint32_t>(qv[9 + 2 * sidx]) & 0xFFu) << 24);
                }
                *reinterpret_cast<uint4*>(Bs + (t * 16 + m) * 16) = make_uint4(reg[0], reg[1], reg[2], reg[3]);
            }
        }
        // every thread's units share one row m = tid % 16
        if (rs != 0) atomicAdd(&ctrl->rowsum_part[tid & 15], rs);
    }
    __syncthreads();

    // -------------------------------------------------------- main loop --
    int part_acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) part_acc[m] = 0;

    if constexpr (PATH == kPathTC) {
        if (warp < 4) {
            const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
            bool ok = true;
            for (int i = 0; i < nkt && ok; ++i) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctrl->full[i]), 0));
                if (!ok) { if (lane == 0) fail(ctrl, P.err, kErrWaitFull); break; }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int u = 2 * i + h;
                    const int b = u & 1;
                    if (u >= 2) {
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait_bounded(smem_u32(&ctrl->a_empty[b]), ((u >> 1) - 1) & 1));
                        if (!ok) { if (lane == 0) fail(ctrl, P.err, kErrWaitAEmpty); break; }
                        tc_fence_after();
                    }
                    const uint4 wv = *reinterpret_cast<const uint4*>(Ws + i * kTileBytes + h * 2048 + tid * 16);
                    uint32_t r[32];
                    unpack_word_f16(wv.x, r + 0);
                    unpack_word_f16(wv.y, r + 8);
                    unpack_word_f16(wv.z, r + 16);
                    unpack_word_f16(wv.w, r + 24);
                    tmem_st32(tmem + lane_base + kACol + b * 32, r);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctrl->a_full[b]));
                }
            }
        } else if (lane == 0 && nkt > 0) {
            const uint32_t bbase = smem_u32(Bs);
            const int nu = 2 * nkt;
            for (int u = 0; u < nu; ++u) {
                const int b = u & 1;
                if (!mbar_wait_bounded(smem_u32(&ctrl->a_full[b]), (u >> 1) & 1)) {
                    fail(ctrl, P.err, kErrWaitAFull);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int t = 4 * u + jj;  // 16-k chunk within the slice
                    const uint64_t bdesc = smem_desc_noswizzle(bbase + t * 512, 256, 128);
                    mma_f16_ts(tmem + kAccCol, tmem + kACol + b * 32 + jj * 8, bdesc, kIdesc,
                               (u | jj) != 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&ctrl->a_empty[b]));
            }
            mma_commit(smem_u32(&ctrl->done));
        }
        __syncwarp();
        if (warp < 4 && nkt > 0) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctrl->done), 0));
            if (ok) {
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kAccCol, v);
                tc_wait_ld();
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    part_acc[m] = __float2int_rn(__uint_as_float(v[m]) * 32768.f);
            } else if (lane == 0) {
                fail(ctrl, P.err, kErrWaitDone);
            }
        }
    } else {
        if (warp < 4) {
            int a0[DPR], a1[DPR], a2[DPR], a3[DPR];
#pragma unroll
            for (int m = 0; m < DPR; ++m) a0[m] = a1[m] = a2[m] = a3[m] = 0;
            for (int i = 0; i < nkt; ++i) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctrl->full[i]), 0))) {
                    if (lane == 0) fail(ctrl, P.err, kErrWaitFull);
                    break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(Ws + i * kTileBytes + h * 2048 + tid * 16);
                    const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int t = i * 8 + h * 4 + jj;
                        const uint32_t w = wd[jj];
                        const uint32_t m0 = w & 0x03030303u, m1 = w & 0x0C0C0C0Cu;
                        const uint32_t m2 = w & 0x30303030u, m3 = w & 0xC0C0C0C0u;
#pragma unroll
                        for (int m = 0; m < DPR; ++m) {
                            const int4 qv = *reinterpret_cast<const int4*>(Bs + (t * 16 + m) * 16);
                            a0[m] = dp4a_us(m0, qv.x, a0[m]);
                            a1[m] = dp4a_us(m1, qv.y, a1[m]);
                            a2[m] = dp4a_us(m2, qv.z, a2[m]);
                            a3[m] = dp4a_us(m3, qv.w, a3[m]);
                        }
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < DPR; ++m)
                part_acc[m] = a0[m] + (a1[m] >> 2) + (a2[m] >> 4) + (a3[m] >> 6);
        }
    }

    // ---------------------------------------------- split-K epilogue --
    if (warp < 4) {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            if (m < M) {
                const int v = part_acc[m] - ctrl->rowsum_part[m];
                if (csize == 1) {
                    const int n = rt * kTileN + tid;
                    if (n < pr.N) store_out(pr, m, n, v, ctrl->a_scale[m]);
                } else {
                    part[m * kTileN + tid] = v;
                }
            }
        }
    }
    __syncwarp();
    if (csize > 1) {
        cluster_sync();
        if (warp < 4) {
            const int rows_per = (kTileN + csize - 1) / csize;
            const int row0 = rank * rows_per;
            const int nrows = min(rows_per, kTileN - row0);
            if (nrows > 0) {
                for (int idx = tid; idx < M * nrows; idx += 128) {
                    const int m = idx / nrows;
                    const int rr = row0 + idx % nrows;
                    const uint32_t a = smem_u32(&part[m * kTileN + rr]);
                    int sum = 0;
                    for (int q = 0; q < csize; ++q) sum += ld_cluster_s32(mapa(a, q));
                    const int n = rt * kTileN + rr;
                    if (n < pr.N) store_out(pr, m, n, sum, ctrl->a_scale[m]);
                }
            }
        }
        cluster_sync();  // peers may still read this CTA's partials until here
    }

    // ------------------------------------------------------- tear-down --
    if (warp == 4 && lane == 0 && failed(ctrl)) {
        // never leave a bulk copy in flight into shared memory we are releasing
        for (int s = 0; s < nkt; ++s) (void)mbar_wait_bounded(smem_u32(&ctrl->full[s]), 0);
    }
    __syncwarp();
    if constexpr (PATH == kPathTC) {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
    }
}

template <int PATH, int DPR>
cudaError_t launch_one(const GemmParams& prm, int total_clusters, bool pdl, cudaStream_t stream) {
    auto kern = &w2a8_gemm_kernel<PATH, DPR>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gemm_smem_bytes(PATH, kMaxKtPerCta)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(total_clusters * prm.csize), 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_smem_bytes(PATH, prm.nkt_max);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(prm.csize);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
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

size_t gemm_smem_bytes(int path, int nkt_max) {
    size_t b = static_cast<size_t>(kCtrlBytes) + static_cast<size_t>(nkt_max) * 2 * kTileBytes + kPartBytes;
    if (path == kPathTC && b < static_cast<size_t>(kTcSmemFloor)) b = kTcSmemFloor;
    return b;
}

cudaError_t launch_gemm(const GemmParams& prm, int path, int dp_rows, int total_clusters,
                        bool pdl, cudaStream_t stream) {
    if (path == kPathTC) return launch_one<kPathTC, 1>(prm, total_clusters, pdl, stream);
    if (dp_rows <= 1) return launch_one<kPathDP, 1>(prm, total_clusters, pdl, stream);
    if (dp_rows <= 2) return launch_one<kPathDP, 2>(prm, total_clusters, pdl, stream);
    return launch_one<kPathDP, 4>(prm, total_clusters, pdl, stream);
}

}  // namespace bitmtp
