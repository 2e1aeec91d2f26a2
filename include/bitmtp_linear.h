/*
 * bitmtp_linear.h -- C ABI of the GB300 (sm_103a) W2A8 ternary linear.
 *
 * The operation is the "packed W2A8" linear of "BitMTP: When Multi-Token
 * Prediction Meets Low-Bit Large Language Models" (AI summary): ternary
 * BitNet b1.58-style weights ("What This Paper Is About"), 2-bit weights and
 * 8-bit activations ("Main Findings", first bullet), run through packed
 * low-bit operators that are picked by block width and by input/output
 * dimensions, including role-dependent output projections ("Methodology in
 * Plain English", third and last paragraphs).  The pages print no formula;
 * the library implements the BitNet b1.58 definitions:
 *
 *   weights      T[n][k] in {-1, 0, +1}, one fp32 per-tensor scale w_scale,
 *                W ~= w_scale * T (from fp32 W: w_scale = max(mean|W|, 1e-5),
 *                T = clamp(rint(W / w_scale), -1, 1); see
 *                bitmtp_linear_ternarize_pack);
 *   activations  per row m: amax = max_k |x[m][k]|, s = RN(127 / amax),
 *                q[m][k] = clamp(rint(RN(x * s)), -127, 127) (fp32, round
 *                half to even), a_scale[m] = RN(amax / 127); a zero row gives
 *                q = 0 and a_scale = 0;
 *   product      acc[m][n] = sum_k T[n][k] * q[m][k]   (exact int32);
 *   epilogue     y[m][n] = acc[m][n] * a_scale[m] * w_scale  (fp32, or that
 *                value rounded to bf16).
 *
 * Conventions for every call:
 *   - Matrices are row-major; ld* arguments count elements between rows.
 *   - Pointers are DEVICE pointers owned by the caller unless stated
 *     otherwise.  The library never allocates device memory; GEMM calls take
 *     a caller-owned workspace (see bitmtp_linear_workspace_bytes).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; only
 *     bitmtp_linear_pack, bitmtp_linear_ternarize_pack and
 *     bitmtp_linear_device_error synchronise it.
 *   - Arguments are validated on the host before any CUDA call; an invalid
 *     call returns a negative status and enqueues nothing.  Nothing is thrown
 *     across the ABI.
 *   - The current CUDA device must be compute capability 10.3 (sm_103a);
 *     otherwise calls return BITMTP_ERR_UNSUPPORTED.
 */
#ifndef BITMTP_LINEAR_H
#define BITMTP_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define BITMTP_OK               0
#define BITMTP_ERR_INVALID     (-1) /* NULL pointer, unknown enum, ld too small   */
#define BITMTP_ERR_ALIGN       (-2) /* packed weights or workspace not 16-byte aligned */
#define BITMTP_ERR_SHAPE       (-3) /* dimension out of the supported range, or a
                                       buffer smaller than its size query         */
#define BITMTP_ERR_NOT_TERNARY (-4) /* pack: an entry of T outside {-1, 0, +1}    */
#define BITMTP_ERR_UNSUPPORTED (-5) /* no device, or device is not sm_103        */
#define BITMTP_ERR_CUDA        (-6) /* a CUDA runtime call failed                 */
#define BITMTP_ERR_DEVICE      (-7) /* a kernel gave up a bounded wait (see
                                       bitmtp_linear_device_error)               */
#define BITMTP_ERR_NOT_FINITE  (-8) /* ternarize_pack: a weight is NaN or +-inf  */

/* ---- element kinds --------------------------------------------------------- */
#define BITMTP_F32  0   /* IEEE fp32                                   */
#define BITMTP_BF16 1   /* bfloat16 (raw 16-bit patterns)              */
#define BITMTP_Q8   2   /* int8 codes plus a per-row fp32 a_scale      */

/* ---- limits --------------------------------------------------------------- */
#define BITMTP_MAX_M      16       /* block width: rows per call (draft + verify rows) */
#define BITMTP_MAX_K      32768    /* in-features                                     */
#define BITMTP_MAX_N      16777216 /* out-features                                    */
#define BITMTP_MAX_GROUP  8        /* problems in one grouped launch                  */

/* ---- gemm flags ------------------------------------------------------------ */
/* Programmatic dependent launch: the GEMM may be scheduled while the kernel
 * launched before it on the same stream is still running, and it starts
 * streaming the packed weights before that kernel has finished.  It waits for
 * that kernel's completion before reading activations or writing outputs.
 * Only valid when the packed weights are not written by the preceding kernel. */
#define BITMTP_FLAG_PDL        0x1u
/* Force one of the two compute paths instead of the width/shape table
 * (testing and measurement): the tensor-core path (tcgen05, all widths) or the
 * integer dot-product path (dp4a, widths 1..4). */
#define BITMTP_FLAG_FORCE_TC   0x2u
#define BITMTP_FLAG_FORCE_DP   0x4u
/* (The default table: dp4a for widths 1..4, tensor cores with an 8-row
 * activation tile for 5..8 and a 16-row tile for 9..16.  Forcing the tensor
 * path at widths 1..4 uses its 8-row tile; forcing dp4a is valid for widths
 * 1..4.) */
/* "Fast" draft projection with FP8 activations.  The pages run cheaper "fast"
 * projections for drafting, more careful "critical" ones for generation and
 * verification, and on H20 FP8 draft projections ("BitMTP: When Multi-Token
 * Prediction Meets Low-Bit Large Language Models", "Methodology in Plain
 * English", M1); they give no formula.  With this flag every problem of the
 * call keeps its ternary weights and quantises its activation rows per row to
 * FP8 E4M3 instead of int8:
 *   s = RN32(448 / amax);  e = E4M3(RN32(x * s));  a_scale = RN32(amax / 448)
 * (E4M3: 3 mantissa bits, exponent bias 7, no infinities, largest finite 448;
 * round to nearest even, saturating), then y = acc * a_scale * w_scale with
 * acc = sum_k T * e accumulated in fp32 on the tensor cores, as
 * sum_k (T + 1) * e - sum_k e.  That accumulation rounds only where a partial
 * sum needs more than 24 significant bits: acc differs from the exact sum by
 * at most (2 * ceil(K/32) + 2) * 2^-23 * sum_k (T + 2) * |e|, and is exact
 * when every partial sum fits in 24 bits (for example all |e| in one binade
 * and |acc| below 2^24 of its steps).  The order of the partial sums may vary
 * from run to run, so rounded results may differ in their last bits.  Every
 * width 1..16 runs on the tensor cores with a 16-row tile.  act.kind must be
 * BITMTP_F32 or BITMTP_BF16 (act.amax may be given, as above); out.acc, if
 * given, receives the fp32 accumulators' bit patterns instead of int32
 * values.  Not combinable with BITMTP_FLAG_FORCE_DP. */
#define BITMTP_FLAG_FP8        0x8u
/* Test only, never for production calls: CTA 0 of the launch never requests
 * its first chunk of packed weights and every wait of the launch gives up
 * after 1 ms instead of 2 s, so the launch exercises its bounded-wait error
 * path: it ends without hanging, sets the device error word (see
 * bitmtp_linear_device_error) and leaves its outputs unspecified.  Zero-fill
 * the workspace before the next call (the no-alloc entry point does this
 * itself once bitmtp_linear_device_error has reported the error). */
#define BITMTP_FLAG_TEST_WITHHOLD 0x100u

/*
 * Packed ternary weights (this library's own layout; the pages only say the
 * weights are executed "packed"): rows in tiles of 128, k in tiles of 128,
 * both padded with T = 0.  Tile (rt, kt) is 4096 contiguous bytes at offset
 * (rt * ceil(K/128) + kt) * 4096.  Inside a tile row r owns eight 32-bit
 * words; word j of row r sits at word index (j/4)*512 + r*4 + j%4 and holds
 * k = kt*128 + 16*j + 2*p + e (p = 0..7, e = 0..1) as u = T + 1 in bits
 * 16*e + 2*p.  A 16-byte trailer {0x38413242, N, K, invalid-count} follows.
 * 2 bits per weight; the trailer is 16 bytes.
 */

/* Bytes needed for the packed form of an N x K ternary matrix:
 * ceil(N/128) * ceil(K/128) * 4096 + 16.  Returns 0 if N < 1 or K < 1. */
size_t bitmtp_linear_packed_bytes(int64_t N, int64_t K);

/* Pack ternary weights (offline step before the linear).
 *   T        device int8 [N][ldt], entries in {-1, 0, +1}
 *   N, K     out- and in-features (1 <= N <= BITMTP_MAX_N, 1 <= K <= BITMTP_MAX_K)
 *   ldt      >= K
 *   pk       device buffer of pk_bytes >= bitmtp_linear_packed_bytes(N, K),
 *            16-byte aligned; fully overwritten (tiles and trailer)
 * Synchronises `stream` to read the invalid-entry count; returns
 * BITMTP_ERR_NOT_TERNARY (pk then holds a clamped, unusable packing) if any
 * entry was outside {-1, 0, +1}. */
int bitmtp_linear_pack(const int8_t* T, int64_t N, int64_t K, int64_t ldt,
                       void* pk, size_t pk_bytes, void* stream);

/* Absmean ternarisation and pack of fp32 weights, on the device (the offline
 * step before bitmtp_linear_pack's input exists).  The pages describe the
 * backbone as BitNet b1.58-style ternary ("BitMTP: When Multi-Token Prediction
 * Meets Low-Bit Large Language Models", "What This Paper Is About" and
 * "Overview") but print no formula; this follows the BitNet b1.58 weight
 * quantiser:
 *   gamma = max(mean|W|, 1e-5),  T = clamp(round_half_even(W / gamma), -1, 1)
 * where mean|W| is the exact sum of |W| rounded once to fp64, divided by N*K
 * in fp64 and rounded to fp32 (so no summation order enters), and W / gamma is
 * one IEEE fp32 division.
 *   W          device fp32 [N][ldw], ldw >= K, finite values
 *   pk         as for bitmtp_linear_pack; receives the packing of T
 *   w_scale    device float, receives gamma (the per-tensor weight scale)
 *   workspace  device scratch of ws_bytes >= bitmtp_linear_ternarize_workspace_bytes(N, K),
 *              16-byte aligned, caller-owned; need not be zeroed, left dirty
 * Stream-ordered; synchronises `stream` at the end to read the non-finite
 * flag and returns BITMTP_ERR_NOT_FINITE (pk and *w_scale then unspecified)
 * if W holds a NaN or an infinity. */
size_t bitmtp_linear_ternarize_workspace_bytes(int64_t N, int64_t K);
int bitmtp_linear_ternarize_pack(const float* W, int64_t N, int64_t K, int64_t ldw,
                                 void* pk, size_t pk_bytes, float* w_scale,
                                 void* workspace, size_t ws_bytes, void* stream);

/* One matrix of a grouped ternarisation (same meaning as the arguments of
 * bitmtp_linear_ternarize_pack). */
typedef struct bitmtp_ternarize_desc {
    const float* W;        /* device fp32 [N][ldw], ldw >= K                        */
    int64_t N, K, ldw;
    void* pk;              /* device, pk_bytes >= bitmtp_linear_packed_bytes(N, K),
                              16-byte aligned                                       */
    size_t pk_bytes;
    float* w_scale;        /* device float: receives gamma                          */
} bitmtp_ternarize_desc;

/* Workspace bytes for a grouped ternarisation of n_desc matrices (0 if
 * n_desc is outside 1..BITMTP_MAX_GROUP). */
size_t bitmtp_linear_ternarize_workspace_bytes_grouped(int n_desc);

/* bitmtp_linear_ternarize_pack for up to BITMTP_MAX_GROUP matrices at once
 * (e.g. the projections of a layer): four launches for the whole group (a
 * memset, the absmean pass over every matrix, one scale per matrix, the pack
 * of every tile) and one stream sync at the end.  Results are identical to
 * calling bitmtp_linear_ternarize_pack on each matrix.  `d` is a HOST array
 * (copied by value into the launches); the packed buffers must not overlap.
 *   workspace  device scratch of ws_bytes >= the query above, 16-byte
 *              aligned, need not be zeroed, left dirty
 * Returns BITMTP_ERR_NOT_FINITE if any matrix holds a NaN or an infinity (pk
 * and *w_scale of that matrix are then unspecified; the others are valid). */
int bitmtp_linear_ternarize_pack_grouped(const bitmtp_ternarize_desc* d, int n_desc,
                                         void* workspace, size_t ws_bytes, void* stream);

/* Quantise a block of activation rows to int8 codes with per-row scales
 * (the quantiser defined at the top of this file).
 *   x        device [M][ldx], element kind x_kind = BITMTP_F32 or BITMTP_BF16,
 *            finite values
 *   M, K     rows (0 <= M <= 2^20) and in-features (1 <= K <= BITMTP_MAX_K)
 *   q        device int8 [M][ldq], ldq >= K
 *   a_scale  device fp32 [M]   = amax/127 (0 for an all-zero row)
 *   rowsum   device int32 [M]  = sum_k q[m][k]; may be NULL
 * M == 0 is a no-op. */
int bitmtp_linear_quant_act(const void* x, int x_kind, int64_t M, int64_t K, int64_t ldx,
                            int8_t* q, int64_t ldq, float* a_scale, int32_t* rowsum,
                            void* stream);

/* Activation operand of a GEMM. */
typedef struct bitmtp_act {
    int kind;              /* BITMTP_F32 / BITMTP_BF16: raw rows, quantised inside the
                              GEMM with the quantiser above (bit-identical to
                              bitmtp_linear_quant_act);  BITMTP_Q8: int8 codes        */
    const void* x;         /* [M][ldx] elements of `kind` (int8 for BITMTP_Q8)        */
    int64_t ldx;           /* >= K                                                   */
    const float* a_scale;  /* BITMTP_Q8 only: [M] per-row scales; ignored otherwise   */
    const float* amax;     /* optional, BITMTP_F32/BF16 only (NULL otherwise): device
                              [M] = max_k |x[m][k]| of exactly these rows, e.g. the
                              amax output of the GEMM that wrote x (a layer chain);
                              the call then skips its own absmax pass, and when
                              every problem of a call at block width 1..4 brings
                              it (the dp4a path, not BITMTP_FLAG_FP8) the call is
                              one launch: the GEMM quantises the rows itself, with
                              the same steps and codes, and no preparation kernel
                              runs.  Any other value gives wrong codes.            */
} bitmtp_act;

/* Output of a GEMM. */
typedef struct bitmtp_out {
    int dtype;             /* BITMTP_F32 or BITMTP_BF16 (round-to-nearest-even)     */
    void* y;               /* [M][ldy]                                              */
    int64_t ldy;           /* >= N                                                  */
    int32_t* acc;          /* optional int32 [M][lda] accumulators, may be NULL     */
    int64_t lda;           /* >= N when acc != NULL                                  */
    float* amax;           /* optional device [M]: receives max_n |y[m][n]| of the
                              values stored (after the bf16 rounding for BITMTP_BF16),
                              ready to be the next call's act.amax; the call zeroes
                              it before its epilogues combine per-CTA maxima with
                              atomics (the first phase of a two-phase row absmax,
                              the next call's quantisation the second).  Must not
                              overlap y, acc or this call's act.amax.              */
} bitmtp_out;

/* Workspace of a GEMM call: a device buffer the caller allocates once,
 * 16-byte aligned, of at least the size these queries return, and
 * zero-fills before its first use (e.g. cudaMemset).  It holds a fixed part
 * of about 2.5 MiB -- one slot of partial sums per CTA for row tiles split
 * between CTAs, a ready flag per slot and two synchronisation words of the
 * one-launch layer-chain calls -- and each problem's quantised
 * activation operand (about 4.5 KiB per 128 in-features).  Every call leaves
 * the flags at zero, so one workspace serves calls of any shapes that fit.
 * Calls that may execute concurrently on the GPU need distinct workspaces;
 * calls ordered on one stream may share one.  After a call that ends in
 * BITMTP_ERR_DEVICE, zero-fill it again.  Returns 0 for out-of-range
 * arguments. */
size_t bitmtp_linear_workspace_bytes(int64_t N, int64_t K, int64_t M);

/* y = dequant(T * q): the W2A8 linear at block width M.
 *   pk        packed weights from bitmtp_linear_pack (16-byte aligned)
 *   w_scale   per-tensor weight scale
 *   N, K      out-/in-features the weights were packed with
 *   M         block width, 0 <= M <= BITMTP_MAX_M (0: no-op)
 *   workspace >= bitmtp_linear_workspace_bytes(N, K, M) bytes, see above
 *   flags     BITMTP_FLAG_* bits
 * Two kernel launches: the first quantises the activation rows
 * (BITMTP_F32/BF16, with the quantiser above; BITMTP_Q8 rows are taken as
 * they are) into the workspace, the second streams the packed weights and
 * writes y (and acc); it starts streaming while the first one runs.  One
 * launch for a layer-chain call at block width 1..4 (see act.amax): the GEMM
 * quantises the rows while its first weights stream in.
 * The compute path is chosen from M (width specialisation); results do not
 * depend on the choice. */
int bitmtp_linear_gemm(const void* pk, float w_scale, int64_t N, int64_t K, int64_t M,
                       const bitmtp_act* act, const bitmtp_out* out,
                       void* workspace, size_t workspace_bytes,
                       unsigned flags, void* stream);

/* One problem of a grouped launch (same meaning as bitmtp_linear_gemm). */
typedef struct bitmtp_gemm_desc {
    const void* pk;
    float w_scale;
    int64_t N, K, M;
    bitmtp_act act;
    bitmtp_out out;
} bitmtp_gemm_desc;

/* Workspace bytes for a grouped launch of these descriptors (0 if invalid). */
size_t bitmtp_linear_workspace_bytes_grouped(const bitmtp_gemm_desc* d, int n_desc);

/* Run up to BITMTP_MAX_GROUP independent problems in one GEMM launch (after
 * one activation-preparation launch covering all of them) --
 * e.g. the role-dependent output projections of one block step (verify rows
 * through one projection and draft rows through another), or the independent
 * projections of a layer.  `d` is a HOST array of n_desc descriptors (copied
 * by value into the launch).  The compute path follows the widest problem.
 * Problems must not write overlapping outputs. */
int bitmtp_linear_gemm_grouped(const bitmtp_gemm_desc* d, int n_desc,
                               void* workspace, size_t workspace_bytes,
                               unsigned flags, void* stream);

/* Size of the library's built-in scratch array used by
 * bitmtp_linear_gemm_noalloc: 4 MiB of device memory, held on every device
 * that loads the library until the process exits. */
#define BITMTP_NOALLOC_SCRATCH_BYTES ((size_t)4 * 1024 * 1024)

/* bitmtp_linear_gemm without a workspace argument: for callers that cannot
 * allocate device memory.  Examples: code called from another runtime's
 * launch hook or plugin that forbids allocation; latency-bound loops where
 * cudaMalloc/cudaFree would stall the device or the host thread; processes
 * whose device memory is entirely owned by a caching allocator they cannot
 * reach.  (The paper has no counterpart: this is a deployment convenience.)
 *
 * Arguments, results and the launched kernel are those of bitmtp_linear_gemm;
 * instead of a caller workspace the call uses one static device array of
 * BITMTP_NOALLOC_SCRATCH_BYTES that the library owns.  It allocates nothing.
 *   - Limit: a shape whose workspace need (bitmtp_linear_workspace_bytes)
 *     exceeds BITMTP_NOALLOC_SCRATCH_BYTES is rejected with BITMTP_ERR_SHAPE
 *     before anything is enqueued.  Every shape inside the library's limits
 *     (M <= BITMTP_MAX_M, K <= BITMTP_MAX_K, N <= BITMTP_MAX_N) fits.
 *   - Set-up: the first call on a device, made with that device current,
 *     looks up the array's device address (one CUDA runtime query, which may
 *     load the library's device code).  Make that first call before any
 *     stream capture begins.
 *   - Sharing: all calls on a device share the one array and it keeps what
 *     the previous call left.  The part that must start at zero (sync
 *     words and ready flags, 40.25 KiB) starts zeroed and every call leaves it at zero; only a
 *     call that gave up a bounded wait can leave it dirty, and once
 *     bitmtp_linear_device_error has reported that, the next call clears it
 *     first (one memset on `stream`).  Calls whose work can overlap on the GPU
 *     (different streams without ordering between them, or different host
 *     threads) race on the array and give wrong results; order them on one
 *     stream or use bitmtp_linear_gemm with distinct workspaces.
 * Enqueues the kernels of bitmtp_linear_gemm on `stream` (preceded by that
 * memset only after a reported error). */
int bitmtp_linear_gemm_noalloc(const void* pk, float w_scale, int64_t N, int64_t K, int64_t M,
                               const bitmtp_act* act, const bitmtp_out* out,
                               unsigned flags, void* stream);

/* Synchronise `stream`, then return and clear the device error word that a
 * kernel sets when one of its bounded waits expires (0 = none; otherwise a
 * code naming the wait).  Never set by correct launches. */
int bitmtp_linear_device_error(void* stream);

/* Human-readable name of a status code (static storage). */
const char* bitmtp_linear_status_string(int status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int bitmtp_linear_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BITMTP_LINEAR_H */
