/*
 * w8a16.h -- C ABI of the GB300 (sm_103a) W8A16 block-scaled GEMM library
 * (libw8a16.so).
 *
 * The operation (page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs",
 * module doc and the doc comments of `w8a16_gemm_pipelined_m32_strided`,
 * `W8A16_M32_K_BLOCK` and `w8a16_gemm_pipelined_by_m`):
 *
 *     C[m][n] = bf16( sum_k  A[m][k] * e4m3(W[n][k]) * block_scale[n/128][k/128] )
 *
 * for m < M, n < N, k < K, with
 *   A            BF16, M rows of a_row_stride elements; the first K of each row are read;
 *   W            FP8 E4M3 ("FN": bias 7, no infinities, 0x7F/0xFF NaN), N rows of K
 *                bytes, row-major;
 *   block_scale  FP32, ceil(N/128) rows of K/128 values: one scale per 128x128 block of W;
 *   C            BF16, M rows of c_row_stride elements; the first N of each row are
 *                written and nothing else is.
 * Strides count elements, not bytes. Accumulation is FP32 on the tensor cores; the
 * block scale is folded into the FP32 accumulator once per 128-K step and the
 * result is rounded to BF16 (round-to-nearest-even). Each call is deterministic:
 * the same arguments on the same plan give bit-identical outputs.
 *
 * Ownership and asynchrony. The caller owns every buffer and the stream; the
 * library allocates nothing and keeps no per-call state besides a host-side
 * cache of TMA descriptors. Device calls are asynchronous on `stream` (NULL is
 * the legacy default stream), as the page's launchers are (`.launch(stream)`):
 * the output is ready once the stream has reached the call. All checks run on
 * the host before any device work; a failed check returns a negative W8A16_ERR_*
 * code, touches no device memory, and leaves a message for w8a16_last_error().
 *
 * Device-side failure. Every wait inside the kernels is bounded (default 2 s,
 * environment variable W8A16_WAIT_TIMEOUT_MS, read once). A wait that runs out
 * makes the kernel record W8A16_STATUS_WAIT_TIMEOUT, release what it holds and
 * return; w8a16_device_status() reports it. The CUDA context stays usable.
 */
#ifndef W8A16_H
#define W8A16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define W8A16_API __attribute__((visibility("default")))
#else
#define W8A16_API
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *w8a16_stream_t;

/* Return codes. The first four are the page's checks (doc comment and `ensure!`
 * clauses of `w8a16_gemm_pipelined_m32_strided`); the rest are this library's. */
enum {
    W8A16_OK = 0,
    W8A16_ERR_M_ZERO = -1,         /* M == 0: no rows to compute */
    W8A16_ERR_K_BLOCK = -2,        /* K is not a positive multiple of 128 */
    W8A16_ERR_PITCH = -3,          /* a_row_stride < K or c_row_stride < N */
    W8A16_ERR_A_PITCH_ALIGN = -4,  /* a_row_stride % 8 != 0 (A rows must stay 16-byte aligned) */
    W8A16_ERR_N_ZERO = -5,         /* N == 0 */
    W8A16_ERR_NULL = -6,           /* a required pointer is NULL */
    W8A16_ERR_ALIGN = -7,          /* A or W not 16-byte aligned, block_scale not 4-byte,
                                      C not 2-byte aligned */
    W8A16_ERR_RANGE = -8,          /* a size past what the kernels address (see w8a16_gemm) */
    W8A16_ERR_DEVICE = -9,         /* no CUDA device, or the current device is not sm_103 */
    W8A16_ERR_LAUNCH = -10,        /* the CUDA launch failed (message has the CUDA error) */
    W8A16_ERR_PLAN = -11,          /* a requested plan is invalid for this shape */
    W8A16_ERR_COPY = -12,          /* a host<->device copy could not be queued */
    W8A16_ERR_ARG = -13            /* another invalid argument (message says which) */
};

/* Device status words (w8a16_device_status). */
enum {
    W8A16_STATUS_OK = 0,
    W8A16_STATUS_WAIT_TIMEOUT = 1  /* a bounded in-kernel wait ran out; output undefined */
};

/* Call flags (w8a16_gemm_ex). */
enum {
    /* Programmatic dependent launch: the kernel may start while the work queued
     * before it on the stream is still running, and reads its first weight tiles
     * and its block scales before waiting for that work to finish; A and C are
     * only touched after the wait. Consecutive calls then overlap one call's
     * start-up with the previous call's tail. Contract: no work queued earlier on
     * the stream may write W or block_scale (the quantised weights are read-only
     * in inference). */
    W8A16_FLAG_PDL = 1u
};

/* Kernel variants. */
enum {
    W8A16_VARIANT_AUTO = 0,  /* the planner's choice (w8a16_plan) */
    W8A16_VARIANT_SIMT = 1,  /* CUDA-core kernel: one warp per weight row, no tensor cores */
    W8A16_VARIANT_TC = 2,    /* TMA weight ring + in-register E4M3->BF16 + tcgen05 MMA
                                (weight rows = MMA M, tokens = MMA N), cluster split-K */
    W8A16_VARIANT_TC8 = 3    /* FP8 tensor datapath: the E4M3 weight tiles feed tcgen05
                                kind::f8f6f4 MMAs as loaded; each BF16 activation enters
                                as two E4M3 terms (exact for |a| >= 2^-14 of its token's
                                128-K block maximum, within 2^-22 of it otherwise); a
                                non-finite activation makes its token's outputs NaN */,
    W8A16_VARIANT_W8A8 = 4,  /* the W8A8 kernel (w8a16_gemm_w8a8 only): FP8 activations with
                                per-token 128-K group scales, one kind::f8f6f4 MMA per 32 K */
    W8A16_VARIANT_PRESPLIT = 5, /* w8a16_gemm_ws only: the activations are split into the
                                two E4M3 terms of W8A16_VARIANT_TC8 once per call, by a
                                pre-pass into the caller's workspace, and the W8A8 kernel
                                multiplies both terms in one MMA of N = 2 x token tile;
                                same accuracy as W8A16_VARIANT_TC8 */
    W8A16_VARIANT_STREAM = 7,  /* w8a16_gemm_ws with a forced plan only, 3 <= M <= 32: the
                                pre-split path on a persistent grid (two CTAs per SM) that
                                splits all (128-row weight tile, 128-K step) units into
                                equal contiguous ranges, a tile split between CTAs being
                                summed through the workspace in K order by the last of
                                them; needs w8a16_workspace_bytes_for(M, N, K) bytes; same
                                accuracy as W8A16_VARIANT_PRESPLIT. Never the planner's
                                choice (slower than the other plans on GB300) */
    W8A16_VARIANT_GEMV = 6     /* decode kernel for M <= 2: the arithmetic of
                                W8A16_VARIANT_TC8; a cluster of split_k CTAs per 128-row
                                weight tile, each on at most 8 K steps, every one of them
                                loaded before the grid-dependency wait (shared memory and
                                TMEM), at most one CTA per SM; the planner's choice for
                                M <= 2 when ceil(N/128) x ceil(K/1024) CTAs fit that rule,
                                for w8a16_gemm and w8a16_gemm_w8a8 alike */
};

/*
 * w8a16_gemm -- the operation above on the current CUDA device.
 *
 * A            device pointer, 16-byte aligned, BF16 [M][a_row_stride]
 * a_row_stride elements between A rows; >= K and a multiple of 8
 * W            device pointer, 16-byte aligned, E4M3 bytes [N][K]
 * block_scale  device pointer, 4-byte aligned, FP32 [ceil(N/128)][K/128]
 * C            device pointer, 2-byte aligned, BF16 [M][c_row_stride]; only columns < N
 *              of the M rows are written
 * c_row_stride elements between C rows; >= N, no alignment rule
 * M, N, K      M >= 1, N >= 1, K a positive multiple of 128. Limits (W8A16_ERR_RANGE):
 *              N, K, M < 2^31; a_row_stride * 2 and K are TMA strides below 2^40 bytes.
 * stream       CUDA stream for the work
 *
 * Returns W8A16_OK once the work is queued, or a W8A16_ERR_* code (nothing queued).
 * The work is one kernel launch, or two when the plan has a split-K tail
 * (w8a16_plan_t.tail_tiles; the second is a programmatic dependent of the first).
 * C may alias neither A, W nor block_scale.
 */
W8A16_API int w8a16_gemm(const void *A, uint32_t a_row_stride, const void *W, const float *block_scale,
               void *C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
               w8a16_stream_t stream);

/* Contiguous form: a_row_stride = K, c_row_stride = N (the page's
 * `w8a16_gemm_pipelined_m32`, which calls the strided launcher with pitches (k, n)). */
W8A16_API int w8a16_gemm_contiguous(const void *A, const void *W, const float *block_scale, void *C,
                          uint32_t M, uint32_t N, uint32_t K, w8a16_stream_t stream);

/* w8a16_gemm with call flags (W8A16_FLAG_*; 0 = the same as w8a16_gemm). */
W8A16_API int w8a16_gemm_ex(const void *A, uint32_t a_row_stride, const void *W,
                            const float *block_scale, void *C, uint32_t c_row_stride, uint32_t M,
                            uint32_t N, uint32_t K, uint32_t flags, w8a16_stream_t stream);

/*
 * w8a16_gemm_host -- the same operation on HOST buffers: queues on `stream` the
 * host-to-device copies of A (M rows, full pitch), W and block_scale into the
 * caller's device buffers dA, dW, dScale, the GEMM into dC, and the copy of dC
 * (M rows, full pitch) back to C_host. Pinned host memory makes the copies
 * asynchronous; pageable memory works but the copies then synchronise with the
 * host. Pass copy_weights = 0 to skip the W and block_scale uploads when dW/dScale
 * already hold them. Buffer rules and return codes are those of w8a16_gemm, plus
 * W8A16_ERR_COPY when a copy cannot be queued. The output is in C_host once the
 * stream has reached the call.
 */
W8A16_API int w8a16_gemm_host(const void *A_host, uint32_t a_row_stride, const void *W_host,
                    const float *scale_host, void *C_host, uint32_t c_row_stride, uint32_t M,
                    uint32_t N, uint32_t K, void *dA, void *dW, float *dScale, void *dC,
                    int copy_weights, w8a16_stream_t stream);

/* ---- planning (pure host code; no device work) -------------------------- */

typedef struct {
    int32_t variant;       /* one of W8A16_VARIANT_SIMT, _TC, _TC8, _W8A8, _PRESPLIT */
    uint32_t token_tile;   /* tokens (rows of A/C) per CTA: the MMA N of the tensor-core
                              variants */
    uint32_t split_k;      /* CTAs (one cluster) sharing a 128-row weight tile, each on a
                              contiguous range of 128-K steps; 1 = no split */
    uint32_t stages;       /* depth of the shared-memory weight ring (tensor-core variants) */
    uint32_t ctas_per_sm;  /* residency the plan assumes */
    uint32_t grid[3];
    uint32_t block[3];
    uint32_t cluster[3];
    uint32_t smem_bytes;   /* dynamic shared memory per CTA */
    uint32_t tmem_cols;    /* tensor-memory columns per CTA (tensor-core variants) */
    uint32_t tail_tiles;   /* TC, W8A8 and PRESPLIT plans with split_k 1 and one token
                              tile: the last tail_tiles 128-row weight tiles run in a
                              second launch, split over clusters of tail_split CTAs, so
                              that a partial second wave of whole tiles becomes a short
                              wave of split ones (grid[0] then counts the first launch's
                              CTAs); 0 = none */
    uint32_t tail_split;   /* split-K of that second launch (>= 2 when tail_tiles > 0) */
} w8a16_plan_t;

/* The page's checks plus this library's (pointers may be NULL here: only sizes,
 * pitches and the alignment of non-NULL pointers are checked). */
W8A16_API int w8a16_check_args(const void *A, uint32_t a_row_stride, const void *W,
                     const float *block_scale, const void *C, uint32_t c_row_stride, uint32_t M,
                     uint32_t N, uint32_t K);

/* The plan for (M, N, K) on a GPU with `sm_count` SMs (pure: no device work).
 * cluster_ctas, if not NULL, has 17 entries: cluster_ctas[s] = how many CTAs of
 * the plan's kernel can be co-resident when launched in clusters of s CTAs
 * (s = 1..16; 0 = that cluster size cannot run), as w8a16_cluster_capacity
 * reports; NULL assumes every size fills every SM slot. */
W8A16_API int w8a16_plan_for(uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count,
                             const uint32_t *cluster_ctas, w8a16_plan_t *out);

/* The plan w8a16_gemm uses for (M, N, K) on the current device. */
W8A16_API int w8a16_plan_current(uint32_t M, uint32_t N, uint32_t K, w8a16_plan_t *out);

/* Co-resident CTAs of a tensor-core variant's kernel for a token tile and stage
 * count on the current device, per cluster size: out[s] for s = 1..16 (out[0] = 0). */
W8A16_API int w8a16_cluster_capacity(int32_t variant, uint32_t token_tile, uint32_t stages,
                                     uint32_t out[17]);

/* Build the plan for an explicit variant / split / stage count (0 = planner's
 * choice for that field). Returns W8A16_ERR_PLAN if it cannot run this shape. */
W8A16_API int w8a16_plan_variant(uint32_t M, uint32_t N, uint32_t K, int32_t variant, uint32_t split_k,
                       uint32_t stages, uint32_t sm_count, w8a16_plan_t *out);

/* w8a16_gemm_ex with a plan from w8a16_plan_variant (for tests and tuning sweeps). */
W8A16_API int w8a16_gemm_with_plan(const void *A, uint32_t a_row_stride, const void *W,
                                   const float *block_scale, void *C, uint32_t c_row_stride,
                                   uint32_t M, uint32_t N, uint32_t K, const w8a16_plan_t *plan,
                                   uint32_t flags, w8a16_stream_t stream);

/* ---- the W8A16 product with a caller-provided workspace ------------------ */

/* Bytes of workspace w8a16_gemm_ws uses for the pre-split path at (M, K): the two
 * E4M3 terms of A ([2M][K] bytes) and one FP32 factor per token and 128-K group
 * ([K/128][M rounded up to 4]). 0 for M = 0 or K not a positive multiple of 128. */
W8A16_API uint64_t w8a16_workspace_bytes(uint32_t M, uint32_t K);

/* Bytes of workspace that every w8a16_gemm_ws plan for (M, N, K) on the current
 * device fits in: w8a16_workspace_bytes(M, K) for M > 16 (the pre-split terms), and
 * where the stream-K plan applies (3 <= M <= 32) its layout: the terms, one counter
 * per 128-row weight tile (256-byte aligned after them) and the FP32 partials of the
 * tiles split between CTAs (256-byte aligned after the counters). 0 where no plan
 * uses a workspace or the sizes are invalid. */
W8A16_API uint64_t w8a16_workspace_bytes_for(uint32_t M, uint32_t N, uint32_t K);

/* The plan w8a16_gemm_ws takes with plan == NULL and `workspace_bytes` bytes of
 * workspace for (M, N, K) on the current device. Checks as w8a16_plan_current. */
W8A16_API int w8a16_plan_ws(uint32_t M, uint32_t N, uint32_t K, uint64_t workspace_bytes,
                            w8a16_plan_t *out);

/* w8a16_gemm with a workspace: the same operation, arguments, checks and result
 * contract (within the tolerance of W8A16_VARIANT_TC8, whose split this path
 * shares). With plan == NULL the library chooses (w8a16_plan_ws reports it): for
 * M > 16 with at least w8a16_workspace_bytes(M, K) bytes, W8A16_VARIANT_PRESPLIT;
 * else exactly what w8a16_gemm runs. On the pre-split plans (PRESPLIT, or a forced
 * STREAM plan) a split kernel writes the workspace (and clears the stream-K tile
 * counters), then the FP8 x FP8 kernel reads it (one launch, or two when the plan
 * has a split-K tail; all on `stream`, each queued as a programmatic dependent
 * launch of the one before;
 * W8A16_FLAG_PDL governs only the split kernel's overlap with the previous kernel,
 * as for w8a16_gemm). A plan from w8a16_plan_variant forces a variant (PRESPLIT
 * and STREAM need their workspace, else W8A16_ERR_ARG).
 *   workspace  device memory, 16-byte aligned, owned by the caller, or NULL; it is
 *              written by the call and must not be used by other work until the
 *              call's kernels have finished (calls that share one workspace must
 *              be ordered on one stream).
 * Returns W8A16_OK once the work is queued, or a W8A16_ERR_* code (nothing queued). */
W8A16_API int w8a16_gemm_ws(const void *A, uint32_t a_row_stride, const void *W,
                            const float *block_scale, void *C, uint32_t c_row_stride,
                            uint32_t M, uint32_t N, uint32_t K, const w8a16_plan_t *plan,
                            void *workspace, uint64_t workspace_bytes, uint32_t flags,
                            w8a16_stream_t stream);

/* The product without a caller's workspace and without any allocation (the paper
 * has no counterpart): w8a16_gemm_ws on a fixed 32 MiB device buffer that is part of
 * the library's module (w8a16_noalloc_scratch_bytes() bytes), whose address is
 * looked up on the current device at each call (so a device reset does not leave
 * a stale address behind). Same arguments, checks and results as w8a16_gemm_ws
 * with plan = NULL; M <= 16 uses no scratch. W8A16_ERR_RANGE when M > 16 and
 * w8a16_workspace_bytes(M, K) exceeds the buffer. Every value the kernels read
 * from the buffer is written earlier in the same call, so nothing needs clearing.
 * The buffer is shared: calls whose kernels may overlap in time (on other streams,
 * or from other host threads without ordering) race on it and must not be issued;
 * calls ordered on one stream are safe. */
W8A16_API int w8a16_gemm_noalloc(const void *A, uint32_t a_row_stride, const void *W,
                                 const float *block_scale, void *C, uint32_t c_row_stride,
                                 uint32_t M, uint32_t N, uint32_t K, uint32_t flags,
                                 w8a16_stream_t stream);
W8A16_API uint64_t w8a16_noalloc_scratch_bytes(void);

/* The two halves of the pre-split path (W8A16_VARIANT_PRESPLIT) as separate calls,
 * so that products which share one activation matrix (the Q, K and V projections
 * of one input, say) split it once. Same operation and result contract as
 * w8a16_gemm_ws on its pre-split path (the reading of W8A16_VARIANT_TC8: each
 * activation of a token's 128-K block is written as two E4M3 terms).
 *
 * w8a16_split_activations -- BF16 A [M][a_row_stride] (first K of a row read;
 * a_row_stride >= K, a multiple of 8) -> the workspace: hi codes [M][K], lo codes
 * [M][K] (E4M3 bytes, rows of K) and one FP32 factor 2^(E-7) per token and 128-K
 * group ([K/128][M rounded up to 4]). workspace: device memory, 16-byte aligned,
 * at least w8a16_workspace_bytes(M, K) bytes, owned by the caller. A and the
 * workspace 16-byte aligned. One kernel, queued as a programmatic dependent launch
 * that waits for the previous kernel of the stream before touching memory. Checks
 * (before any device work): those of w8a16_gemm on M, K and a_row_stride, NULL,
 * alignment, and the workspace size (W8A16_ERR_ARG). */
W8A16_API int w8a16_split_activations(const void *A, uint32_t a_row_stride, uint32_t M, uint32_t K,
                                      void *workspace, uint64_t workspace_bytes,
                                      w8a16_stream_t stream);

/* w8a16_gemm_split_terms -- C = the W8A16 product of the activations that
 * w8a16_split_activations wrote into `workspace` for the same (M, K), with W,
 * block_scale, C, c_row_stride, N as in w8a16_gemm. The FP8 x FP8 kernel on the
 * planner's W8A16_VARIANT_PRESPLIT plan (one launch, or two with a split-K tail).
 * flags: W8A16_FLAG_PDL lets the kernel read its first weight tiles and block
 * scales before the previous kernel of the stream has finished (which must not
 * write W or block_scale); the workspace, A's terms, is read only after it. The
 * workspace is only read. Checks as for w8a16_gemm (the workspace takes A's place
 * in the NULL and alignment checks), plus its size (W8A16_ERR_ARG). */
W8A16_API int w8a16_gemm_split_terms(const void *workspace, uint64_t workspace_bytes, const void *W,
                                     const float *block_scale, void *C, uint32_t c_row_stride,
                                     uint32_t M, uint32_t N, uint32_t K, uint32_t flags,
                                     w8a16_stream_t stream);

/* ---- errors and status -------------------------------------------------- */

/* Message of the last failed call on this host thread ("" if none). */
W8A16_API const char *w8a16_last_error(void);

/* Weight element types accepted by w8a16_quantize_weights. */
enum {
    W8A16_WEIGHTS_F32 = 0,
    W8A16_WEIGHTS_BF16 = 1
};

/* Block quantiser: produces the W and block_scale operands of w8a16_gemm from
 * higher-precision weights. Output format: page "metrale_model_layers/layers/ops/
 * w8a16_gemm_pipelined_m32.rs", doc comment of `w8a16_gemm_pipelined_m32_strided`
 * (W as FP8 E4M3 [N][K], block_scale FP32 [N/128][K/128], one scale per 128x128
 * block). The page does not print the quantiser; our reading, consistent with the
 * 448 range of E4M3: per block, amax = max |w|; scale = amax / 448 (FP32, round to
 * nearest); code = E4M3 round-to-nearest-even of w / scale (FP32 quotient),
 * saturating at +-448; a block with amax = 0 gets scale 0 and all codes 0.
 *   W           FP32 or BF16 (w_dtype = W8A16_WEIGHTS_*), [N][w_row_stride], first K
 *               of each row read; device pointer, 16-byte aligned.
 *   codes       [N][K] E4M3 bytes (row pitch K), 4-byte aligned, written.
 *   block_scale [ceil(N/128)][K/128] FP32, 4-byte aligned, written.
 * Checks, before any device work: N >= 1, K a positive multiple of 128,
 * w_row_stride >= K and a multiple of 4, known w_dtype, non-NULL and aligned
 * pointers. NaN weights do not enter a block's amax and encode as the NaN code.
 * Asynchronous on `stream`. */
W8A16_API int w8a16_quantize_weights(const void *W, uint32_t w_dtype, uint32_t w_row_stride,
                                     uint32_t N, uint32_t K, void *codes, float *block_scale,
                                     w8a16_stream_t stream);

/* Per-token group activation quantiser, the first half of the W8A8 variant: BF16
 * activations -> E4M3 codes with one FP32 scale per token and 128-K group. The page
 * ("metrale_model_layers/layers/ops/fp8_act_quant.rs", module doc) gives the
 * grouping (one 128-element K group per scale) but not the arithmetic; our reading,
 * the same rule as w8a16_quantize_weights on 1x128 groups: amax = max |a|, scale =
 * amax / 448 (FP32, round to nearest), code = E4M3 RNE of a / scale, saturating;
 * amax = 0 gives scale 0 and codes 0; NaN values do not enter amax.
 *   A      BF16 [M][a_row_stride] (first K of a row read), a_row_stride a multiple of 8.
 *   codes  E4M3 [M][K], written (row pitch K).
 *   scales FP32 [K/128][scale_stride], written: K-group major, so one K step's scales
 *          of consecutive tokens are contiguous; scale_stride >= M, a multiple of 4.
 * A, codes and scales 16-byte aligned. Checks before any device work. The kernel is
 * queued as a programmatic dependent launch that waits for the previous kernel of the
 * stream before it reads or writes memory (nothing for the caller to do); a following
 * w8a16_gemm_w8a8 with W8A16_FLAG_PDL then prefetches its weights while it runs. */
W8A16_API int w8a16_quantize_activations(const void *A, uint32_t a_row_stride, uint32_t M,
                                         uint32_t K, void *codes, float *scales,
                                         uint32_t scale_stride, w8a16_stream_t stream);

/* W8A8 GEMM, the adjacent precision variant:
 *   C[m][n] = bf16( sum_k (e4m3(A[m][k]) * a_scale[k/128][m]) *
 *                         (e4m3(W[n][k]) * block_scale[n/128][k/128]) )
 * with A and a_scale as w8a16_quantize_activations writes them (a_row_stride in bytes,
 * >= K and a multiple of 16; a_scale_stride >= M, a multiple of 4), W, block_scale
 * and C as in w8a16_gemm. Per 128-K step one FP8 x FP8 product on the tensor cores,
 * folded in FP32 as acc += (block_scale * a_scale) * P, split-K partials added in rank
 * order (deterministic). One or two tokens run on the decode kernel where its rule
 * admits the shape (W8A16_VARIANT_GEMV, the codes copied in as its hi term), else on
 * the W8A8 kernel. A, a_scale and W 16-byte aligned. flags: W8A16_FLAG_PDL (the
 * previous grid must not write W or block_scale). Same error codes and checks as
 * w8a16_gemm, plus the two pitches above. */
W8A16_API int w8a16_gemm_w8a8(const void *A, uint32_t a_row_stride, const float *a_scale,
                              uint32_t a_scale_stride, const void *W, const float *block_scale,
                              void *C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
                              uint32_t flags, w8a16_stream_t stream);

/* w8a16_gemm_w8a8 with an explicit plan (variant W8A16_VARIANT_W8A8, or
 * W8A16_VARIANT_GEMV for M <= 2, from w8a16_plan_variant); a plan of another variant
 * is refused with W8A16_ERR_PLAN. */
W8A16_API int w8a16_gemm_w8a8_with_plan(const void *A, uint32_t a_row_stride,
                                        const float *a_scale, uint32_t a_scale_stride,
                                        const void *W, const float *block_scale, void *C,
                                        uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
                                        const w8a16_plan_t *plan, uint32_t flags,
                                        w8a16_stream_t stream);

/* Fixed description of a W8A16_ERR_* code. */
W8A16_API const char *w8a16_strerror(int code);

/* Synchronises `stream`, then reports the first device-side failure recorded on the
 * current device since the last clear: *status = W8A16_STATUS_*, *where =
 * blockIdx.x | blockIdx.y << 16 of the failing CTA, *detail = which wait. Any
 * pointer may be NULL. clear != 0 resets the record. Returns W8A16_OK or
 * W8A16_ERR_DEVICE. */
W8A16_API int w8a16_device_status(w8a16_stream_t stream, int clear, uint32_t *status, uint32_t *where,
                        uint32_t *detail);

/* Failure-path self-test: launches one CTA whose mbarrier wait can never complete
 * (nothing arrives on it) with a limit of `timeout_us` microseconds, so the kernel
 * must record W8A16_STATUS_WAIT_TIMEOUT (detail 0xFF) and return. It allows a
 * programmatic dependent launch to start at once. Used by the tests to show a wait
 * that runs out leaves the context usable, and that a call queued behind a long
 * kernel with W8A16_FLAG_PDL does not charge that kernel's time to its own waits. */
W8A16_API int w8a16_selftest_wait_timeout(uint32_t timeout_us, w8a16_stream_t stream);

/* Library version string. */
W8A16_API const char *w8a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W8A16_H */
