/*
 * fgemm.h -- C ABI of the fgemm library: dense half-precision matrix
 * multiplication C = epi(alpha * A * B + bias) on one GB300 (sm_103a), in a
 * classical form and in Strassen-like low-complexity forms (one or two
 * recursion levels), with an analytical picker that chooses the algorithm
 * and the tile per shape.
 *
 * Sources of the operations declared here:
 *  - Low-complexity matrix multiplication (LCMA), Strassen-like, with a
 *    recursion depth; a runtime model that picks algorithm and tiling from
 *    compute throughput, memory bandwidth and the per-depth overhead; runtime
 *    dispatch on the actual (M, N, K): FalconGEMM summary (arXiv 2605.06057),
 *    "Methodology" items 1, 3, 4, 5 and "Results & Findings".
 *  - Mainloop + epilogue split, epilogue fusion of scaling, elementwise ops
 *    and SwiGLU: PingPong GEMM / CODA note (tilnote), opening section and
 *    "How CODA applies it".
 *  - 16-bit inputs with fp32 accumulation: CS336 Lecture 05 notes, "Page 26.
 *    Low precision drives faster matrix multiplies".
 *  - Tile and wave quantization, roofline: CS336 Lecture 05 notes, "Page 21",
 *    "Page 43" and "Page 48".
 *
 * Conventions for every entry point:
 *  - All matrices are row-major. Leading dimensions (lda, ldb, ldc) are in
 *    elements. A is M x K, B is K x N, C is M x N_out with N_out = N, except
 *    for FGEMM_EPI_SWIGLU where N_out = N / 2.
 *  - Matrix and bias pointers are DEVICE pointers owned by the caller. The
 *    library never frees, reads back or retains them beyond the call.
 *  - Calls are asynchronous on the handle's stream: fgemm_matmul returns once
 *    the kernel is enqueued. Errors found on the device (a bounded wait that
 *    ran out) are latched in the handle and returned by fgemm_get_error.
 *  - Argument errors are returned before anything is launched.
 *  - A handle is used by one host thread at a time.
 */
#ifndef FGEMM_H
#define FGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fgemm_handle_s* fgemm_handle_t;

/* Element type of A, B, C and bias (all four share it). */
typedef enum { FGEMM_F16 = 0, FGEMM_BF16 = 1 } fgemm_dtype_t;

/* AUTO lets the decision model choose; the others force a form. */
typedef enum {
  FGEMM_ALGO_AUTO = 0,
  FGEMM_ALGO_CLASSICAL = 1,
  FGEMM_ALGO_STRASSEN1 = 2, /* one Strassen level: 7 half-size products */
  FGEMM_ALGO_STRASSEN2 = 3, /* two levels: 49 quarter-size products. One-CTA
                             * tiles (tile_m 128, sums formed on chip) or CTA
                             * pairs (tile_m 256: the 49 leaf operands of each
                             * side formed by a pre-pass, each from the 16
                             * quarter blocks with one rounding; no SWIGLU) */
  FGEMM_ALGO_WINOGRAD1 = 4  /* one level of Winograd's variant: 7 half-size
                             * products whose operands are sums of up to four
                             * blocks (FalconGEMM summary, "Methodology" item 1
                             * names it; standard identities). One-CTA tiles
                             * (tile_m 128) or CTA pairs (tile_m 256), tile_n
                             * 128 or 256. */
} fgemm_algo_t;

/*
 * Epilogue applied to the fp32 accumulator before the single rounding to the
 * output type (PingPong GEMM / CODA note: the epilogue scales and applies
 * elementwise operations before the write-back; CODA fuses SwiGLU there):
 *   v = alpha * acc[i][j] + bias[j]            (bias term only if bias != NULL)
 *   NONE, SCALE_BIAS : C[i][j] = v
 *   SILU             : C[i][j] = v / (1 + exp(-v))
 *   SWIGLU           : C[i][j] = silu(v[i][j]) * v[i][j + N/2], j < N/2
 *                      (columns [0, N/2) of A*B are the gate, [N/2, N) the up
 *                      projection; bias, if given, has N entries).
 * SCALE_BIAS requires bias. bias has N entries of the element type, device
 * memory, 2-byte aligned.
 */
typedef enum {
  FGEMM_EPI_NONE = 0,
  FGEMM_EPI_SCALE_BIAS = 1,
  FGEMM_EPI_SILU = 2,
  FGEMM_EPI_SWIGLU = 3
} fgemm_epi_kind_t;

typedef struct {
  int32_t kind;     /* fgemm_epi_kind_t */
  float alpha;      /* scale of the accumulator */
  const void* bias; /* device pointer or NULL */
} fgemm_epilogue_t;

typedef enum {
  FGEMM_OK = 0,
  FGEMM_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, ld too small, bad enum */
  FGEMM_ERR_ALIGNMENT = 2,   /* pointer or row stride not 16-byte aligned */
  FGEMM_ERR_UNSUPPORTED = 3, /* forced algorithm / tile not legal for shape */
  FGEMM_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  FGEMM_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel ran out */
  FGEMM_ERR_NO_DEVICE = 6,   /* no usable sm_103 device */
  FGEMM_ERR_CALIBRATION = 7  /* calibration file unreadable or malformed */
} fgemm_status_t;

/*
 * Creates a handle on the CURRENT CUDA device. The handle owns: a device
 * error word, a plan cache, a tensor-descriptor cache, the partial-tile
 * workspace (grown on demand), the split-piece counters and the device model.
 * The device model starts from the device's SM count and the rates measured
 * on a GB300 (fgemm_model_default) and, if the environment variable
 * FGEMM_CALIB names a JSON file, from that file (fgemm_model_load_json: a
 * calibration written by fgemm_calibrate, or measured peaks).
 * Returns FGEMM_ERR_NO_DEVICE if no device is present or it is not sm_103,
 * FGEMM_ERR_CALIBRATION if FGEMM_CALIB names a bad file.
 */
fgemm_status_t fgemm_create(fgemm_handle_t* out);

/* Frees everything the handle owns. NULL is accepted. Synchronises the
 * handle's stream first. */
fgemm_status_t fgemm_destroy(fgemm_handle_t h);

/* Sets the cudaStream_t (passed as void*) later calls are enqueued on.
 * NULL selects the legacy default stream (the initial value). */
fgemm_status_t fgemm_set_stream(fgemm_handle_t h, void* cuda_stream);

/*
 * C = epi(alpha * A * B + bias); see the conventions above.
 *   M, N, K    >= 0. M == 0 or N_out == 0: nothing is done. K == 0: C = epi(bias).
 *   A, lda     device pointer, M x K, lda >= K.
 *   B, ldb     device pointer, K x N, ldb >= N.
 *   C, ldc     device pointer, M x N_out, ldc >= N_out. C is only written.
 *   epi        NULL means NONE with alpha = 1 and no bias.
 *   algo       FGEMM_ALGO_AUTO or a forced form.
 * Alignment: A, B, C 16-byte aligned and lda, ldb, ldc multiples of 8
 * elements (the tensor-memory-access engine needs 16-byte rows), and for
 * SWIGLU N a multiple of 16 -> else FGEMM_ERR_ALIGNMENT.
 * Strassen forms need M, N, K (for SWIGLU: M, N/2, K) divisible into 2^d
 * blocks that are whole numbers of tiles (128 rows, 128 or 256 columns, 64
 * along K) -> else FGEMM_ERR_UNSUPPORTED; AUTO never picks an illegal form.
 * Strassen forms use the handle's workspace (4^d partial tiles per SM); a
 * classical CTA-pair launch whose last wave is split along K (see
 * fgemm_set_split_mode) uses it for the pieces' fp32 partial tiles and a
 * small counter buffer the handle allocates once.
 */
fgemm_status_t fgemm_matmul(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                            const void* A, int64_t lda, const void* B,
                            int64_t ldb, void* C, int64_t ldc,
                            fgemm_dtype_t dtype, const fgemm_epilogue_t* epi,
                            fgemm_algo_t algo);

/*
 * As fgemm_matmul, with the output tile forced (used for exhaustive timing of
 * the decision model's choices). tile_m = 128: one CTA per tile, tile_n in
 * {64, 128, 256}; tile_m = 256: a pair of CTAs (one M = 256 tensor-core
 * operation across two SMs), tile_n in {128, 256}, every form (two
 * Strassen levels without SWIGLU); tile_m = 16, 32 or 64: the small-M kernel for M <= tile_m
 * (classical, no SWIGLU, tile_n = 128 columns of C per tile): it computes
 * C^T = B^T A^T so that the tensor-core rows run over N, and shares the K
 * blocks of all tiles evenly over the CTAs of the grid fgemm_small_m_grid
 * picks (pieces of a tile are summed in a fixed order). SWIGLU needs tile_n >= 128; the Strassen forms use tile_n in
 * {128, 256}. tile_m = tile_n = 0 lets
 * the model choose; a zero in only one of them lets the model choose the
 * other.
 */
fgemm_status_t fgemm_matmul_ex(fgemm_handle_t h, int64_t M, int64_t N,
                               int64_t K, const void* A, int64_t lda,
                               const void* B, int64_t ldb, void* C, int64_t ldc,
                               fgemm_dtype_t dtype, const fgemm_epilogue_t* epi,
                               fgemm_algo_t algo, int32_t tile_m,
                               int32_t tile_n);

/*
 * RMSNorm statistics carried by the epilogue (PingPong GEMM / CODA note,
 * CODA section: the epilogue also produces what the following normalisation
 * needs). RMSNorm of a row x of width n with gain g is
 *   y_j = x_j g_j / sqrt(mean_j x_j^2 + eps),
 * and y W = diag(r) x (diag(g) W) with r = 1 / sqrt(mean_j x_j^2 + eps), so
 * a product can hand the next one its rows' sums of squares and the next one
 * scales its accumulator rows by r (g folded into its weights by the caller).
 *   sumsq_out   NULL, or device fp32 [ceil(N_out / 64)][M] (row-major: block
 *               p's M sums are contiguous): for each row and block of 64
 *               output columns, the sum of squares of the values as stored in
 *               C (after rounding), accumulated in column order in fp32.
 *   sumsq_in    NULL, or device fp32 [sumsq_parts][M] written by an earlier
 *               call: the accumulator of row i is multiplied by
 *               r_i = 1 / sqrt(sum_p sumsq_in[p][i] / norm_width + eps)
 *               (blocks summed in order, fp32) before alpha, bias and the
 *               activation.
 *   sumsq_parts blocks in sumsq_in (>= 1 with sumsq_in); norm_width >= 1 the
 *               normalised width; eps >= 0.
 * Both pointers 4-byte aligned, else FGEMM_ERR_ALIGNMENT.
 */
typedef struct {
  float* sumsq_out;
  const float* sumsq_in;
  int32_t sumsq_parts;
  int64_t norm_width;
  float eps;
} fgemm_rms_t;

/*
 * fgemm_matmul_ex with A, B, C and the bias (epi->bias) in HOST memory: the
 * call a user with host buffers makes (PingPong GEMM / CODA note: keep the
 * tensor cores busy during data movement). B and the bias are copied to the
 * device first; A is cut into row blocks (up to 8, each a multiple of 512
 * rows and at least about six waves of 256 x 256 tiles; one block when M does
 * not divide so) that are uploaded on the handle's upload stream while the
 * earlier blocks are multiplied on the handle's stream and their C blocks are
 * downloaded on its download stream, two device slots of each, ordered by
 * events. Every block runs the same form (AUTO's plan for the block's shape,
 * or the forced algo / tile). The copies overlap only for page-locked host
 * memory (cudaHostAlloc / cudaHostRegister); pageable memory works but
 * serialises. Returns once everything is enqueued: C is written when the
 * handle's stream reaches this point (cudaStreamSynchronize on it), and the
 * host buffers must stay valid until then. lda >= K, ldb >= N, ldc >= N_out
 * (any alignment). The device copies live in handle-owned buffers (grown on
 * demand; two slots each of B with the bias, of A row blocks and of C row
 * blocks). Errors as for fgemm_matmul_ex, plus FGEMM_ERR_CUDA for a failed
 * copy. RMSNorm statistics are not offered here.
 */
fgemm_status_t fgemm_matmul_host(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                 const void* A, int64_t lda, const void* B, int64_t ldb,
                                 void* C, int64_t ldc, fgemm_dtype_t dtype,
                                 const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                 int32_t tile_m, int32_t tile_n);

/*
 * fgemm_matmul_host with flags. FGEMM_HOST_OVERLAP: the call's uploads do not
 * wait for work already on the handle's stream, only for the device slots
 * they reuse (two each of B, A blocks and C blocks, cycled over calls) and
 * for the last two host calls on this handle whose C overlaps this call's A,
 * B or bias; so the next call's uploads run under this call's products.
 * The caller then guarantees that no other pending work on the handle's
 * stream writes this call's host inputs. C is still written when the
 * handle's stream reaches the point after the call. Unknown flags ->
 * FGEMM_ERR_INVALID_ARG.
 */
#define FGEMM_HOST_OVERLAP 1
fgemm_status_t fgemm_matmul_host_ex(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, const void* B, int64_t ldb,
                                    void* C, int64_t ldc, fgemm_dtype_t dtype,
                                    const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                    int32_t tile_m, int32_t tile_n, int32_t flags);

/*
 * As fgemm_matmul_ex, with RMSNorm statistics (rms may be NULL). Classical
 * form on one-CTA or CTA-pair tiles only (tile_m 128 or 256; AUTO chooses
 * among those), never with the last-wave K split; K >= 1. Other forced forms
 * or tiles return FGEMM_ERR_UNSUPPORTED.
 */
fgemm_status_t fgemm_matmul_rms(fgemm_handle_t h, int64_t M, int64_t N,
                                int64_t K, const void* A, int64_t lda,
                                const void* B, int64_t ldb, void* C, int64_t ldc,
                                fgemm_dtype_t dtype, const fgemm_epilogue_t* epi,
                                fgemm_algo_t algo, int32_t tile_m, int32_t tile_n,
                                const fgemm_rms_t* rms);

/*
 * Block-scaled 8-bit inputs (MX; CS336 Lecture 05 notes, "Page 27. Frontiers
 * in low precision - FP8 and MXFP8" and "Page 28. MXFP8 training in
 * practice"): C = epi(alpha * A * B + bias) where every element of A and B is
 * an 8-bit float times the E8M0 scale (2^(e - 127), e = 255 NaN) of its block
 * of 32 values along K.
 *   A, lda          device, M x K bytes, lda >= K.
 *   scale_a, ld_sa  device, M x ceil(K/32) E8M0 bytes: row i, block k/32.
 *   B, ldb          device, K x N bytes, ldb >= N.
 *   scale_b, ld_sb  device, ceil(K/32) x N E8M0 bytes: block k/32, column j.
 *   a_format, b_format  FGEMM_FP8_E4M3 or FGEMM_FP8_E5M2.
 *   C, ldc, epi     as fgemm_matmul_ex, in bf16 (bias bf16 too).
 * Each value is written to bf16 first, which is exact while it lies in
 * bf16's normal range; outside it the exact value is rounded once (RNE, to
 * a subnormal or infinity). Those bf16 matrices live in a handle-owned
 * buffer (grown on demand), and the product then runs as fgemm_matmul_ex
 * with algo / tile_m / tile_n. This function has no fused 8-bit tensor-core
 * path: the product runs at the bf16 rate.
 */
typedef enum { FGEMM_FP8_E4M3 = 0, FGEMM_FP8_E5M2 = 1 } fgemm_fp8_format_t;

/*
 * The first step of fgemm_matmul_mx on its own: Y (rows x cols bf16, ld ldy,
 * 16-byte aligned rows for the fast path) = the values of the block-scaled
 * matrix X (rows x cols bytes, ld ldx) with E8M0 scales S (ld lds): blocks of
 * 32 along each row (along 0, S is rows x ceil(cols/32)) or down each column
 * (along 1, S is ceil(rows/32) x cols). Each value is rounded once to bf16
 * (exact while in bf16's normal range). Asynchronous on the handle's stream.
 * Errors: FGEMM_ERR_INVALID_ARG for a bad format or along, a negative size,
 * cols above 2^31 - 1, NULL pointers or leading dimensions below the row
 * lengths; FGEMM_ERR_ALIGNMENT for an odd Y address.
 */
fgemm_status_t fgemm_mx_to_bf16(fgemm_handle_t h, int64_t rows, int64_t cols,
                                const void* X, int64_t ldx, const void* S, int64_t lds,
                                int32_t format, int32_t along, void* Y, int64_t ldy);

fgemm_status_t fgemm_matmul_mx(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* scale_a,
                               int64_t ld_sa, int32_t a_format, const void* B,
                               int64_t ldb, const void* scale_b, int64_t ld_sb,
                               int32_t b_format, void* C, int64_t ldc,
                               const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                               int32_t tile_m, int32_t tile_n);

/*
 * Runs the decision model (no launch): the algorithm, tile and predicted
 * time AUTO would use for this shape (FalconGEMM summary, "Methodology"
 * items 4 and 5): the same choice as fgemm_model_plan on the handle's model,
 * lcma_margin included. Output pointers may be NULL.
 */
fgemm_status_t fgemm_plan(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                          fgemm_dtype_t dtype, const fgemm_epilogue_t* epi,
                          fgemm_algo_t* algo_out, int32_t* tile_m,
                          int32_t* tile_n, double* predicted_us);

/*
 * As fgemm_plan, with the choice restricted: algo (FGEMM_ALGO_AUTO: any
 * form), tile_m_in and tile_n_in (0: any) constrain the candidates the model
 * ranks, as a forced form or tile in fgemm_matmul_ex does; the result is
 * what that call would launch (under AUTO a low-complexity candidate must
 * beat the best classical one by lcma_margin). FGEMM_ERR_UNSUPPORTED if no
 * candidate is legal for the shape.
 */
fgemm_status_t fgemm_plan_ex(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                             fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                             int32_t tile_m_in, int32_t tile_n_in, fgemm_algo_t* algo_out,
                             int32_t* tile_m, int32_t* tile_n, double* predicted_us);

/* Synchronises the handle's stream, then returns and clears the latched
 * device error (FGEMM_OK, FGEMM_ERR_TIMEOUT or FGEMM_ERR_CUDA). */
fgemm_status_t fgemm_get_error(fgemm_handle_t h);

/*
 * How many kernels of this library one fgemm_matmul_ex call with these
 * arguments launches on the handle with its current settings (the plan AUTO
 * or the forced form resolves to; for one Strassen-like level on CTA pairs,
 * the operand pre-pass unless the product kernel forms the sums itself, see
 * fgemm_set_lcma_formation; for two levels on CTA pairs, always the
 * pre-pass and the product kernel). Host only: launches nothing. Writes *launches;
 * returns the plan's errors (FGEMM_ERR_UNSUPPORTED for an illegal forced
 * form) or FGEMM_ERR_INVALID_ARG for a NULL handle, a NULL output or an
 * unknown algorithm.
 */
fgemm_status_t fgemm_call_launches(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                   const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                   int32_t tile_m, int32_t tile_n, int32_t* launches);

/*
 * Measures the device (tensor throughput of each classical tile width and
 * of each Strassen form, streaming bandwidth) with the library's own
 * kernels, updates the handle's device model, and writes it as JSON to
 * json_out_path if that is not NULL (FalconGEMM summary, "Methodology" item
 * 4: the model is built from measured compute throughput and bandwidth).
 * Allocates and frees its own scratch matrices. Takes about a second.
 */
fgemm_status_t fgemm_calibrate(fgemm_handle_t h, const char* json_out_path);

/*
 * fgemm_calibrate on n x n x n products (n a multiple of 1024 in [1024,
 * 16384]; fgemm_calibrate uses 8192). Besides the mainloop rates it
 * measures the launch cost (back-to-back K = 0 calls) and the pipeline fill
 * and drain (the intercept in K of a one-tile product's time, less the
 * launch). FGEMM_ERR_INVALID_ARG for another n.
 */
fgemm_status_t fgemm_calibrate_ex(fgemm_handle_t h, int64_t n, const char* json_out_path);

/*
 * Failure-detection self-test. Launches a one-block kernel that waits on an
 * mbarrier nothing will ever complete, through the same bounded wait every
 * GEMM kernel uses, with the limit set to limit_ms (1..10000) for this
 * launch. The wait gives up, the kernel latches a timeout in the handle's
 * error word and exits normally: no fault, no trap, and the handle stays
 * usable. Asynchronous; fgemm_get_error then returns FGEMM_ERR_TIMEOUT.
 */
fgemm_status_t fgemm_selftest_wait_timeout(fgemm_handle_t h, int32_t limit_ms);

/* Static string naming a status. */
const char* fgemm_status_string(fgemm_status_t s);

/* Text of the last error reported on this handle (or, for h == NULL, on this
 * thread by a call without a handle). Valid until the next call. */
const char* fgemm_last_message(fgemm_handle_t h);

/*
 * Host-only argument check used by fgemm_matmul_ex (no device needed):
 * returns the status fgemm_matmul_ex would return before launching.
 */
fgemm_status_t fgemm_validate(int64_t M, int64_t N, int64_t K, const void* A,
                              int64_t lda, const void* B, int64_t ldb,
                              const void* C, int64_t ldc, fgemm_dtype_t dtype,
                              const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                              int32_t tile_m, int32_t tile_n);

/*
 * Strassen product (depth 1 or 2) that allocates no device memory. The paper
 * has no counterpart; it exists for callers that may not call cudaMalloc:
 * code running under a framework whose pool owns all device memory, serving
 * loops that must not pay cudaMalloc's implicit device synchronisation, or
 * plug-ins that are handed nothing but buffers and a stream.
 *
 * It computes what fgemm_matmul_ex(..., FGEMM_ALGO_STRASSEN1 or 2, 128, tile_n)
 * computes, with no handle: the scratch it needs (the kernel's error word and
 * the fp32 partial tiles of the Strassen combination) lives in a 64 MiB
 * array built into the library, which every device that loads the library
 * keeps until the process exits.
 *   depth      1 or 2.   tile_n  128 or 256 (0 = 128).
 *   cuda_stream  the cudaStream_t (as void*) to enqueue on; NULL = legacy.
 *   other arguments, layouts, alignment and legality: as fgemm_matmul_ex.
 * Limit: the launch uses min(tiles, SMs) CTAs, each needing 4^depth partial
 * tiles of 128 x tile_n floats (depth 1: 256 KiB at tile_n 128, 512 KiB at
 * 256; depth 2: 1 or 2 MiB). A product that needs more than the array's
 * 64 MiB returns FGEMM_ERR_UNSUPPORTED (message: how much it needs) before
 * anything is enqueued.
 * The first call on each device finds the array's device address
 * (cudaGetSymbolAddress, which loads the library's device code): make that
 * first call before capturing a stream. Every call shares the one array and
 * leaves its contents behind; calls whose kernels overlap on the GPU (other
 * streams, or other host threads) race on it and must be serialised by the
 * caller. A bounded wait that runs out inside the kernel (it does not happen
 * unless the GPU stalls for about a second) leaves C incomplete; the kernel
 * latches a code in the array's error word, which stays set until
 * fgemm_strassen_static_get_error reads and clears it. While it is set,
 * later calls on the same device give up their waits early (as a handle's
 * calls do until fgemm_get_error), so check it before trusting results.
 */
fgemm_status_t fgemm_strassen_matmul_static(
    int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
    int64_t ldb, void* C, int64_t ldc, fgemm_dtype_t dtype,
    const fgemm_epilogue_t* epi, int32_t depth, int32_t tile_n,
    void* cuda_stream);

/*
 * The error word of fgemm_strassen_matmul_static on the current device:
 * synchronises cuda_stream (NULL = legacy stream), then returns FGEMM_OK, or
 * FGEMM_ERR_TIMEOUT (fgemm_last_message(NULL) names the role and block)
 * after clearing the word. Allocates nothing.
 */
fgemm_status_t fgemm_strassen_static_get_error(void* cuda_stream);

/*
 * Failure-detection self-test of the allocation-free path: one block waits
 * on an mbarrier nothing completes, through the bounded wait of the GEMM
 * kernels, with the limit limit_ms (1..10000); it gives up, latches a timeout
 * in the static error word and exits normally (no fault, no trap).
 * Asynchronous on cuda_stream. Allocates nothing.
 */
fgemm_status_t fgemm_strassen_static_selftest_timeout(int32_t limit_ms, void* cuda_stream);

/* ------------------------------------------------------------------------
 * Decision model, host only (no device needed). FalconGEMM summary,
 * "Methodology" item 4 (analytical runtime model: compute throughput, memory
 * bandwidth, overhead per recursion depth) with the tile and wave
 * quantization terms of the CS336 Lecture 05 notes, "Page 43" and "Page 48",
 * and the roofline of "Page 21".
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t num_sms;         /* SMs: one persistent CTA per SM, one pair per 2 */
  int32_t reserved;
  double peak_tflops;      /* dense 16-bit tensor peak, TFLOP/s */
  double hbm_gbs;          /* streaming HBM bandwidth, GB/s */
  double eff_classical[3]; /* mainloop fraction of peak, 128 x {64, 128, 256} */
  double eff_pair[2];      /* same for CTA-pair tiles 256 x {128, 256} */
  double eff_strassen[2][2]; /* [depth-1][tile_n 128, 256]: executed-MAC rate
                              * of the Strassen mainloop as a fraction of peak */
  double eff_strassen_pair[2]; /* one level on CTA pairs, 256 x {128, 256} */
  double launch_us;        /* fixed cost of one launch */
  double tile_fill_us;     /* pipeline fill + drain cost per tile visit */
  double l2_bytes;         /* L2 capacity (bytes) */
  double l2_gbs;           /* L2 -> SM operand bandwidth, GB/s */
  double split_fix_us;     /* fixed cost of splitting the last wave of CTA-pair
                            * tiles along K (partial stores, the sum by the last
                            * piece, its exposed epilogue) */
  double eff_winograd[2];  /* one Winograd level, 128 x {128, 256}: executed-MAC
                            * rate of its mainloop as a fraction of peak */
  double eff_small_m[3];   /* small-M tiles (tile_m 16, 32, 64): MMA rate as a
                            * fraction of peak (an N = tile_m MMA runs at most
                            * tile_m / 256 of the full rate) */
  double hbm_stream_eff;   /* fraction of hbm_gbs a kernel streaming B reaches */
  double small_m_stream_eff; /* the same for the small-M kernel on a grid of more
                              * than 4 phases: its CTAs draw unequal shares of
                              * the bandwidth and the slowest sets the time */
  double small_m_fix_us;   /* its per-launch cost beyond the stream: the pieces'
                            * partial store, count and sum, and the slowest CTA */
  double small_m_aligned_eff; /* fraction of hbm_gbs the small-M kernel reaches on
                               * a grid whose shares start at no more than 4 K
                               * offsets of a tile (fgemm_small_m_grid) */
  double form_in_kernel_eff; /* fraction of hbm_gbs at which a one-level pair
                              * launch's own idle warps form the summed operands
                              * beside the products (fgemm_set_lcma_formation) */
  double form_in_kernel_drag; /* time the products lose to that formation, as a
                               * fraction of the formation's duration */
  double lcma_margin;      /* AUTO picks a low-complexity form only when its
                            * prediction is below (1 - lcma_margin) times the
                            * best classical one (clamped to [0, 0.9]; 0.9 keeps
                            * AUTO on the classical forms: the Strassen-like
                            * forms carry their larger rounding error, e.g.
                            * 6.4e-3 normwise for one Winograd level against
                            * 2.5e-4 classical on U[-1,1] bf16 inputs) */
  double dram_miss_slope;  /* share of the tiled operand reads re-read from
                            * DRAM per unit of (panel bytes of one wave / L2 - 1),
                            * capped at 1 */
  double dram_exposed;     /* part of that DRAM time not hidden by the MMAs */
  double eff_strassen2_pair[2]; /* two levels on CTA pairs, 256 x {128, 256}:
                                 * the product kernel's MMA rate */
  double fold2_unit_us;    /* two levels on CTA pairs: the epilogue's fold of
                            * one 256 x 256 product unit into its ~3 output
                            * blocks (fp32 reductions at the L2), which
                            * overlaps the unit's MMAs only in part */
} fgemm_device_model_t;

/*
 * Grid of the small-M kernel for `tiles` 128-column tiles of `k_blocks` K
 * blocks each on `num_sms` SMs. The K blocks of all tiles, laid end to end,
 * are cut into equal shares, one per CTA. Among the CTA counts from 3/4 of
 * the largest grid (every SM, each CTA at least 8 blocks) up to that grid,
 * the ones that divide tiles * k_blocks exactly are scored by their phases:
 * the number of distinct K offsets inside a tile at which shares start. The
 * count with the fewest phases wins (the larger count on a tie). Fewer
 * phases mean the CTAs read fewer distinct rows of B at a time. If no count
 * has 4 phases or fewer, the largest grid is returned with phases set to its
 * CTA count. Returns the CTA count (0 on invalid arguments) and writes the
 * phases to *phases_out when it is not NULL. Host-only.
 */
int32_t fgemm_small_m_grid(int64_t tiles, int32_t k_blocks, int32_t num_sms, int32_t* phases_out);

/*
 * CTA pairs a Strassen-like launch on CTA pairs uses for `positions` output
 * positions (256 x tile_n tiles of the 2^-depth-size block space) when `fit`
 * pairs fit on the device. One level: min(fit, 7 positions). Two levels:
 * every pair while the positions of the partial last wave, cut into 49
 * product units each, give at most 24 units per pair; with fewer positions
 * than pairs, one pair per position; otherwise the largest pair count from
 * fit down to fit / 2 that divides the positions into whole waves, if any
 * (else fit). Returns 0 for positions <= 0 or fit <= 0.
 * Host-only.
 */
int64_t fgemm_lcma_pair_clusters(int64_t positions, int32_t depth, int32_t fit);

/*
 * Default model for a device with the given SM count: the mainloop, launch
 * and streaming rates fgemm_calibrate measured on a GB300 (for 152 SMs,
 * scaled by the SM count), expressed as efficiencies against peak_tflops
 * (<= 0: 1891.3 TFLOP/s, the dense bf16 rate a GB300 measured, scaled by the
 * SM count) and hbm_gbs (<= 0: 6789 GB/s, its measured copy bandwidth). The
 * predicted times do not depend on the two denominators.
 */
void fgemm_model_default(fgemm_device_model_t* out, int32_t num_sms,
                         double peak_tflops, double hbm_gbs);

/*
 * Reads a flat JSON object into *model (host only), starting from its
 * current contents. Either a calibration as fgemm_model_save_json writes it
 * (keys named after the fields, e.g. "peak_tflops", "eff_pair_256",
 * "launch_us"; absent keys keep their values), or measured peaks: a dense
 * bf16 GEMM rate "bf16_tflops" and a copy bandwidth "hbm_gbs" with no
 * "peak_tflops", which become the model's denominators with every
 * efficiency rescaled so that the predicted rates do not change.
 * FGEMM_ERR_CALIBRATION if the file cannot be read, holds no known key, or
 * gives a non-positive peak or bandwidth or a negative fixed cost (then
 * *model is unchanged); FGEMM_ERR_INVALID_ARG for NULL arguments.
 */
fgemm_status_t fgemm_model_load_json(const char* path, fgemm_device_model_t* model);

/* Writes *model as the flat JSON object fgemm_model_load_json reads (host
 * only). FGEMM_ERR_CALIBRATION if the file cannot be written. */
fgemm_status_t fgemm_model_save_json(const fgemm_device_model_t* model, const char* path);

/* Tile quantization: ceil(M / tile_m) * ceil(N / tile_n). */
int64_t fgemm_model_tiles(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n);

/* Wave quantization: number of waves ceil(tiles / slots); *tail_util (may be
 * NULL) receives the occupancy of the last wave, (tiles mod slots) / slots,
 * or 1 when tiles is a multiple of slots. */
int64_t fgemm_model_waves(int64_t tiles, int32_t slots, double* tail_util);

/* Elements a tiled product reads from global memory: each tile_m x tile_n
 * output tile reads a tile_m x K block of A and a K x tile_n block of B, so
 * tiles * (tile_m + tile_n) * K; for square N with T x T tiles that is
 * 2 N^3 / T (CS336 Lecture 05 notes, "Page 42. Tiling math"). */
double fgemm_model_tiled_reads(int64_t M, int64_t N, int64_t K, int32_t tile_m,
                               int32_t tile_n);

/* Roofline: min(peak_flops, (flops / bytes) * bandwidth) in FLOP/s. */
double fgemm_model_roofline(double flops, double bytes, double peak_flops,
                            double bandwidth);

/* Predicted time (us) of one form and tile for a shape; returns
 * FGEMM_ERR_UNSUPPORTED if that form/tile is illegal for the shape. */
fgemm_status_t fgemm_model_predict(const fgemm_device_model_t* dev, int64_t M,
                                   int64_t N, int64_t K, int32_t epi_kind,
                                   fgemm_algo_t algo, int32_t tile_m,
                                   int32_t tile_n, double* predicted_us);

/* The argmin over every legal (form, tile): what AUTO launches. */
fgemm_status_t fgemm_model_plan(const fgemm_device_model_t* dev, int64_t M,
                                int64_t N, int64_t K, int32_t epi_kind,
                                fgemm_algo_t* algo_out, int32_t* tile_m,
                                int32_t* tile_n, double* predicted_us);

/*
 * Last-wave K split of the classical CTA-pair kernel (no counterpart on the
 * pages, which quantize waves but do not split them; the pages' own remedy
 * for wave quantization, CS336 Lecture 05 notes "Page 48", is choosing tile
 * sizes). With `tiles` output tiles on `clusters` pairs, the last wave would
 * run R = tiles % clusters tiles on R pairs while the rest idle. When
 * 2R <= clusters, the first R tiles (in rasterised order) are each cut into
 * S = min(clusters / R, k_blocks, 4) pieces of equal K range; piece s of
 * split tile t is the first work item of pair t * S + s, and every pair then
 * runs its (tiles - R) / clusters whole tiles. Each piece stores an fp32
 * partial; the last piece to finish sums the pieces in piece order
 * (deterministic) and applies the epilogue.
 *
 * fgemm_model_split_tail returns R (0 = no split) and writes S to *pieces
 * (1 when no split; pieces may be NULL). mode 0: never; 1 (auto): when at
 * least one whole wave remains (tiles >= clusters) and (1 - 1/S) * tile time
 * > (S - 1) * dev->split_fix_us; 2: whenever the conditions above allow. Requires 2 <= clusters <= 255; dev may be NULL for
 * modes 0 and 2.
 */
int32_t fgemm_model_split_tail(const fgemm_device_model_t* dev, int64_t tiles,
                               int32_t clusters, int32_t k_blocks, int32_t tile_n,
                               int32_t mode, int32_t* pieces);

/*
 * The n-th work item (n = 0, 1, ...) of pair `cluster` in the schedule
 * above: writes {unit, k0, k1, piece, npieces} (tile index, K blocks
 * [k0, k1), piece index among the tile's npieces; whole tiles have
 * npieces = 1) to out5 and returns 1, or returns 0 past the end of the list
 * (or on invalid arguments). Host-only; the kernel runs the same function.
 */
int32_t fgemm_split_work_item(int64_t tiles, int32_t split_tiles, int32_t split_pieces,
                              int32_t clusters, int32_t k_blocks, int32_t cluster,
                              int32_t n, int32_t* out5);

/*
 * The n-th work item of CTA `cta` of the small-M kernel (tile_m 16/32/64):
 * the K blocks of all `tiles` 128-column tiles, laid end to end, are cut into
 * `ctas` equal contiguous shares (stream-K). Writes {unit, k0, k1, piece,
 * npieces, slot} to out6 and returns 1, or returns 0 past the end of the
 * share (or on invalid arguments; ctas must not exceed tiles * k_blocks).
 * `slot` is the partial slot (0 .. 2 ctas - 1) the piece stores to when the
 * tile has more than one piece. Host-only; the kernel runs the same code.
 */
int32_t fgemm_stream_k_work_item(int64_t tiles, int32_t k_blocks, int32_t ctas, int32_t cta,
                                 int32_t n, int64_t* out6);

/*
 * K-split mode of the handle's classical CTA-pair launches: 0 never, 1 auto
 * (the default: fgemm_model_split_tail with the handle's device model), 2
 * whenever possible. Returns FGEMM_ERR_INVALID_ARG for other modes.
 */
fgemm_status_t fgemm_set_split_mode(fgemm_handle_t h, int32_t mode);

/*
 * Where the handle's one-level Strassen-like launches on CTA pairs (tile_m
 * 256) form their summed operands (FalconGEMM summary, "Methodology" item 3:
 * the operand sums of the low-complexity scheme): 1 a streaming pre-pass
 * launch before the product kernel; 2 inside the product kernel, by its two
 * otherwise idle warps per CTA, while the products that do not read those
 * sums run first: both sides' sums for Winograd's scheme (its A11 B11 and
 * A12 B21 read none), B's for Strassen's (its M2 and M5 read no sum of B;
 * A's then come from a pre-pass of half the size); 0 auto (the default):
 * mode 2 when those products span at least 16 waves of the launch, else
 * mode 1.  The result is the same
 * bit for bit in every mode.  Returns FGEMM_ERR_INVALID_ARG for other modes.
 */
fgemm_status_t fgemm_set_lcma_formation(fgemm_handle_t h, int32_t mode);

/* Copies the handle's current device model into *out. */
fgemm_status_t fgemm_get_device_model(fgemm_handle_t h,
                                      fgemm_device_model_t* out);

/* Replaces the handle's device model (clears the plan cache). */
fgemm_status_t fgemm_set_device_model(fgemm_handle_t h,
                                      const fgemm_device_model_t* model);

#ifdef __cplusplus
}
#endif

#endif /* FGEMM_H */
