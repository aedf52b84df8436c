/*
 * gptq.h -- C ABI of a GB300 (sm_103a) library for GPTQ's per-layer second-order
 * weight quantization.
 *
 * The operation (three web pages on GPTQ: "GPTQ › Mathematical Details of the Update";
 * "tm_gptq_math"; "GPTQ Hessian", excerpt of "GPTQ: Block Structure in Quantization"):
 * for one linear layer with weights W [d_out, d_in] and calibration inputs X, find a
 * few-bit W_hat whose outputs on X stay close to W's, one row at a time, all rows sharing
 * the Hessian H = 2 X X^T of the per-row quadratic error.  The path is split into the
 * three calls below, in the pages' order:
 *
 *   gptq_hessian_accumulate   X -> H          ("tm_gptq_math", "Why it is second-order:
 *                                               the Hessian")
 *   gptq_prepare              H -> U          ("tm_gptq_math", "The Cholesky trick for the
 *                                               inverse Hessian"; "GPTQ Hessian")
 *   gptq_quantize_layer       W, U -> codes   ("tm_gptq_math", "Greedy quantization with
 *                                               error compensation" and "GPTQ's speedups:
 *                                               fixed order and lazy batches"; "GPTQ Hessian")
 *
 * Conventions shared by every call
 *   - All matrices are row-major.  X is token-major [n_tok, d_in] (row t = input x_t, so
 *     the pages' X of shape [d_in, N] is X^T here).  W is [d_out, d_in].
 *   - Every pointer is a DEVICE pointer on the current CUDA device unless marked "host".
 *     The library never allocates, frees or keeps device memory beyond a call; the caller
 *     owns every buffer.  Scratch memory is a caller-supplied workspace whose size the
 *     *_workspace_bytes functions give; it must be 256-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Kernels are
 *     enqueued on it; calls return once work is enqueued unless stated otherwise.
 *   - Argument errors are reported synchronously, before anything is enqueued.  A failed
 *     kernel launch returns GPTQ_ERR_CUDA.
 *   - The calls are thread-compatible: concurrent calls must use distinct outputs and
 *     workspaces.
 */
#ifndef GPTQ_GB300_H
#define GPTQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GPTQ_ABI_VERSION 1

typedef struct CUstream_st *gptq_stream_t; /* identical to cudaStream_t */

typedef enum gptq_status {
  GPTQ_OK = 0,
  GPTQ_ERR_INVALID_ARG = 1,  /* bad size, dtype, bit width, block, null or misaligned ptr */
  GPTQ_ERR_NOT_PD = 2,       /* damped Hessian not positive definite (gptq_prepare)       */
  GPTQ_ERR_NONFINITE = 3,    /* NaN/Inf found in an input                                 */
  GPTQ_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up                        */
  GPTQ_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed               */
  GPTQ_ERR_UNSUPPORTED = 6,  /* valid request this library does not implement             */
  GPTQ_ERR_WORKSPACE = 7     /* workspace missing, too small or not 256-byte aligned      */
} gptq_status;

typedef enum gptq_dtype { GPTQ_F16 = 0, GPTQ_BF16 = 1, GPTQ_F32 = 2 } gptq_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *gptq_status_str(int status);

/* GPTQ_ABI_VERSION of the loaded library. */
int gptq_abi_version(void);

/* Number of CUDA kernels this library has launched in this process (all threads). */
unsigned long long gptq_kernel_launches(void);

/*
 * gptq_hessian_accumulate: H = (accumulate ? H : 0) + 2 * X^T X.
 *
 * Source: "tm_gptq_math", "Why it is second-order: the Hessian" -- the per-row output
 * error is a quadratic in the row's weights whose constant Hessian is twice the Gram
 * matrix of the inputs; "GPTQ Hessian" -- every row of the layer shares it.  Calling this
 * once per token chunk with accumulate=1 after the first accumulates the Hessian of the
 * whole calibration set while only one chunk of X is resident.
 *
 *   X          [n_tok, ldx] elements of type `xdtype`, first d_in columns used; 16-byte
 *              aligned, ldx * sizeof(elem) a multiple of 16 bytes.
 *   xdtype     GPTQ_F16 / GPTQ_BF16 (tensor-core path, fp32 accumulation) or GPTQ_F32.
 *   n_tok      >= 0 tokens (0 leaves H as is, or zero when accumulate=0).
 *   d_in       >= 1 input channels.
 *   H          [d_in, d_in] fp32, both triangles written.  With accumulate=1 the lower
 *              triangle of the existing H is read and the result is written symmetric.
 * Asynchronous.  Errors: INVALID_ARG, CUDA.
 */
gptq_status gptq_hessian_accumulate(const void *X, int xdtype, int64_t n_tok, int64_t d_in,
                                    int64_t ldx, float *H, int accumulate,
                                    gptq_stream_t stream);

/*
 * gptq_hessian_host_workspace_bytes: device staging workspace that
 * gptq_hessian_accumulate_host needs for inputs of d_in channels streamed in chunks of
 * chunk_tok tokens (0 = the default chunk: about 64 MiB of X, a multiple of 512 tokens, and
 * at least 8192 tokens, or 32768 from d_in = 16384 on, since every chunk's products read and
 * write all of H).
 * Returns 0 for an unknown dtype, d_in < 1 or chunk_tok < 0.
 */
size_t gptq_hessian_host_workspace_bytes(int xdtype, int64_t d_in, int64_t chunk_tok);

/*
 * gptq_hessian_accumulate_host: gptq_hessian_accumulate with X in HOST memory.
 *
 * Source: as gptq_hessian_accumulate ("tm_gptq_math", "Why it is second-order: the
 * Hessian"); the pages accumulate the Gram matrix over the calibration set, which is what
 * the chunks below do.  The pages have no counterpart to the host staging itself: it
 * exists so that the calibration activations need not be resident on the GPU, and so that
 * their transfer overlaps the Gram products.
 *
 * X is copied to the device in chunks of chunk_tok tokens through two staging buffers in
 * `ws`; the copy of chunk c + 1 runs on a copy stream this library keeps per device while
 * chunk c is accumulated into H on `stream`.  Chunks are accumulated in token order, each
 * exactly as one gptq_hessian_accumulate call over that chunk would (so the fp32 sums are
 * grouped by chunk; the result can differ in the last bits from one call over all tokens).
 *
 *   X_host     HOST [n_tok, ldx] elements of xdtype, first d_in columns used.  Page-locked
 *              memory (cudaHostAlloc / cudaHostRegister) lets the copies overlap; pageable
 *              memory gives the same result, but each copy then blocks the calling thread.
 *              Must stay valid and unchanged until the work on `stream` has completed.
 *   xdtype     GPTQ_F16, GPTQ_BF16 or GPTQ_F32;  d_in * sizeof(elem) a multiple of 16 bytes.
 *   n_tok      >= 0;  ldx >= d_in (host rows may be strided; no alignment needed).
 *   H          as gptq_hessian_accumulate (DEVICE, 16-byte aligned); `accumulate` applies
 *              to the first chunk, later chunks always accumulate.
 *   chunk_tok  tokens per chunk (0 = default); the same value as in the size query.
 *   ws         DEVICE workspace, 256-byte aligned, of ws_bytes >=
 *              gptq_hessian_host_workspace_bytes(xdtype, d_in, chunk_tok).
 * Returns once everything is enqueued (for page-locked X); every copy and product is
 * ordered before later work on `stream`, and the copies start only after earlier work on
 * `stream` (which may still use `ws`) has finished.  Calls from several host threads are
 * serialized while they enqueue.  Errors: INVALID_ARG, WORKSPACE, CUDA.
 */
gptq_status gptq_hessian_accumulate_host(const void *X_host, int xdtype, int64_t n_tok,
                                         int64_t d_in, int64_t ldx, float *H, int accumulate,
                                         int64_t chunk_tok, void *ws, size_t ws_bytes,
                                         gptq_stream_t stream);

/*
 * gptq_prepare_workspace_bytes: workspace size gptq_prepare needs for this d_in.
 */
size_t gptq_prepare_workspace_bytes(int64_t d_in);

/*
 * gptq_prepare: dead columns, damping and the inverse-Hessian Cholesky factor.
 *
 * Source: "tm_gptq_math", "The Cholesky trick for the inverse Hessian" -- channels with a
 * zero Hessian diagonal are skipped, the diagonal is damped by lambda = damp * mean(diag)
 * (about 1 %), and one Cholesky factorization of the inverse supplies every row the
 * fixed-order sweep needs; "GPTQ Hessian" -- U is the upper-triangular factor with
 * H^-1 = U^T U; "GPTQ › Mathematical Details of the Update" writes it as L = U^T.
 *
 * Steps: dead = {i : H_ii == 0}; H_ii = 1 for dead i; lambda = damp * mean(diag H) (after
 * that fix, over all d_in entries); H += lambda I; U = upper Cholesky factor of H^-1.
 * U is computed as the inverse of the reversed-order ("UL") Cholesky factor R of H
 * (H = R R^T, R upper), which is the same matrix.
 *
 *   H          [d_in, d_in] fp32 symmetric, CONSUMED: overwritten as scratch.  Only the
 *              upper triangle and the diagonal are read (the lower triangle may hold anything).
 *   d_in       >= 1.
 *   damp       >= 0 relative damping (0.01 for the pages' 1 %).
 *   U          [d_in, d_in] fp32 out, upper triangular (lower triangle written as 0).
 *   dead_mask  [d_in] uint8 out (1 = dead), may be NULL.
 *   n_dead     HOST int32 out, may be NULL.
 *   ws         workspace of ws_bytes >= gptq_prepare_workspace_bytes(d_in).
 * SYNCHRONIZES `stream` before returning.  Errors: INVALID_ARG, WORKSPACE, NOT_PD (a
 * pivot <= 0: U is then undefined), NONFINITE (NaN/Inf in the part of H read), CUDA.
 *
 * Repeatability: the factorization runs on several streams of this library that add into
 * shared blocks of the workspace in an order that is not fixed, so two calls on the same
 * H can give U's that differ in their last bits (relative row differences of order 1e-6).
 * A sweep on either gives the same codes except where a weight sits within rounding noise
 * of a grid boundary (the two codes are then adjacent).
 */
gptq_status gptq_prepare(float *H, int64_t d_in, float damp, float *U, uint8_t *dead_mask,
                         int32_t *n_dead, void *ws, size_t ws_bytes, gptq_stream_t stream);

/*
 * gptq_quantize_workspace_bytes: workspace size gptq_quantize_layer needs.
 */
size_t gptq_quantize_workspace_bytes(int64_t d_out, int64_t d_in, int bits, int block);

/*
 * gptq_quantize_layer: the GPTQ column sweep of one layer.
 *
 * Source: "tm_gptq_math", "Greedy quantization with error compensation" (quantize one
 * weight, move the still-free weights by the optimal correction), "GPTQ's speedups:
 * fixed order and lazy batches" (one left-to-right column order for all rows; blocks of
 * `block` columns, corrections inside the block applied at once, corrections of later
 * columns deferred to one product per block); "GPTQ Hessian" (row j of U supplies the
 * correction of column j); "GPTQ › Mathematical Details of the Update" (O(d_in) work per
 * column once the factor exists).
 *
 * Grid (the pages define none; this library's reading): per output row i, asymmetric
 * min-max over W's row as given, with 0 inside the range:
 *   x_min = min(0, min_j W_ij), x_max = max(0, max_j W_ij),
 *   scale_i = (x_max - x_min) / (2^bits - 1)  (1 if that is 0),  zero_i = rint(-x_min/scale_i)
 * in fp32.  Dead columns (dead_mask) are set to 0 before the sweep.  For each column j in
 * order, with w the current fp32 working value:
 *   code = clamp(rint(w / scale) + zero, 0, 2^bits - 1)      (IEEE division, ties to even)
 *   q = scale * (code - zero);  e = (w - q) / U_jj
 *   w_k -= e * U_jk for every later column k (inside the block at once, later columns
 *   through the deferred block product).
 *
 *   W          [d_out, ldw] of type `wdtype` (GPTQ_BF16, GPTQ_F16 or GPTQ_F32), not modified.
 *   d_out      >= 1 rows;  d_in >= 1 columns;  ldw >= d_in.
 *   U          [d_in, d_in] fp32 upper factor from gptq_prepare (only the upper triangle
 *              is read).
 *   dead_mask  [d_in] uint8 (nonzero = dead) or NULL.
 *   bits       2, 3, 4 or 8.
 *   block      lazy-batch width B: 1 <= B <= 128 (128 is the pages' value).
 *   qpacked    [d_out, ceil(d_in/32) * bits] uint32 out: row-wise little-endian
 *              bitstream, the code of column c in bits [c*bits, (c+1)*bits) of its row
 *              (bit b of the stream = bit b%32 of word b/32); padding bits are 0.
 *   scale      [d_out] fp32 out;  zero: [d_out] int32 out.
 *   W_hat      [d_out, d_in] fp32 out (scale * (code - zero)), or NULL.
 *   ws         workspace of ws_bytes >= gptq_quantize_workspace_bytes(d_out, d_in, bits,
 *              block); its contents need no initialisation.
 * Asynchronous.  Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED, CUDA.  Non-finite weights
 * are flagged in the workspace; read the flag with gptq_workspace_status.
 */
gptq_status gptq_quantize_layer(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                                int64_t ldw, const float *U, const uint8_t *dead_mask,
                                int bits, int block, uint32_t *qpacked, float *scale,
                                int32_t *zero, float *W_hat, void *ws, size_t ws_bytes,
                                gptq_stream_t stream);

/*
 * GPTQ_MAX_SHARED_LAYERS: most layers one gptq_quantize_layers_shared call takes.
 */
#define GPTQ_MAX_SHARED_LAYERS 64

/*
 * gptq_quantize_shared_workspace_bytes: workspace size gptq_quantize_layers_shared needs
 * for n_layers layers of d_out[i] rows (HOST array) and d_in columns.  0 for bad arguments.
 */
size_t gptq_quantize_shared_workspace_bytes(int n_layers, const int64_t *d_out, int64_t d_in,
                                            int bits, int block);

/*
 * gptq_quantize_layers_shared: the column sweep of several layers that read the same
 * inputs, sharing one U.
 *
 * Source: "GPTQ Hessian" -- H depends on the layer inputs only and every row of W shares
 * it, and the rows are quantized independently of one another.  Layers fed by the same
 * inputs (the query, key and value projections of an attention block; the gate and up
 * projections of an MLP) therefore share H, its damping and U, and their rows can be swept
 * as one stack.  The pages have no multi-layer call; this one avoids concatenating the
 * weights on the caller's side and runs one sweep and one trailing update per block over
 * all rows.
 *
 * Each layer's outputs are exactly those of gptq_quantize_layer on that layer alone (same
 * codes, scales, zeros and W_hat, bit for bit).
 *
 *   n_layers   1 .. GPTQ_MAX_SHARED_LAYERS.
 *   W, wdtype, d_out, ldw, qpacked, scale, zero
 *              HOST arrays of n_layers entries; entry i describes layer i exactly as the
 *              same-named argument of gptq_quantize_layer (the pointers are DEVICE pointers).
 *   W_hat      HOST array of n_layers DEVICE pointers (entries may be NULL), or NULL.
 *   d_in, U, dead_mask, bits, block: shared by all layers, as in gptq_quantize_layer.
 *   ws         workspace of ws_bytes >= gptq_quantize_shared_workspace_bytes(...).
 * The host arrays are read during the call only.  Asynchronous.  Errors: INVALID_ARG,
 * WORKSPACE, UNSUPPORTED, CUDA; non-finite weights are flagged in the workspace
 * (gptq_workspace_status).
 */
gptq_status gptq_quantize_layers_shared(int n_layers, const void *const *W, const int *wdtype,
                                        const int64_t *d_out, const int64_t *ldw, int64_t d_in,
                                        const float *U, const uint8_t *dead_mask, int bits,
                                        int block, uint32_t *const *qpacked,
                                        float *const *scale, int32_t *const *zero,
                                        float *const *W_hat, void *ws, size_t ws_bytes,
                                        gptq_stream_t stream);

/*
 * gptq_recon_error_workspace_bytes: workspace size gptq_recon_error needs.  0 for bad
 * arguments.
 */
size_t gptq_recon_error_workspace_bytes(int xdtype, int64_t d_out, int64_t d_in,
                                        int64_t n_tok);

/*
 * gptq_recon_error: per-row output error of a quantized layer on its inputs,
 *   err[i] = sum_t ( (W_i - W_hat_i) . x_t )^2 ,   W_hat = scale * (code - zero),
 * so that sum_i err[i] = ||W X^T - W_hat X^T||_F^2 with X token-major.
 *
 * Source: "tm_gptq_math", "The reconstruction objective, written out" -- GPTQ minimizes
 * this squared output error, one row at a time, over the calibration inputs.  The codes are
 * read from the packed form gptq_quantize_layer writes, so this is the consumer of the
 * quantized layer; it evaluates the objective on X directly rather than through H.
 *
 *   X          [n_tok, ldx] of xdtype: GPTQ_F16 / GPTQ_BF16 (tensor cores: W - W_hat is
 *              rounded to the same type, fp32 accumulation) or GPTQ_F32 (CUDA cores);
 *              16-byte aligned, ldx * sizeof(elem) a multiple of 16 bytes.
 *   W          [d_out, ldw] of wdtype, the layer's original weights.
 *   qpacked, bits, scale, zero
 *              as written by gptq_quantize_layer for this W (packed rows of
 *              ceil(d_in/32) * bits words).
 *   err        [d_out] fp32 out.
 *   ws         workspace of ws_bytes >= gptq_recon_error_workspace_bytes(...).
 * The row sums are combined in a fixed order: repeated calls give identical results.
 * Asynchronous.  Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED, CUDA.
 */
gptq_status gptq_recon_error(const void *X, int xdtype, int64_t n_tok, int64_t d_in,
                             int64_t ldx, const void *W, int wdtype, int64_t d_out, int64_t ldw,
                             const uint32_t *qpacked, int bits, const float *scale,
                             const int32_t *zero, float *err, void *ws, size_t ws_bytes,
                             gptq_stream_t stream);

/*
 * GPTQ_OBQ_MAX_D_IN: widest layer gptq_quantize_obq takes (its per-row inverse Hessian
 * lives in on-chip shared memory).
 */
#define GPTQ_OBQ_MAX_D_IN 128

/*
 * gptq_quantize_obq_workspace_bytes: workspace size gptq_quantize_obq needs.  0 for bad
 * arguments.
 */
size_t gptq_quantize_obq_workspace_bytes(int64_t d_out, int64_t d_in);

/*
 * gptq_quantize_obq: the greedy-order variant that GPTQ's fixed order replaces.
 *
 * Source: "tm_gptq_math", "Greedy quantization with error compensation" -- per row,
 * quantize next the free weight whose rounding raises the output error least,
 * (w_q - quant(w_q))^2 / [H_F^-1]_qq, and correct the other free weights by
 * -((w_q - quant(w_q)) / [H_F^-1]_qq) H_F^-1[:, q]; "GPTQ › Mathematical Details of the
 * Update" -- remove q from the free set by the rank-one Schur downdate of H_F^-1.  Every
 * row follows its own order, so each row carries its own H_F^-1: O(d_in^3) per row, for
 * small layers.  Costs are compared in fp32; ties go to the lowest column index.
 *
 * Same grid, dead-column handling and outputs as gptq_quantize_layer, plus:
 *   U          [d_in, d_in] fp32 upper factor from gptq_prepare (H^-1 = U^T U is formed
 *              from it).
 *   d_in       1 .. GPTQ_OBQ_MAX_D_IN (else UNSUPPORTED).
 *   order      [d_out, d_in] int32 out, or NULL: row i's columns in the order quantized.
 *   ws         workspace of ws_bytes >= gptq_quantize_obq_workspace_bytes(d_out, d_in).
 * Asynchronous.  Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED, CUDA.
 */
gptq_status gptq_quantize_obq(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                              int64_t ldw, const float *U, const uint8_t *dead_mask, int bits,
                              uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                              int32_t *order, void *ws, size_t ws_bytes, gptq_stream_t stream);

/*
 * GPTQ_NOALLOC_SCRATCH_BYTES: size of the fixed scratch array behind
 * gptq_quantize_layer_noalloc (32 MiB per GPU, from the first call on that GPU until the
 * process exits).  A layer fits when
 * gptq_quantize_workspace_bytes(d_out, d_in, bits, block) <= GPTQ_NOALLOC_SCRATCH_BYTES
 * (for example 1024 x 1024 at 4 bits, B = 128).
 */
#define GPTQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * gptq_quantize_layer_noalloc: gptq_quantize_layer for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for callers that cannot call
 * cudaMalloc: code embedded in a host framework that owns all device memory and forbids
 * allocations while it runs, or code that must not cause the device-wide synchronization
 * an allocation or free can bring.  It computes exactly what gptq_quantize_layer computes,
 * with the same arguments minus the workspace: its scratch is a fixed array inside the
 * library (GPTQ_NOALLOC_SCRATCH_BYTES per GPU), and the call itself allocates nothing.
 *
 *   - Sizes: returns GPTQ_ERR_WORKSPACE, before touching the GPU, when the layer needs more
 *     scratch than GPTQ_NOALLOC_SCRATCH_BYTES; use gptq_quantize_layer with a workspace then.
 *   - First call on a device: looks up the array's device address (once per device, with
 *     that device current).  Under CUDA's default lazy module loading this look-up is also
 *     what loads the library code that holds the array, so the first call reserves the
 *     32 MiB on that device and may synchronize it: make the first call during set-up, and
 *     before any stream capture.  Only the later calls allocate nothing.
 *   - Sharing: every call on a device uses the same array, which keeps the last call's
 *     contents (each call clears what it needs).  Calls whose GPU work overlaps (e.g. on
 *     two unordered streams) race and give wrong results: keep them on one stream.
 *   - Device-side status (non-finite weights; a bounded wait that gave up, after which the
 *     outputs are undefined) is recorded in the shared array: read it with
 *     gptq_noalloc_status after the call.
 * Asynchronous.  Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED, CUDA.
 */
gptq_status gptq_quantize_layer_noalloc(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                                        int64_t ldw, const float *U, const uint8_t *dead_mask,
                                        int bits, int block, uint32_t *qpacked, float *scale,
                                        int32_t *zero, float *W_hat, gptq_stream_t stream);

/*
 * gptq_noalloc_status: synchronize `stream`, then return the device-side status the last
 * gptq_quantize_layer_noalloc on the current device recorded: GPTQ_OK, GPTQ_ERR_NONFINITE
 * (a NaN or Inf in W) or GPTQ_ERR_TIMEOUT (a bounded device wait gave up; the outputs of
 * that call are undefined).  Allocates nothing after the first gptq_quantize_layer_noalloc
 * call on the device (see there).  Errors of its own: CUDA.
 */
gptq_status gptq_noalloc_status(gptq_stream_t stream);

/*
 * gptq_workspace_status: synchronize `stream`, then return the device-side status the
 * last gptq_quantize_layer on workspace `ws` recorded (GPTQ_OK, GPTQ_ERR_NONFINITE or
 * GPTQ_ERR_TIMEOUT).  `ws` must be a workspace that call used.
 */
gptq_status gptq_workspace_status(const void *ws, gptq_stream_t stream);

/*
 * gptq_debug_hessian_lost_stage: test hook of the bounded device waits (the pages have no
 * counterpart; it exists so that the failure path of the tensor-core kernels can be tested
 * without hanging a GPU).
 *
 * Runs the fp16/bf16 tensor-core Hessian exactly as gptq_hessian_accumulate with
 * accumulate = 0 would, except that its TMA producer issues nothing for token stage
 * `lost_stage` (stages are 128 tokens): no copy and no arrival, so the MMA issuer's wait for
 * that stage can never complete.  Every wait of the launch gives up after `wait_ns`
 * nanoseconds of the GPU's global timer, records GPTQ_ERR_TIMEOUT in the status block and
 * returns; the CTA then leaves with no copy or tensor-core operation of its own in flight
 * and its tensor memory freed, so the context stays usable.
 *
 *   X, xdtype, n_tok, d_in, ldx, H
 *              as gptq_hessian_accumulate; xdtype GPTQ_F16 or GPTQ_BF16 with d_in >= 64
 *              and n_tok >= 64 (else UNSUPPORTED).  H is left undefined.
 *   lost_stage 0 <= lost_stage < ceil(n_tok / 128).
 *   wait_ns    1e3 .. 1e10: budget of every wait (the regular calls use 2 s).
 *   status_ws  DEVICE buffer of >= 256 bytes, 256-byte aligned, for the status block.
 * SYNCHRONIZES `stream` and returns the device status: GPTQ_ERR_TIMEOUT when the waits ran
 * out as designed.  Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED, CUDA.
 */
gptq_status gptq_debug_hessian_lost_stage(const void *X, int xdtype, int64_t n_tok,
                                          int64_t d_in, int64_t ldx, float *H,
                                          int64_t lost_stage, uint64_t wait_ns, void *status_ws,
                                          gptq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_GB300_H */
