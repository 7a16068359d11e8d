/*
 * gb300norm.h -- C ABI of the GB300 (sm_103a) row-normalisation library
 * libgb300norm.so: RMSNorm, LayerNorm and FusedAddRMSNorm, forward and
 * backward, over an M x N activation matrix.
 *
 * Operations (per row i of M, columns j < N; W'_j = float(w_j) + offset is
 * formed in FP32 inside the kernels, never pre-added in the weight's storage
 * type -- "fix(cutedsl): fuse Gemma RMSNorm weight offset in FP32", Summary):
 *
 *   RMSNorm     rstd = 1/sqrt(mean_j(x_j^2) + eps);  y_j = x_j*rstd*W'_j
 *   LayerNorm   mean = mean_j(x_j); rstd = 1/sqrt(mean_j((x_j-mean)^2) + eps)
 *               y_j = (x_j-mean)*rstd*W'_j + b_j
 *   FusedAdd    h_j = x_j + residual_j;  y = RMSNorm(h);  h is also an output
 *
 * Backward passes compute dx always and the column-reduced dW (and dB) only
 * when the caller passes a non-NULL dw (db) pointer: a NULL pointer selects a
 * kernel instantiation with every weight-gradient instruction, partial buffer
 * and reduction compiled out ("perf(norm): skip dW/dB calculation when
 * parameters are frozen", Motivation and Key Changes).
 *
 * Common conventions
 *   - Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *     owned by the caller.  The library never allocates or frees memory and
 *     never synchronises the host; every call only enqueues kernels on
 *     `stream` (NULL = the legacy default stream) and returns.
 *   - 2-D tensors are row-major with a per-tensor row stride in ELEMENTS
 *     (stride >= N); row i of x starts at x + i*x_stride.
 *   - dtype codes: NORM_F32, NORM_F16, NORM_BF16.  Activations (x, y,
 *     residual, h, dy, dx, dh_out) have type `dtype`; weights and bias have
 *     type `w_dtype`.  Supported (dtype, w_dtype): (F32,F32), (F16,F16),
 *     (BF16,BF16), (BF16,F32), (F16,F32).  All arithmetic is FP32.
 *   - mean / rstd are FP32 arrays of length M (contiguous).
 *   - dW / dB outputs are length-N contiguous arrays of type `dw_dtype`, which
 *     must be NORM_F32 or equal to w_dtype.  They are reduced over all rows in
 *     a fixed order (bit-reproducible run to run).
 *   - A backward with dW or dB needs a caller-provided device workspace of at
 *     least the size norm_bwd_workspace_bytes() reports (16-byte aligned); a
 *     frozen backward (dw = db = NULL) needs none (workspace may be NULL).
 *     The workspace is scratch: the call writes its FP32 partial sums there
 *     and leaves its contents unspecified.  Bytes beyond the reported size
 *     are never touched, and results do not depend on the workspace's
 *     previous contents or on its alignment beyond 16 bytes.
 *   - Aliasing: y may be x, dx may be dy, h_out may be x or residual, and the
 *     fused-add dx may be dy or dh_out, each only with equal row strides.  Any
 *     other overlap between an output and any other argument is undefined.
 *   - M == 0 is a successful no-op (dW/dB, if requested, are set to zero).
 *   - Return value: NORM_OK or an error code.  Argument errors are detected on
 *     the host before anything is enqueued.  NORM_ERR_CUDA reports a CUDA
 *     runtime error returned while querying the device or launching.
 *     Faults that happen later on the device surface at the caller's next
 *     synchronisation, as with any CUDA kernel.
 */
#ifndef GB300NORM_H
#define GB300NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GB300NORM_API __attribute__((visibility("default")))
#else
#define GB300NORM_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *gb300norm_stream_t;

/* Element type codes. */
enum { NORM_F32 = 0, NORM_F16 = 1, NORM_BF16 = 2 };

/* Status codes. */
enum {
    NORM_OK = 0,
    NORM_ERR_NULL = 1,      /* a required pointer is NULL                      */
    NORM_ERR_SHAPE = 2,     /* M < 0, N <= 0 or N > 2^31 - 1                    */
    NORM_ERR_STRIDE = 3,    /* a row stride < N                                 */
    NORM_ERR_DTYPE = 4,     /* unsupported dtype / w_dtype / dw_dtype           */
    NORM_ERR_WORKSPACE = 5, /* workspace NULL, too small or not 16-B aligned    */
    NORM_ERR_ALIGN = 6,     /* a pointer is not aligned to its element size     */
    NORM_ERR_VALUE = 7,     /* eps < 0, or eps / offset not finite              */
    NORM_ERR_ALIAS = 8,     /* an output overlaps an input in a way not allowed */
    NORM_ERR_CUDA = 9,      /* CUDA runtime error while querying or launching   */
    NORM_ERR_ARG = 10,      /* inconsistent optional arguments (see each call)  */
    NORM_ERR_TOO_LARGE = 11 /* problem exceeds the library's fixed scratch      */
};

/* Human-readable name of a status code (static string, never NULL). */
GB300NORM_API const char *norm_status_str(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
GB300NORM_API int norm_version(void);

/*
 * Workspace a backward call needs for its dW / dB partial sums, in bytes, for
 * the current device: *bytes = 0 when has_dw == has_db == 0 (frozen).  The
 * same (M, N, has_dw, has_db) on the same device always gives the same size,
 * and one workspace of that size serves norm_rms_bwd, norm_ln_bwd and
 * norm_fused_add_rms_bwd.  Returns NORM_ERR_NULL if bytes is NULL,
 * NORM_ERR_SHAPE for a bad M / N, NORM_ERR_CUDA if the device cannot be
 * queried.
 */
GB300NORM_API int norm_bwd_workspace_bytes(int64_t M, int64_t N, int has_dw, int has_db,
                             size_t *bytes);

/*
 * RMSNorm forward ("fix(cutedsl): fuse Gemma RMSNorm weight offset in FP32",
 * Summary; offset = 1 gives the Gemma form y = x*rstd*(1 + w)).
 *   x    [M, x_stride]  in    dtype
 *   w    [N]            in    w_dtype
 *   y    [M, y_stride]  out   dtype
 *   rstd [M]            out   FP32, may be NULL (inference)
 */
GB300NORM_API int norm_rms_fwd(const void *x, int64_t x_stride, const void *w,
                 void *y, int64_t y_stride, float *rstd,
                 int64_t M, int64_t N, float offset, float eps,
                 int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * RMSNorm backward ("perf(norm): skip dW/dB calculation when parameters are
 * frozen", Key Changes, rms_norm):
 *   xhat = x*rstd, g = dy*W', c = mean_j(g_j*xhat_j),
 *   dx = rstd*(g - xhat*c),  dw = sum over rows of dy*xhat.
 *   dy   [M, dy_stride] in;  x [M, x_stride] in;  w [N] in
 *   rstd [M] in, FP32 as saved by the forward; NULL = recompute from x, eps
 *   dx   [M, dx_stride] out (may alias dy)
 *   dw   [N] out of type dw_dtype, NULL = frozen weight (no dW work at all)
 *   workspace / workspace_bytes: see norm_bwd_workspace_bytes (unused if
 *   dw is NULL)
 */
GB300NORM_API int norm_rms_bwd(const void *dy, int64_t dy_stride,
                 const void *x, int64_t x_stride,
                 const void *w, const float *rstd,
                 void *dx, int64_t dx_stride,
                 void *dw, int dw_dtype,
                 void *workspace, size_t workspace_bytes,
                 int64_t M, int64_t N, float offset, float eps,
                 int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * LayerNorm forward ("perf(norm): skip dW/dB ...", Key Changes, layer_norm),
 * biased variance.  Never E[x^2] - mean^2: each thread takes sums of its
 * elements about one of them and the block merges them exactly (the
 * pairwise update of Chan, Golub and LeVeque), one pass over the row held on
 * chip.
 *   b may be NULL (no bias); mean and rstd may each be NULL.
 */
GB300NORM_API int norm_ln_fwd(const void *x, int64_t x_stride,
                const void *w, const void *b,
                void *y, int64_t y_stride,
                float *mean, float *rstd,
                int64_t M, int64_t N, float offset, float eps,
                int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * LayerNorm backward ("perf(norm): skip dW/dB ...", Key Changes, layer_norm;
 * dW and dB are independent):
 *   xhat = (x-mean)*rstd, g = dy*W',
 *   dx = rstd*(g - mean_j(g_j) - xhat*mean_j(g_j*xhat_j)),
 *   dw = sum over rows of dy*xhat, db = sum over rows of dy.
 *   mean and rstd must both be given or both be NULL (NULL = recompute from
 *   x and eps; one NULL and one not gives NORM_ERR_ARG).
 *   dw, db: NULL = frozen; both use dw_dtype.
 */
GB300NORM_API int norm_ln_bwd(const void *dy, int64_t dy_stride,
                const void *x, int64_t x_stride,
                const void *w, const float *mean, const float *rstd,
                void *dx, int64_t dx_stride,
                void *dw, void *db, int dw_dtype,
                void *workspace, size_t workspace_bytes,
                int64_t M, int64_t N, float offset, float eps,
                int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * FusedAddRMSNorm forward ("perf(norm): skip dW/dB ...", Key Changes,
 * fused_add_rms_norm; "fix(cutedsl): ...", Summary):
 *   h = x + residual in FP32;  h_out = h rounded to dtype;
 *   y = RMSNorm of the FP32 h with scale W';  rstd saved (may be NULL).
 *   h_out may alias x or residual (vLLM-style in-place residual update).
 */
GB300NORM_API int norm_fused_add_rms_fwd(const void *x, int64_t x_stride,
                           const void *residual, int64_t residual_stride,
                           const void *w,
                           void *y, int64_t y_stride,
                           void *h_out, int64_t h_stride,
                           float *rstd,
                           int64_t M, int64_t N, float offset, float eps,
                           int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * FusedAddRMSNorm backward, at the saved (rounded) h rows ("fix(cutedsl):
 * ...", PyTorch accuracy comparison: the backward uses the rounded saved
 * residual):
 *   dx = RMSNorm-backward(h, dy) + dh_out.  dx is both d(x) and d(residual).
 *   dh_out: gradient arriving on the h output, NULL = zero.
 *   rstd: as saved by the forward, NULL = recompute from h and eps.
 *   dw: NULL = frozen.
 */
GB300NORM_API int norm_fused_add_rms_bwd(const void *dy, int64_t dy_stride,
                           const void *dh_out, int64_t dh_stride,
                           const void *h, int64_t h_stride,
                           const void *w, const float *rstd,
                           void *dx, int64_t dx_stride,
                           void *dw, int dw_dtype,
                           void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, float offset, float eps,
                           int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * norm_rms_bwd_noalloc -- the RMSNorm backward of norm_rms_bwd for callers
 * that cannot allocate device memory (no cudaMalloc where they run: inside an
 * allocator-free runtime, a plugin whose host owns all device memory, or
 * code that must not touch the allocator while a stream is being captured).
 * The pages have no counterpart to this entry point.
 *
 * Same arguments, meaning and results as norm_rms_bwd, without workspace:
 * the dW partial sums go to a fixed scratch array compiled into the library
 * (norm_noalloc_scratch_bytes() bytes, 16 MiB), which every GPU that loads
 * the library holds until the process exits.  A trainable call (dw != NULL)
 * whose partial sums would not fit -- norm_bwd_workspace_bytes(M, N, 1, 0)
 * larger than the scratch -- returns NORM_ERR_TOO_LARGE before anything is
 * enqueued.  The first call on each device looks up the scratch's device
 * address (with that device current) and caches it; make that first call
 * before capturing a stream.  All calls on a device share the scratch, so
 * calls whose kernels may overlap on the GPU (unordered streams) race and
 * give wrong dW; order them on one stream or with events.  Nothing in the
 * scratch has to be cleared: each call writes every value it reads.
 */
GB300NORM_API size_t norm_noalloc_scratch_bytes(void);
GB300NORM_API int norm_rms_bwd_noalloc(const void *dy, int64_t dy_stride,
                                       const void *x, int64_t x_stride,
                                       const void *w, const float *rstd,
                                       void *dx, int64_t dx_stride,
                                       void *dw, int dw_dtype,
                                       int64_t M, int64_t N, float offset, float eps,
                                       int dtype, int w_dtype, gb300norm_stream_t stream);

/*
 * norm_sum_ranks -- the one exchange step of a backward whose rows are
 * sharded over GPUs (M split across ranks): each rank's dW (or dB) is the
 * FP32 column sum of its own rows (a backward call with dw_dtype NORM_F32),
 * and the gradient of the whole problem is their sum over ranks -- the
 * cross-program column reduction of "perf(norm): skip dW/dB calculation when
 * parameters are frozen" (Motivation), taken across GPUs.  After the ranks'
 * vectors have been gathered (e.g. an all-gather) into one device array,
 *   out[j] = ((parts[0*N + j] + parts[1*N + j]) + parts[2*N + j]) + ...
 * added in FP32 in rank order and converted once to out_dtype, so every rank
 * that runs it gets the same bits in every run.
 *   parts: device, FP32, world rows of N contiguous values (4-byte aligned);
 *   out: device, N values of out_dtype (NORM_F32, NORM_F16 or NORM_BF16),
 *        aligned to its element size; must not overlap parts.
 * Both are owned by the caller; the call only reads parts and writes out,
 * asynchronously on `stream`.  Errors, before anything is enqueued:
 * NORM_ERR_SHAPE (world < 1, N <= 0, either above 2^31 - 1), NORM_ERR_NULL,
 * NORM_ERR_DTYPE, NORM_ERR_ALIGN, NORM_ERR_ALIAS; NORM_ERR_CUDA if the launch
 * fails.
 */
GB300NORM_API int norm_sum_ranks(const float *parts, int64_t world, int64_t N, void *out, int out_dtype,
                                 gb300norm_stream_t stream);

/*
 * Device-side status word shared by all kernels of this library on the
 * current device: 0 when no kernel has reported a problem.  A kernel whose
 * bounded wait for an asynchronous row copy runs out sets it (non-zero) and
 * returns early instead of hanging.  While the word is non-zero the outputs
 * of the calls issued since it was last cleared are undefined: rows after
 * the failed wait are not written, and dW / dB are not valid (the CTA that
 * gave up writes no partial sums, but the column reduction still runs).
 * This call synchronises the device; with reset != 0 the word is cleared
 * afterwards.  Returns NORM_OK or NORM_ERR_CUDA; *value receives the word.
 */
GB300NORM_API int norm_device_status(int reset, int *value);

/*
 * The CUDA runtime error code (a cudaError_t value) behind the most recent
 * NORM_ERR_CUDA returned to the calling thread, 0 if there was none, and its
 * text (static string, never NULL).
 */
GB300NORM_API int norm_last_cuda_error(void);
GB300NORM_API const char *norm_cuda_error_string(int code);

/*
 * Test hook: mode 0 (default) lets each call pick its kernel family from the
 * arguments; mode 2 makes every subsequent call in the process use the
 * general (any alignment) row kernels, so tests can compare both families
 * on the same inputs.  Returns NORM_OK or NORM_ERR_ARG.
 */
GB300NORM_API int norm_debug_set_path(int mode);

/*
 * Test hook for launch-shape sweeps: key 1 = 16-byte chunks per thread of the
 * aligned-row kernels (1, 2, 4 or 8), key 2 = maximum CTAs per SM, key 3 =
 * maximum pipeline stages, key 4 = cap on row bytes in flight per SM in
 * units of 16 KB (64 = no cap in practice), key 5 = CTAs per row (1, 2, 4
 * or 8: a thread-block cluster splitting each row into equal column
 * slices; a split that does not divide the row's 16-byte chunks is not
 * used); value 0 restores the automatic choice (values 0..64).  Keys 1-5
 * affect speed only, never results of the same kernel family except through
 * the reduction tree shape.  Key 6 (value 1) is a failure-detection test
 * hook: the aligned-row kernels then issue no copy for each row group's last
 * row, so the bounded wait for it runs out (after 2 s): the kernel sets the
 * device status word (norm_device_status) and returns without writing that
 * row's outputs; every copy it did issue has landed by then.  Returns NORM_OK
 * or NORM_ERR_ARG.
 */
GB300NORM_API int norm_debug_tune(int key, int value);

/*
 * Number of kernels this library has launched (successful launches, on every
 * device and thread) since it was loaded or last reset; with reset != 0 the
 * count is cleared after it is read.  For tests and benchmarks that check how
 * many kernels a call enqueues: one row kernel per forward and per frozen
 * backward, plus the column reduce per trainable backward.
 */
GB300NORM_API int64_t norm_debug_launches(int reset);

#ifdef __cplusplus
}
#endif

#endif /* GB300NORM_H */
