/*
 * normfuse: the fused normalization block on one GPU (sm_103a).
 *
 * Forward: bias + residual add, then LayerNorm or RMSNorm over the hidden
 * dimension, with an optional amax of |y| for FP8 scaling, in one pass over
 * HBM. Backward: the per-row dx reduction over the hidden dimension and the
 * dgamma/dbeta reductions over the rows in one persistent kernel, followed by
 * a small deterministic finalize.
 *
 * Conventions shared by every entry point:
 *  - Matrices are row-major and contiguous, [rows, hidden]. gamma, beta and
 *    bias are [hidden] in the I/O dtype. mean and rstd are fp32 [rows].
 *    dgamma and dbeta are fp32 [hidden]. amax is one fp32 scalar.
 *  - Every tensor pointer is a DEVICE pointer on the current device, owned by
 *    the caller; the library never allocates, frees or keeps one. Pointers
 *    must be aligned to their element size. When every matrix/vector pointer
 *    is 16-byte aligned and hidden * sizeof(dtype) is a multiple of 16, the
 *    128-bit vectorised kernels run; otherwise a scalar kernel handles the
 *    call with the same results.
 *  - Outputs must not overlap inputs or each other (ln_softmax_fwd alone
 *    also runs in place).
 *  - Work is enqueued on `stream` (0 = the legacy default stream) and the call
 *    returns without waiting for it. The library calls no allocating CUDA API,
 *    and none that synchronises except ln_device_error().
 *  - Failure: arguments are validated on the host first; a validation failure
 *    returns its status before anything is enqueued and leaves every output
 *    untouched. A CUDA error from an enqueue returns LN_ERR_CUDA; the CUDA
 *    error code is then available from ln_last_cuda_error() on the calling
 *    thread. No entry point aborts, throws or prints.
 *  - Limits: rows >= 0; 1 <= hidden <= LN_MAX_HIDDEN_VEC16 (bf16/fp16) or
 *    LN_MAX_HIDDEN_VEC32 (fp32) on the vectorised path, and
 *    1 <= hidden <= LN_MAX_HIDDEN_SCALAR on the scalar path. Element
 *    offsets are 64-bit: rows * hidden may exceed 2^31 (tensors past 4 GiB).
 *
 * Citations are to the four pages the method comes from: NVIDIA/cutlass
 * discussion 874 (GEMM -> residual add -> LayerNorm), iree-org/iree issue
 * 9139 (LayerNorm as mean, variance and normalize over one read of the input),
 * NVIDIA/Fuser issue 1660 (bias + residual -> LayerNorm -> FP8 amax, with the
 * amax split into a fused partial and a final reduction) and pytorch/pytorch
 * PR 165370 (mixed-order fusion of the norm-backward reductions).
 */
#ifndef NORMFUSE_H
#define NORMFUSE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LN_MAX_HIDDEN_VEC16 16384
#define LN_MAX_HIDDEN_VEC32 8192
#define LN_MAX_HIDDEN_SCALAR 8192

/* Size of the static device scratch array behind ln_bwd_noalloc (16 MiB). */
#define LN_NOALLOC_SCRATCH_BYTES (16u << 20)

typedef enum { LN_F32 = 0, LN_BF16 = 1, LN_F16 = 2 } ln_dtype;
typedef enum { LN_LAYERNORM = 0, LN_RMSNORM = 1 } ln_mode;
typedef enum {
  LN_OK = 0,
  LN_ERR_NULL = 1,        /* a required pointer is NULL */
  LN_ERR_ALIGN = 2,       /* a pointer is not aligned to its element size */
  LN_ERR_SHAPE = 3,       /* rows < 0, hidden out of range */
  LN_ERR_UNSUPPORTED = 4, /* unknown dtype or mode */
  LN_ERR_CUDA = 5,        /* a CUDA call failed; see ln_last_cuda_error() */
  LN_ERR_WORKSPACE = 6,   /* backward workspace missing, misaligned or too small */
  LN_ERR_INVALID = 7,     /* eps negative or not finite; outputs overlap inputs */
  LN_ERR_SCRATCH_LIMIT = 8 /* ln_bwd_noalloc: the shape needs more scratch than
                              LN_NOALLOC_SCRATCH_BYTES */
} ln_status;

/*
 * ln_fwd: out_sum = (x + bias) + residual; y = norm(out_sum) * w + beta;
 * amax = max |y|.
 *
 * Defined by the forward snippet of NVIDIA/Fuser issue 1660 (bias and
 * residual add, w = gamma or 1 + gamma, layer_norm, amax of |y| written into
 * a preallocated scalar) and by iree-org/iree issue 9139 (mean, variance and
 * normalize over a single read of the input; bias and skip operands optional).
 * RMSNorm, named on pytorch/pytorch PR 165370, is y = s * rstd * w with
 * rstd = 1/sqrt(mean(s^2) + eps).
 *
 * Per row, in fp32 arithmetic:
 *   s      = (x + bias) + residual, stored to out_sum rounded to dtype;
 *   the statistics are taken from the stored (rounded) sum:
 *   LayerNorm: mean = sum(s)/H, var = sum((s - mean)^2)/H (biased),
 *              rstd = 1/sqrt(var + eps), y = (s - mean) * rstd * w + beta;
 *   RMSNorm:   rstd = 1/sqrt(sum(s^2)/H + eps), y = s * rstd * w;
 *   w = gamma, or 1 + gamma (formed in fp32) when zero_centered_gamma != 0;
 *   y is rounded to dtype; amax = max over all stored y of |y| (exact).
 *
 * x         [rows, hidden] dtype, required.
 * bias      [hidden] dtype, NULL = no bias.
 * residual  [rows, hidden] dtype, NULL = no residual.
 * gamma     [hidden] dtype, required.
 * beta      [hidden] dtype, NULL = 0; ignored for RMSNorm.
 * eps       >= 0 and finite.
 * out_sum   [rows, hidden] dtype, NULL = not stored (the backward needs it
 *           whenever bias or residual is given).
 * y         [rows, hidden] dtype, required.
 * mean      [rows] fp32, NULL = not stored; ignored for RMSNorm.
 * rstd      [rows] fp32, NULL = not stored.
 * amax      one fp32, NULL = not computed. When given it is overwritten
 *           (set to 0 on `stream`, then maxed into), not accumulated.
 */
ln_status ln_fwd(const void* x, const void* bias, const void* residual,
                 const void* gamma, const void* beta, float eps, ln_mode mode,
                 int zero_centered_gamma, void* out_sum, void* y, float* mean,
                 float* rstd, float* amax, cudaStream_t stream, int64_t rows,
                 int64_t hidden, ln_dtype dtype);

/*
 * ln_fwd_ex: ln_fwd plus an FP8 (E4M3) copy of y.
 *
 * NVIDIA/Fuser issue 1660 computes the amax of |y| to scale y for an FP8
 * cast; the pages stop at the amax. This entry point also writes that cast,
 * with a per-tensor scale the caller provides (delayed scaling: typically
 * 448 / an amax from an earlier step). Per element:
 *   y_fp8 = E4M3(round_fp32(y_stored * scale)), round to nearest even,
 *   finite values beyond +-448 saturate to +-448 (no infinities in E4M3);
 * y_stored is y rounded to dtype (what y holds), so y_fp8 is the FP8 cast of
 * the stored y. amax is that of y_stored, as in ln_fwd.
 *
 * y_fp8      [rows, hidden] bytes (E4M3 codes), NULL = not written.
 * fp8_scale  one fp32 on the device, required when y_fp8 is given.
 * y          may be NULL when y_fp8 is given (only the FP8 copy is written).
 * Every other argument and the errors are those of ln_fwd; y_fp8 counts as a
 * tensor pointer for the 16-byte alignment of the vectorised path.
 */
ln_status ln_fwd_ex(const void* x, const void* bias, const void* residual,
                    const void* gamma, const void* beta, float eps, ln_mode mode,
                    int zero_centered_gamma, void* out_sum, void* y, float* mean,
                    float* rstd, float* amax, void* y_fp8, const float* fp8_scale,
                    cudaStream_t stream, int64_t rows, int64_t hidden,
                    ln_dtype dtype);

/* Form of the per-tile partial statistics ln_fwd_from_partials reads. */
typedef enum {
  LN_PARTIALS_SUM_SQ = 0, /* psum = sum of the tile's values, psq = sum of their squares */
  LN_PARTIALS_SUM_M2 = 1  /* psum as above, psq = sum of squares about the tile's own mean */
} ln_partials;

/*
 * ln_fwd_from_partials: y = norm(x) * w + beta with the row statistics
 * combined from per-column-tile partial sums instead of a pass over the row.
 *
 * Defined by NVIDIA/cutlass discussion 874 (the reply pointing at example
 * 37, gemm_with_layernorm.h): the GEMM that produces the row (with the
 * residual added in its epilogue) also sums each row over the column tile
 * every threadblock owns, and the LayerNorm that follows combines those
 * partials into the row's mean and variance. The producing GEMM is not part
 * of this library; this is the consumer: one read of x, one write of y.
 *
 * Column tiles are tile_cols wide from column 0; the last one holds the
 * hidden - (n_tiles - 1) * tile_cols columns left, n_tiles =
 * ceil(hidden / tile_cols). With S and Q the per-row sums over the tiles of
 * psum and of the second quantity, and n_t a tile's width, in fp32:
 *   LN_PARTIALS_SUM_SQ: LayerNorm mean = S / H, var = max(Q / H - mean^2, 0)
 *     (Q = sum psq); RMSNorm mean square = Q / H.
 *   LN_PARTIALS_SUM_M2: LayerNorm var = (sum_t psq_t +
 *     sum_t (psum_t - n_t mean)^2 / n_t) / H (the parallel-variance
 *     identity); RMSNorm mean square = sum_t (psq_t + psum_t^2 / n_t) / H.
 *   rstd = 1/sqrt(var or mean square + eps); y = (x - mean) * rstd * w + beta
 *   (RMSNorm: x * rstd * w), w = gamma or 1 + gamma; y rounded to dtype;
 *   amax = max |y| over the stored y, as in ln_fwd.
 * The sum-of-squares form loses precision when |mean| is large against the
 * row's spread (Q / H and mean^2 cancel); the M2 form does not.
 *
 * x          [rows, hidden] dtype, the stored row (what the producer wrote),
 *            required when rows > 0.
 * psum, psq  [rows, n_tiles] fp32, row-major, 4-byte aligned, required when
 *            rows > 0.
 * n_tiles    must equal ceil(hidden / tile_cols), else LN_ERR_SHAPE.
 * tile_cols  >= 1 (a value >= hidden means one tile).
 * kind       LN_PARTIALS_SUM_SQ or LN_PARTIALS_SUM_M2, else LN_ERR_UNSUPPORTED.
 * gamma, beta, eps, mode, zero_centered_gamma, y, mean, rstd, amax: as in
 *            ln_fwd (mean, rstd are the statistics used, rounded to fp32).
 * Shapes, alignment, limits, streams and errors: the header's conventions.
 */
ln_status ln_fwd_from_partials(const void* x, const float* psum, const float* psq,
                               int64_t n_tiles, int64_t tile_cols, ln_partials kind,
                               const void* gamma, const void* beta, float eps,
                               ln_mode mode, int zero_centered_gamma, void* y,
                               float* mean, float* rstd, float* amax,
                               cudaStream_t stream, int64_t rows, int64_t hidden,
                               ln_dtype dtype);

/*
 * ln_bwd: dx, dgamma, dbeta of the normalization given dy and the forward's
 * saved sum and statistics.
 *
 * Defined by pytorch/pytorch PR 165370: the dx reduction runs over the hidden
 * dimension, the dgamma/dbeta reductions over the rows, and both share dy,
 * x_sum and the statistics, so one persistent kernel loads each input once,
 * keeps per-CTA partial sums of the row reduction (the PR's partial
 * accumulation) and a finalize adds the partials. Per row, in fp32:
 *   xhat = (x_sum - mean) * rstd   (RMSNorm: x_sum * rstd);  g = dy * w;
 *   c1 = sum(g)/H (LayerNorm only); c2 = sum(g * xhat)/H;
 *   dx = rstd * (g - c1 - xhat * c2)   (RMSNorm: no c1), rounded to dtype;
 *   dgamma = sum over rows of dy * xhat; dbeta = sum over rows of dy.
 * dx is also the gradient of the residual and of x through the identity add.
 * dgamma and dbeta are bitwise reproducible from run to run on the same GPU
 * model: the row-to-CTA assignment depends only on the SM count and the
 * finalize adds the partials in a fixed order (compensated fp32 sums, exact
 * up to the rounding of the compensation term, rounded once at the end).
 *
 * dy, x_sum [rows, hidden] dtype, required (x_sum is the forward's out_sum,
 *           or x itself when the forward had neither bias nor residual).
 * gamma     [hidden] dtype, required; w = gamma or 1 + gamma as in ln_fwd.
 * mean      [rows] fp32, required for LayerNorm, ignored for RMSNorm.
 * rstd      [rows] fp32, required.
 * dx        [rows, hidden] dtype, required.
 * dgamma    [hidden] fp32, required, overwritten.
 * dbeta     [hidden] fp32, NULL = not computed; ignored for RMSNorm.
 * workspace device scratch of at least ln_bwd_workspace_bytes() bytes,
 *           16-byte aligned, owned by the caller; may be NULL only when
 *           rows == 0. Its contents need no initialisation and are not
 *           meaningful after the call. Calls that share one workspace must
 *           not run concurrently.
 */
ln_status ln_bwd(const void* dy, const void* x_sum, const void* gamma,
                 const float* mean, const float* rstd, void* dx, float* dgamma,
                 float* dbeta, cudaStream_t stream, int64_t rows,
                 int64_t hidden, ln_dtype dtype, ln_mode mode,
                 int zero_centered_gamma, void* workspace,
                 size_t workspace_bytes);

/*
 * ln_bwd_ex: ln_bwd plus the gradient of the forward's bias, and a choice
 * of precision for the parameter gradients.
 *
 * The forward adds `bias` to every row before the norm (NVIDIA/Fuser issue
 * 1660), so dbias = sum over rows of dx, the gradient of the norm's input;
 * the gradients of x and of residual are dx itself (identity add). dbias is
 * a third column reduction over the rows, accumulated in the same persistent
 * kernel from the fp32 dx (before its rounding to dtype) and added up by the
 * same fixed-order finalize (pytorch/pytorch PR 165370's partial
 * accumulation of the outer reductions).
 *
 * dbias     [hidden] grad_dtype, NULL = not computed.
 * grad_dtype  the type of dgamma, dbeta and dbias: LN_F32 (as in ln_bwd), or
 *           LN_BF16 / LN_F16 for the low-precision epilogue PR 165370 names
 *           (a down cast after the outer reduction): the fixed-order
 *           compensated total of each column is rounded once, to nearest
 *           even, to that type. dgamma/dbeta/dbias must then be aligned to its size.
 * With dbias NULL and grad_dtype LN_F32 this is ln_bwd. Every other
 * argument, the workspace rule and the errors are those of ln_bwd;
 * ln_bwd_workspace_bytes() covers both entry points.
 */
ln_status ln_bwd_ex(const void* dy, const void* x_sum, const void* gamma,
                    const float* mean, const float* rstd, void* dx,
                    void* dgamma, void* dbeta, void* dbias,
                    cudaStream_t stream, int64_t rows, int64_t hidden,
                    ln_dtype dtype, ln_mode mode, int zero_centered_gamma,
                    void* workspace, size_t workspace_bytes,
                    ln_dtype grad_dtype);

/*
 * Bytes of workspace ln_bwd / ln_bwd_ex need for this shape on the current
 * device (the maximum over the vectorised and the scalar kernel and over
 * the layouts with and without dbias, so it holds whatever the pointers'
 * alignment). Queries device attributes; returns LN_ERR_CUDA when no device
 * is usable.
 */
ln_status ln_bwd_workspace_bytes(int64_t rows, int64_t hidden, ln_dtype dtype,
                                 ln_mode mode, size_t* bytes);

/*
 * ln_bwd_noalloc: ln_bwd for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that must not call cudaMalloc or any allocator around a backward pass: a
 * framework that owns every device allocation through its own caching pool
 * (a raw cudaMalloc behind its back fragments the pool and escapes its
 * accounting), a runtime whose device memory budget is fixed up front, and a
 * hot path where an allocation is not allowed because cudaMalloc may
 * synchronise the device. It computes exactly what ln_bwd
 * computes, with the same kernels, arguments and results; the difference is
 * that the per-CTA dgamma/dbeta partials go to a static device array of
 * LN_NOALLOC_SCRATCH_BYTES inside the library instead of a caller workspace.
 *
 * - The array belongs to the library's device code: a context holds its
 *   bytes from the moment the library's module is loaded in it until the
 *   context is destroyed. Under lazy module loading (the CUDA default) that
 *   is the first call of this entry point in the context, so that first call
 *   commits the array; make it before any stream capture and before any
 *   phase with a fixed memory budget. Later calls allocate and free nothing.
 * - Set-up: every call looks up the array's device address in the current
 *   context (the caller's device current), a host-side query that enqueues
 *   nothing; an address is never reused across contexts, so a
 *   cudaDeviceReset or a context of the caller's own is handled.
 * - Limit: shapes whose partials need more than LN_NOALLOC_SCRATCH_BYTES
 *   return LN_ERR_SCRATCH_LIMIT before anything is enqueued
 *   (ln_bwd_workspace_bytes() gives a bound of the need: it also covers
 *   ln_bwd_ex's dbias columns, which this entry point does not compute).
 *   The backward keeps one to three partial rows per SM for 16-byte
 *   aligned rows (one for rows wider than 4096 16-bit elements), so on a
 *   152-SM GB300 aligned LayerNorm rows fit up to about 13,700 elements
 *   and RMSNorm rows up to the 16,384 maximum.
 * - Every call on a device shares the one array and nothing in it needs to
 *   start at zero (each call overwrites the partials it reads). Calls whose
 *   execution overlaps on the GPU (different streams, or different host
 *   threads) race on the array; serialise them, e.g. on one stream.
 * - Other arguments, errors and results: as ln_bwd.
 */
ln_status ln_bwd_noalloc(const void* dy, const void* x_sum, const void* gamma,
                         const float* mean, const float* rstd, void* dx,
                         float* dgamma, float* dbeta, cudaStream_t stream,
                         int64_t rows, int64_t hidden, ln_dtype dtype,
                         ln_mode mode, int zero_centered_gamma);

/*
 * ln_softmax_fwd: row softmax, y[r, :] = exp(x[r, :] - m_r) / s_r with
 * m_r = max_j x[r, j] and s_r = sum_j exp(x[r, j] - m_r).
 *
 * Defined by iree-org/iree issue 9139 (the softmax IR: a max reduction, the
 * exponential of the shifted row, a sum reduction and a division, fused into
 * one dispatch). The ln_ prefix is the library's; this call has nothing to do
 * with a normalization's parameters. Each row is read from HBM once and
 * written once; the max, exponentials, sum and reciprocal are fp32, and y is
 * rounded to dtype. A row that is all -inf, or holds a NaN or +inf, gives NaN
 * in every column, as the definition does; -inf entries of an otherwise
 * finite row give exactly 0 (masking).
 *
 * x, y  [rows, hidden] dtype, device, required when rows > 0. y == x (in
 *       place) is allowed; any other overlap returns LN_ERR_INVALID.
 * Shapes, alignment, limits, streams and errors are those of the header's
 * conventions (no statistics or parameters are involved).
 */
ln_status ln_softmax_fwd(const void* x, void* y, cudaStream_t stream, int64_t rows,
                         int64_t hidden, ln_dtype dtype);

/* Static, human-readable name of a status code. */
const char* ln_status_string(ln_status status);

/* The cudaError_t behind the last LN_ERR_CUDA on the calling thread. */
int ln_last_cuda_error(void);

/*
 * Device-side failure report. The pipelined kernels wait on shared-memory
 * barriers for their bulk copies; every such wait gives up after one second,
 * sets a bit in a device error word and lets the kernel finish early (its
 * outputs are then not valid). This call waits for `stream`, ORs the error
 * words of all kernels into *flags (bit 0: a wait timed out) and clears them.
 * It synchronises `stream`; 0 in *flags means no kernel reported a failure.
 */
ln_status ln_device_error(cudaStream_t stream, unsigned* flags);

#ifdef __cplusplus
}
#endif

#endif /* NORMFUSE_H */
