/*
 * normfuse testing hook: choose which kernel family the library plans with.
 *
 * Not part of the library's API for computing (include/normfuse.h). The
 * library picks one kernel per shape by itself and reads no environment
 * variable, so what a caller gets depends only on its arguments and the
 * device. For each direction the library also carries the bulk-copy ring
 * kernels (tiles of rows stream into a shared-memory ring by cp.async.bulk),
 * which compute the same operation; this hook lets a test or a benchmark run
 * them instead of the default ones, so that they stay correct. The pages
 * have no counterpart to it.
 *
 * forward, backward, softmax: LN_TESTING_DEFAULT_KERNELS (the kernels the
 *   library picks by shape) or LN_TESTING_RING_KERNELS (the ring kernels for
 *   every 16-byte aligned row of that direction; rows the scalar kernels
 *   take are unchanged).
 * Returns LN_ERR_INVALID for any other value, leaving the choice unchanged.
 * The choice is process-wide and applies to calls planned after it returns;
 * change it only while no other thread calls into the library.
 *
 * ln_testing_plan (below) reports the launch a shape would get.
 */
#ifndef NORMFUSE_TESTING_H
#define NORMFUSE_TESTING_H

#include "normfuse.h"

#ifdef __cplusplus
extern "C" {
#endif

#define LN_TESTING_DEFAULT_KERNELS 0
#define LN_TESTING_RING_KERNELS 1

ln_status ln_testing_select_kernels(int forward, int backward, int softmax);

/*
 * The launch the library would plan for a call of this shape on the current
 * device (16-byte aligned pointers assumed), so that a test can check which
 * kernel layout a width gets. Nothing is launched or allocated.
 *
 * direction: LN_TESTING_PLAN_FORWARD (ln_fwd; option != 0: with a residual),
 *   LN_TESTING_PLAN_BACKWARD (ln_bwd / ln_bwd_ex; option != 0: with dbias),
 *   LN_TESTING_PLAN_SOFTMAX (ln_softmax_fwd; mode ignored),
 *   LN_TESTING_PLAN_PARTIALS (ln_fwd_from_partials; option ignored).
 * out: six ints, caller-owned: kernel kind (0 pipelined lane group, 1
 *   pipelined CTA per row, 2 scalar, 3 pipelined row group, 4 lane group
 *   from registers, 5 CTA per row from registers, 6 prefetching CTA-per-row
 *   backward, 7 and 8 the same with column sums in shared memory), threads
 *   per row (lanes or row group), 16-byte vectors per thread, threads per
 *   CTA, CTAs, dynamic shared-memory bytes.
 * Returns LN_ERR_NULL (out null), LN_ERR_UNSUPPORTED (dtype, mode or
 * direction unknown), LN_ERR_SHAPE (rows < 1, or hidden outside what the
 * entry point accepts), LN_ERR_CUDA (no usable device); out is written only
 * on LN_OK.
 */
#define LN_TESTING_PLAN_FORWARD 0
#define LN_TESTING_PLAN_BACKWARD 1
#define LN_TESTING_PLAN_SOFTMAX 2
#define LN_TESTING_PLAN_PARTIALS 3

ln_status ln_testing_plan(int direction, int64_t rows, int64_t hidden, ln_dtype dtype,
                          ln_mode mode, int option, int* out);

#ifdef __cplusplus
}
#endif

#endif /* NORMFUSE_TESTING_H */
