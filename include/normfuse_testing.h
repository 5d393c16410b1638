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

#ifdef __cplusplus
}
#endif

#endif /* NORMFUSE_TESTING_H */
