// Normalize-from-partials kernels, bf16 I/O.
#include "launch.h"
#include "partials_kernels.cuh"

const void* nf::partials_table_bf16(int kind, int group, int n) {
  return partials_table_impl<nf::bf16>(kind, group, n);
}
