// Normalize-from-partials kernels, f16 I/O.
#include "launch.h"
#include "partials_kernels.cuh"

const void* nf::partials_table_f16(int kind, int group, int n) {
  return partials_table_impl<nf::f16>(kind, group, n);
}
