// Normalize-from-partials kernels, f32 I/O.
#include "launch.h"
#include "partials_kernels.cuh"

const void* nf::partials_table_f32(int kind, int group, int n) {
  return partials_table_impl<float>(kind, group, n);
}
