// Scalar forward kernel (any width and alignment), f32 I/O.
#include "tables.cuh"

const void* nf::fwd_reg_table_f32(int kind, int group, int n) {
  return fwd_reg_table_impl<float>(kind, group, n);
}
