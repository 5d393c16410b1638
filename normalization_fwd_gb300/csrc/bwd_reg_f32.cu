// Scalar backward kernel (any width and alignment), f32 I/O.
#include "tables.cuh"

const void* nf::bwd_reg_table_f32(int kind, int group, int n) {
  return bwd_reg_table_impl<float>(kind, group, n);
}
