// Scalar backward kernel (any width and alignment), bf16 I/O.
#include "tables.cuh"

const void* nf::bwd_reg_table_bf16(int kind, int group, int n) {
  return bwd_reg_table_impl<nf::bf16>(kind, group, n);
}
