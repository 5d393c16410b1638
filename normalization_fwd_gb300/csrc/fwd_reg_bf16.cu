// Scalar forward kernel (any width and alignment), bf16 I/O.
#include "tables.cuh"

const void* nf::fwd_reg_table_bf16(int kind, int group, int n) {
  return fwd_reg_table_impl<nf::bf16>(kind, group, n);
}
