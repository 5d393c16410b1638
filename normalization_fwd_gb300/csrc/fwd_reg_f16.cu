// Scalar forward kernel (any width and alignment), f16 I/O.
#include "tables.cuh"

const void* nf::fwd_reg_table_f16(int kind, int group, int n) {
  return fwd_reg_table_impl<nf::f16>(kind, group, n);
}
