// Pipelined forward kernels, f16 I/O.
#include "tables.cuh"

const void* nf::fwd_bulk_table_f16(int kind, int group, int n) {
  return fwd_bulk_table_impl<nf::f16>(kind, group, n);
}
cudaError_t nf::take_error_fwd_bulk_f16(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
