// Pipelined forward kernels, f32 I/O.
#include "tables.cuh"

const void* nf::fwd_bulk_table_f32(int kind, int group, int n) {
  return fwd_bulk_table_impl<float>(kind, group, n);
}
cudaError_t nf::take_error_fwd_bulk_f32(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
