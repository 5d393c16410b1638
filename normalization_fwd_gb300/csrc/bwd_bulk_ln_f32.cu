// Pipelined backward kernels (LayerNorm), f32 I/O.
#include "tables.cuh"

const void* nf::bwd_bulk_ln_table_f32(int kind, int group, int n, bool exact) {
  return bwd_bulk_table_impl<float, false, false>(kind, group, n, exact);
}
cudaError_t nf::take_error_bwd_bulk_ln_f32(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
