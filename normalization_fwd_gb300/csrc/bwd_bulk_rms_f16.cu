// Pipelined backward kernels (RMSNorm), f16 I/O.
#include "tables.cuh"

const void* nf::bwd_bulk_rms_table_f16(int kind, int group, int n, bool exact) {
  return bwd_bulk_table_impl<nf::f16, true, false>(kind, group, n, exact);
}
cudaError_t nf::take_error_bwd_bulk_rms_f16(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
