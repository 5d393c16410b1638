// Pipelined backward kernels (RMSNorm, with dbias), bf16 I/O.
#include "tables.cuh"

const void* nf::bwd_bulk_rms_dbias_table_bf16(int kind, int group, int n, bool exact) {
  return bwd_bulk_table_impl<nf::bf16, true, true>(kind, group, n, exact);
}
cudaError_t nf::take_error_bwd_bulk_rms_dbias_bf16(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
