// Row softmax kernels, f32 I/O.
#include "launch.h"
#include "softmax_kernels.cuh"

const void* nf::softmax_table_f32(int kind, int group, int n) {
  return smx_table_impl<float>(kind, group, n);
}
cudaError_t nf::take_error_softmax_f32(cudaStream_t st, unsigned* out) {
  return take_tu_error(st, out);
}
