// Second stage of the backward's outer reductions: adds the per-CTA
// dgamma/dbeta partials in a fixed order (pytorch/pytorch PR 165370, the
// epilogue that follows the converted outer reduction).
#include "launch.h"

namespace nf {

// dgamma[j] = sum_p ws[p][j] (and likewise dbeta, dbias from their column
// ranges) over the P CTA partials in a fixed order: CTA row p goes to slice
// p % 32, each slice is summed in increasing p, then the 32 slices in
// increasing order, all in fp64. Block (32, 32): 32 columns per block.
__global__ void __launch_bounds__(1024) bwd_finalize_kernel(const float* __restrict__ ws, int P,
                                                            int C, int H, int beta_cols,
                                                            float* dgamma, float* dbeta,
                                                            float* dbias) {
  __shared__ double part[32][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  double acc = 0.0;
  if (c < C) {
#pragma unroll 4
    for (int p = threadIdx.y; p < P; p += 32) acc += (double)ws[(int64_t)p * C + c];
  }
  part[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && c < C) {
    double t = 0.0;
#pragma unroll
    for (int i = 0; i < 32; ++i) t += part[i][threadIdx.x];
    if (c < H) {
      dgamma[c] = (float)t;
    } else if (beta_cols && c < 2 * H) {
      if (dbeta) dbeta[c - H] = (float)t;
    } else if (dbias) {
      dbias[c - (C - H)] = (float)t;
    }
  }
}

cudaError_t launch_bwd_finalize(const float* ws, int P, int C, int H, bool beta_cols,
                                float* dgamma, float* dbeta, float* dbias, cudaStream_t st) {
  bwd_finalize_kernel<<<(C + 31) / 32, dim3(32, 32), 0, st>>>(ws, P, C, H, beta_cols ? 1 : 0,
                                                               dgamma, dbeta, dbias);
  return cudaGetLastError();
}

}  // namespace nf
