// Second stage of the backward's outer reductions: adds the per-CTA
// dgamma/dbeta partials in a fixed order (pytorch/pytorch PR 165370, the
// epilogue that follows the converted outer reduction).
#include "launch.h"

namespace nf {

constexpr int kFinCols = 8;      // columns per block: one 32-byte sector of a partial row
constexpr int kFinSlices = 128;  // partial rows are dealt round-robin to this many slices

// dgamma[j] = sum_p ws[p][j] (and likewise dbeta, dbias from their column
// ranges) over the P CTA partials, in a fixed order that depends only on P:
// partial row p goes to slice p % 128; each slice is summed in increasing p;
// then slices 32q .. 32q + 31 are summed in increasing order for q = 0..3, and
// the four results in increasing q. All sums are fp64.
//
// The totals are written as fp32, or (out_dtype 1 / 2) rounded once from
// fp64 to bf16 / fp16: the low-precision epilogue of the outer reductions.
//
// Block (8, 128): thread (x, y) owns column blockIdx.x * 8 + x and slice y,
// so one warp reads four partial rows of 8 consecutive columns (four full
// 32-byte sectors) and every thread has only ceil(P / 128) loads to wait for.
__global__ void __launch_bounds__(kFinCols* kFinSlices)
    bwd_finalize_kernel(const float* __restrict__ ws, int P, int C, int H, int beta_cols,
                        void* dgamma, void* dbeta, void* dbias, int out_dtype) {
  __shared__ double part[kFinSlices][kFinCols];
  __shared__ double quarter[4][kFinCols];
  const int x = threadIdx.x, y = threadIdx.y;
  const int c = blockIdx.x * kFinCols + x;
  double acc = 0.0;
  if (c < C) {
#pragma unroll 4
    for (int p = y; p < P; p += kFinSlices) acc += (double)ws[(int64_t)p * C + c];
  }
  part[y][x] = acc;
  __syncthreads();
  if (y < 4) {
    double t = 0.0;
#pragma unroll 8
    for (int i = 0; i < 32; ++i) t += part[32 * y + i][x];
    quarter[y][x] = t;
  }
  __syncthreads();
  if (y == 0 && c < C) {
    const double t = ((quarter[0][x] + quarter[1][x]) + quarter[2][x]) + quarter[3][x];
    void* out = nullptr;
    int j = 0;
    if (c < H) {
      out = dgamma;
      j = c;
    } else if (beta_cols && c < 2 * H) {
      out = dbeta;
      j = c - H;
    } else {
      out = dbias;
      j = c - (C - H);
    }
    if (out != nullptr) {
      if (out_dtype == 1) {
        static_cast<bf16*>(out)[j] = __double2bfloat16(t);
      } else if (out_dtype == 2) {
        static_cast<f16*>(out)[j] = __double2half(t);
      } else {
        static_cast<float*>(out)[j] = (float)t;
      }
    }
  }
}

cudaError_t launch_bwd_finalize(const float* ws, int P, int C, int H, bool beta_cols,
                                void* dgamma, void* dbeta, void* dbias, int out_dtype,
                                cudaStream_t st) {
  bwd_finalize_kernel<<<(C + kFinCols - 1) / kFinCols, dim3(kFinCols, kFinSlices), 0, st>>>(
      ws, P, C, H, beta_cols ? 1 : 0, dgamma, dbeta, dbias, out_dtype);
  return cudaGetLastError();
}

}  // namespace nf
