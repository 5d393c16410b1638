// Second stage of the backward's outer reductions: adds the per-CTA
// dgamma/dbeta partials in a fixed order (pytorch/pytorch PR 165370, the
// epilogue that follows the converted outer reduction).
#include "launch.h"

namespace nf {

constexpr int kFinCols = 32;    // columns per block: one 128-byte line of a partial row
constexpr int kFinSlices = 32;  // partial rows are dealt round-robin to this many slices

// Error-free sum of two floats (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}

// (s, c) += x, carrying the rounding error of every add in c (compensated
// summation): the pair holds the exact running sum up to the rounding of c.
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
  float e;
  two_sum(s, x, s, e);
  c += e;
}

// dgamma[j] = sum_p ws[p][j] (and likewise dbeta, dbias from their column
// ranges) over the P CTA partials, in an order that depends only on P:
// partial row p goes to slice p % 32, each slice is summed in increasing p,
// and the 32 slices are combined by a fixed pairwise tree (slice y with
// y + 16, then y + 8, ...). Sums are compensated fp32 pairs; the column
// total s + c is formed once in fp64 and rounded once to the output type
// (out_dtype 0 fp32, 1 bf16, 2 fp16). fp64 arithmetic is slow on this part,
// so it is used for that single add only.
//
// Block (32, 32): thread (x, y) owns column blockIdx.x * 32 + x and slice y,
// so a warp reads 128 contiguous bytes of one partial row and every thread
// waits for only ceil(P / 32) independent loads.
__global__ void __launch_bounds__(kFinCols* kFinSlices)
    bwd_finalize_kernel(const float* __restrict__ ws, int P, int C, int H, int beta_cols,
                        void* dgamma, void* dbeta, void* dbias, int out_dtype) {
  __shared__ float ps[kFinSlices][kFinCols + 1];
  __shared__ float pc[kFinSlices][kFinCols + 1];
  // Launched as a programmatic dependent of the backward kernel: wait until
  // that grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int x = threadIdx.x, y = threadIdx.y;
  const int c = blockIdx.x * kFinCols + x;
  float s = 0.f, e = 0.f;
  if (c < C) {
#pragma unroll 8
    for (int p = y; p < P; p += kFinSlices) comp_add(s, e, ws[(int64_t)p * C + c]);
  }
  ps[y][x] = s;
  pc[y][x] = e;
  __syncthreads();
#pragma unroll
  for (int half = kFinSlices / 2; half > 0; half >>= 1) {
    if (y < half) {
      float t, r;
      two_sum(ps[y][x], ps[y + half][x], t, r);
      ps[y][x] = t;
      pc[y][x] = pc[y][x] + pc[y + half][x] + r;
    }
    __syncthreads();
  }
  if (y == 0 && c < C) {
    const double t = (double)ps[0][x] + (double)pc[0][x];   // exact
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
  // Programmatic stream serialization: the finalize may be scheduled while
  // the backward kernel drains; griddepcontrol.wait above orders its reads.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((C + kFinCols - 1) / kFinCols);
  cfg.blockDim = dim3(kFinCols, kFinSlices);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int bc = beta_cols ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, bwd_finalize_kernel, ws, P, C, H, bc, dgamma, dbeta, dbias,
                            out_dtype);
}

}  // namespace nf
