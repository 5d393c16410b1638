// Internal interface between the C entry points (api.cu) and the per-dtype
// translation units that instantiate and launch the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace nf {

// Largest hidden size each path accepts.
constexpr int kMaxVecSlots = 2048;        // 16-byte vectors per row, vector kernels
constexpr int kMaxHiddenScalar = 8192;    // scalar kernels (shared-memory staged)

// Which kernel a call runs and how it is launched.
struct Plan {
  const void* fn = nullptr;
  int kind = -1;       // 0 warp-per-row, 1 CTA-per-row, 2 scalar
  int group = 0;       // lanes per row (kind 0) or threads per CTA (kind 1, 2)
  int n = 0;           // 16-byte vectors per thread per row
  int block = 0;
  size_t smem = 0;
  int grid = 0;        // CTAs; for the backward also the number of partials
  int ws_cols = 0;     // backward: floats per partial row
};

// Per-device facts, cached (api.cu).
int device_sm_count(int* sms);                                  // returns cudaError_t
int resident_blocks(const void* fn, int block, size_t smem, int* out);  // returns cudaError_t

template <typename T> cudaError_t fwd_plan(int64_t rows, int hidden, bool vec, Plan* p);
template <typename T> cudaError_t fwd_launch(const FwdArgs& a, const Plan& p, cudaStream_t st);
template <typename T> cudaError_t bwd_plan(int64_t rows, int hidden, bool rms, bool vec, Plan* p);
template <typename T>
cudaError_t bwd_launch(const BwdArgs& a, const Plan& p, float* dgamma, float* dbeta,
                       cudaStream_t st);

// Fixed-order sum of the backward's per-CTA partials (finalize.cu).
cudaError_t launch_bwd_finalize(const float* ws, int P, int C, int H, float* dgamma,
                                float* dbeta, cudaStream_t st);

}  // namespace nf
