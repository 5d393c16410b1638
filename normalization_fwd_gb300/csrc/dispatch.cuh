// Kernel selection and launch for one I/O dtype. Included by one translation
// unit per dtype and direction so the instantiations compile in parallel.
#pragma once

#include <algorithm>

#include "bwd_kernels.cuh"
#include "fwd_kernels.cuh"
#include "launch.h"

namespace nf {

// Shape -> kernel family. Rows of up to 256 vectors go to a lane group of a
// warp (exact fit preferred: LANES * N == vectors per row), longer rows to a
// CTA; unaligned or odd-width rows to the scalar kernel.
struct Choice {
  int kind, group, n;
};
inline Choice choose(int hidden, int vec_elems, bool vec) {
  if (!vec) return {2, kScalarCta, 0};
  const int V = hidden / vec_elems;
  if (V <= 256) {
    for (int lanes : {32, 16, 8}) {
      if (V % lanes == 0) {
        const int n = V / lanes;
        if (n <= 8 && n != 7) return {0, lanes, n};
      }
    }
    for (int lanes : {8, 16, 32}) {
      if (lanes * 8 >= V) {
        int n = (V + lanes - 1) / lanes;
        if (n == 7) n = 8;
        return {0, lanes, n};
      }
    }
  }
  for (int threads : {128, 256, 512}) {
    if (threads * 4 >= V) {
      const int n = (V + threads - 1) / threads;
      return {1, threads, n < 3 ? 3 : n};
    }
  }
  return {-1, 0, 0};
}

#define NF_WARP_CASES(KERNEL, T, L)                \
  switch (n) {                                     \
    case 1: return (const void*)KERNEL<T, L, 1>;   \
    case 2: return (const void*)KERNEL<T, L, 2>;   \
    case 3: return (const void*)KERNEL<T, L, 3>;   \
    case 4: return (const void*)KERNEL<T, L, 4>;   \
    case 5: return (const void*)KERNEL<T, L, 5>;   \
    case 6: return (const void*)KERNEL<T, L, 6>;   \
    case 8: return (const void*)KERNEL<T, L, 8>;   \
    default: return nullptr;                       \
  }
#define NF_CTA_CASES(KERNEL, T, TH)                \
  switch (n) {                                     \
    case 3: return (const void*)KERNEL<T, TH, 3>;  \
    case 4: return (const void*)KERNEL<T, TH, 4>;  \
    default: return nullptr;                       \
  }

template <typename T> const void* fwd_fn(const Choice& c) {
  const int n = c.n;
  if (c.kind == 0) {
    if (c.group == 8) { NF_WARP_CASES(fwd_warp_kernel, T, 8) }
    if (c.group == 16) { NF_WARP_CASES(fwd_warp_kernel, T, 16) }
    if (c.group == 32) { NF_WARP_CASES(fwd_warp_kernel, T, 32) }
  } else if (c.kind == 1) {
    if (c.group == 128) { NF_CTA_CASES(fwd_cta_kernel, T, 128) }
    if (c.group == 256) { NF_CTA_CASES(fwd_cta_kernel, T, 256) }
    if (c.group == 512) { NF_CTA_CASES(fwd_cta_kernel, T, 512) }
  } else if (c.kind == 2) {
    return (const void*)fwd_scalar_kernel<T>;
  }
  return nullptr;
}

template <typename T> const void* bwd_fn(const Choice& c) {
  const int n = c.n;
  if (c.kind == 0) {
    if (c.group == 8) { NF_WARP_CASES(bwd_warp_kernel, T, 8) }
    if (c.group == 16) { NF_WARP_CASES(bwd_warp_kernel, T, 16) }
    if (c.group == 32) { NF_WARP_CASES(bwd_warp_kernel, T, 32) }
  } else if (c.kind == 1) {
    if (c.group == 128) { NF_CTA_CASES(bwd_cta_kernel, T, 128) }
    if (c.group == 256) { NF_CTA_CASES(bwd_cta_kernel, T, 256) }
    if (c.group == 512) { NF_CTA_CASES(bwd_cta_kernel, T, 512) }
  } else if (c.kind == 2) {
    return (const void*)bwd_scalar_kernel<T>;
  }
  return nullptr;
}

// Fill block, shared memory and the rows one CTA covers per loop step.
inline int64_t fill_shape(Plan* p, const Choice& c, int hidden, bool bwd) {
  p->kind = c.kind;
  p->group = c.group;
  p->n = c.n;
  if (c.kind == 0) {
    p->block = kWarpCta;
    p->smem = 0;
    return (kWarpCta / 32) * (32 / c.group);
  }
  if (c.kind == 1) {
    p->block = c.group;
    p->smem = 0;
    return 1;
  }
  p->block = kScalarCta;
  p->smem = (size_t)hidden * sizeof(float) * (bwd ? 4 : 1);
  return 1;
}

// Persistent grid: every CTA resident at once, never more CTAs than row steps.
inline cudaError_t size_grid(Plan* p, int64_t rows, int64_t rows_per_cta) {
  if (p->fn == nullptr) return cudaErrorInvalidValue;
  if (p->smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(p->fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p->smem);
    if (e != cudaSuccess) return e;
  }
  int sms = 0, per_sm = 0;
  cudaError_t e = (cudaError_t)device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  e = (cudaError_t)resident_blocks(p->fn, p->block, p->smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t steps = (rows + rows_per_cta - 1) / rows_per_cta;
  p->grid = (int)std::max<int64_t>(1, std::min<int64_t>(steps, (int64_t)per_sm * sms));
  return cudaSuccess;
}

template <typename T> cudaError_t fwd_plan(int64_t rows, int hidden, bool vec, Plan* p) {
  const Choice c = choose(hidden, Vec<T>::N, vec);
  p->fn = fwd_fn<T>(c);
  const int64_t rpc = fill_shape(p, c, hidden, false);
  return size_grid(p, rows, rpc);
}

template <typename T> cudaError_t fwd_launch(const FwdArgs& a, const Plan& p, cudaStream_t st) {
  void* args[] = {const_cast<FwdArgs*>(&a)};
  return cudaLaunchKernel(p.fn, dim3(p.grid), dim3(p.block), args, p.smem, st);
}

template <typename T> cudaError_t bwd_plan(int64_t rows, int hidden, bool rms, bool vec, Plan* p) {
  const Choice c = choose(hidden, Vec<T>::N, vec);
  p->fn = bwd_fn<T>(c);
  const int64_t rpc = fill_shape(p, c, hidden, true);
  p->ws_cols = rms ? hidden : 2 * hidden;
  return size_grid(p, rows, rpc);
}

template <typename T>
cudaError_t bwd_launch(const BwdArgs& a, const Plan& p, float* dgamma, float* dbeta,
                       cudaStream_t st) {
  void* args[] = {const_cast<BwdArgs*>(&a)};
  cudaError_t e = cudaLaunchKernel(p.fn, dim3(p.grid), dim3(p.block), args, p.smem, st);
  if (e != cudaSuccess) return e;
  return launch_bwd_finalize(a.ws, p.grid, p.ws_cols, a.hidden, dgamma, a.rms ? nullptr : dbeta,
                             st);
}

}  // namespace nf

#define NF_INSTANTIATE_FWD(T)                                                              \
  template cudaError_t nf::fwd_plan<T>(int64_t, int, bool, nf::Plan*);                     \
  template cudaError_t nf::fwd_launch<T>(const nf::FwdArgs&, const nf::Plan&, cudaStream_t);
#define NF_INSTANTIATE_BWD(T)                                                              \
  template cudaError_t nf::bwd_plan<T>(int64_t, int, bool, bool, nf::Plan*);               \
  template cudaError_t nf::bwd_launch<T>(const nf::BwdArgs&, const nf::Plan&, float*, float*, \
                                         cudaStream_t);
