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
// whole CTA; unaligned or odd-width rows to the scalar kernel.
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

// Vectors per consumer thread when the 256 consumers of a pipelined CTA
// share one row (rows of more than 256 vectors).
inline int bulk_cta_n(int hidden, int vec_elems) {
  const int V = hidden / vec_elems;
  int n = (V + kConsumerThreads - 1) / kConsumerThreads;
  if (n == 7) n = 8;
  return n < 2 ? 2 : n;
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
#define NF_BULK_CTA_CASES(KERNEL, T)               \
  switch (n) {                                     \
    case 2: return (const void*)KERNEL<T, 2>;      \
    case 3: return (const void*)KERNEL<T, 3>;      \
    case 4: return (const void*)KERNEL<T, 4>;      \
    case 5: return (const void*)KERNEL<T, 5>;      \
    case 6: return (const void*)KERNEL<T, 6>;      \
    case 8: return (const void*)KERNEL<T, 8>;      \
    default: return nullptr;                       \
  }

template <typename T> const void* fwd_fn(const Choice& c, bool bulk) {
  const int n = c.n;
  if (c.kind == 0) {
    if (bulk) {
      if (c.group == 8) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 8) }
      if (c.group == 16) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 16) }
      if (c.group == 32) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 32) }
    } else {
      if (c.group == 8) { NF_WARP_CASES(fwd_warp_kernel, T, 8) }
      if (c.group == 16) { NF_WARP_CASES(fwd_warp_kernel, T, 16) }
      if (c.group == 32) { NF_WARP_CASES(fwd_warp_kernel, T, 32) }
    }
  } else if (c.kind == 1) {
    if (bulk) { NF_BULK_CTA_CASES(fwd_bulk_cta_kernel, T) }
    if (c.group == 128) { NF_CTA_CASES(fwd_cta_kernel, T, 128) }
    if (c.group == 256) { NF_CTA_CASES(fwd_cta_kernel, T, 256) }
    if (c.group == 512) { NF_CTA_CASES(fwd_cta_kernel, T, 512) }
  } else if (c.kind == 2) {
    return (const void*)fwd_scalar_kernel<T>;
  }
  return nullptr;
}

template <typename T> const void* bwd_fn(const Choice& c, bool bulk) {
  const int n = c.n;
  if (c.kind == 0) {
    if (bulk) {
      if (c.group == 8) { NF_WARP_CASES(bwd_bulk_warp_kernel, T, 8) }
      if (c.group == 16) { NF_WARP_CASES(bwd_bulk_warp_kernel, T, 16) }
      if (c.group == 32) { NF_WARP_CASES(bwd_bulk_warp_kernel, T, 32) }
    } else {
      if (c.group == 8) { NF_WARP_CASES(bwd_warp_kernel, T, 8) }
      if (c.group == 16) { NF_WARP_CASES(bwd_warp_kernel, T, 16) }
      if (c.group == 32) { NF_WARP_CASES(bwd_warp_kernel, T, 32) }
    }
  } else if (c.kind == 1) {
    if (bulk) { NF_BULK_CTA_CASES(bwd_bulk_cta_kernel, T) }
    if (c.group == 128) { NF_CTA_CASES(bwd_cta_kernel, T, 128) }
    if (c.group == 256) { NF_CTA_CASES(bwd_cta_kernel, T, 256) }
    if (c.group == 512) { NF_CTA_CASES(bwd_cta_kernel, T, 512) }
  } else if (c.kind == 2) {
    return (const void*)bwd_scalar_kernel<T>;
  }
  return nullptr;
}

// Ring sizing: the slots of one CTA should fill about kRingTarget bytes so
// two pipelined CTAs fit on an SM; never fewer than 2 nor more than 8 slots.
constexpr size_t kRingTarget = 104 * 1024;
constexpr size_t kMaxDynSmem = 200 * 1024;

// Fill in a pipelined plan; false when the ring does not fit. `extra`:
// shared bytes after the ring's barriers (the backward's fp32 weight row).
inline bool fill_bulk(Plan* p, const Choice& c, int64_t rows, int hidden, size_t esize, int n_in,
                      size_t extra) {
  const int tile_rows = c.kind == 0 ? kConsumerWarps * (32 / c.group) : 1;
  const size_t slot = (size_t)n_in * tile_rows * hidden * esize;
  const size_t room = kRingTarget > extra ? kRingTarget - extra : 0;
  int stages = (int)std::min<size_t>(8, std::max<size_t>(2, room / slot));
  size_t smem = (size_t)stages * slot + 2 * stages * sizeof(uint64_t) + extra;
  if (smem > kMaxDynSmem) return false;
  p->bulk = true;
  p->kind = c.kind;
  p->group = c.kind == 0 ? c.group : kConsumerThreads;
  p->n = c.n;
  p->block = kBulkThreads;
  p->smem = smem;
  p->cfg.stages = stages;
  p->cfg.tile_rows = tile_rows;
  p->cfg.num_tiles = (rows + tile_rows - 1) / tile_rows;
  return true;
}

// Fill block, shared memory and the rows one CTA covers per loop step of the
// register or scalar kernels.
inline int64_t fill_shape(Plan* p, const Choice& c, int hidden, bool bwd) {
  p->bulk = false;
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
inline cudaError_t size_grid(Plan* p, int64_t steps) {
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
  p->grid = (int)std::max<int64_t>(1, std::min<int64_t>(steps, (int64_t)per_sm * sms));
  return cudaSuccess;
}

// Plan shared by both directions. n_in: streamed [rows, hidden] inputs.
template <typename T>
cudaError_t make_plan(int64_t rows, int hidden, bool vec, bool bwd, int n_in, Plan* p) {
  Choice c = choose(hidden, Vec<T>::N, vec);
  const bool want_bulk = vec && path_override() != kPathRegisters;
  if (want_bulk) {
    Choice b = c;
    if (c.kind == 1) b.n = bulk_cta_n(hidden, Vec<T>::N);
    const size_t extra = bwd ? (size_t)hidden * sizeof(float) : 0;
    if (fill_bulk(p, b, rows, hidden, sizeof(T), n_in, extra)) {
      p->fn = bwd ? bwd_fn<T>(b, true) : fwd_fn<T>(b, true);
      return size_grid(p, p->cfg.num_tiles);
    }
  }
  p->fn = bwd ? bwd_fn<T>(c, false) : fwd_fn<T>(c, false);
  const int64_t rpc = fill_shape(p, c, hidden, bwd);
  return size_grid(p, (rows + rpc - 1) / rpc);
}

template <typename T>
cudaError_t fwd_plan(int64_t rows, int hidden, bool vec, bool has_residual, Plan* p) {
  return make_plan<T>(rows, hidden, vec, false, has_residual ? 2 : 1, p);
}

// Pipelined kernels take (args, BulkCfg); the others take (args) only.
inline cudaError_t launch_plan(const Plan& p, void* args0, cudaStream_t st) {
  BulkCfg cfg = p.cfg;
  void* args_bulk[] = {args0, &cfg};
  void* args_one[] = {args0};
  return cudaLaunchKernel(p.fn, dim3(p.grid), dim3(p.block), p.bulk ? args_bulk : args_one,
                          p.smem, st);
}

template <typename T> cudaError_t fwd_launch(const FwdArgs& a, const Plan& p, cudaStream_t st) {
  return launch_plan(p, const_cast<FwdArgs*>(&a), st);
}

template <typename T> cudaError_t bwd_plan(int64_t rows, int hidden, bool rms, bool vec, Plan* p) {
  cudaError_t e = make_plan<T>(rows, hidden, vec, true, 2, p);
  p->ws_cols = rms ? hidden : 2 * hidden;
  return e;
}

template <typename T>
cudaError_t bwd_launch(const BwdArgs& a, const Plan& p, float* dgamma, float* dbeta,
                       cudaStream_t st) {
  cudaError_t e = launch_plan(p, const_cast<BwdArgs*>(&a), st);
  if (e != cudaSuccess) return e;
  return launch_bwd_finalize(a.ws, p.grid, p.ws_cols, a.hidden, dgamma, a.rms ? nullptr : dbeta,
                             st);
}

// Read and clear this translation unit's device error word, after `st`.
inline cudaError_t take_tu_error(cudaStream_t st, unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tu_error, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tu_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  *out |= v;
  return e;
}

}  // namespace nf

#define NF_INSTANTIATE_FWD(T, NAME)                                                        \
  template cudaError_t nf::fwd_plan<T>(int64_t, int, bool, bool, nf::Plan*);               \
  template cudaError_t nf::fwd_launch<T>(const nf::FwdArgs&, const nf::Plan&, cudaStream_t); \
  cudaError_t nf::take_error_fwd_##NAME(cudaStream_t st, unsigned* out) {                  \
    return take_tu_error(st, out);                                                         \
  }
#define NF_INSTANTIATE_BWD(T, NAME)                                                        \
  template cudaError_t nf::bwd_plan<T>(int64_t, int, bool, bool, nf::Plan*);               \
  template cudaError_t nf::bwd_launch<T>(const nf::BwdArgs&, const nf::Plan&, float*, float*, \
                                         cudaStream_t);                                    \
  cudaError_t nf::take_error_bwd_##NAME(cudaStream_t st, unsigned* out) {                  \
    return take_tu_error(st, out);                                                         \
  }
