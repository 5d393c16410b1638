// Host-side planning and launching: which kernel runs a call, its grid,
// block and shared memory, and the launch itself. Kernels come from the
// per-family tables of the kernel translation units (tables.cuh).
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "bulk.cuh"
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

// Accumulator floats per thread a pipelined backward may keep without
// spilling (ptxas, 2 CTAs per SM: LayerNorm lane groups spill from 6 vectors
// of 8 per lane, LayerNorm with dbias from 4).
constexpr int kMaxAccFloats = 80;

// A backward lane group whose accumulators (n * VEC floats per reduction:
// dgamma; dbeta for LayerNorm; dbias) would not fit moves to a row group of
// 64 or 128 threads (kind 3), the smallest that fits.
inline Choice bwd_choice(const Choice& c, int hidden, int vec_elems, bool rms, bool dbias) {
  if (c.kind != 0) return c;
  const int n_acc = 1 + (rms ? 0 : 1) + (dbias ? 1 : 0);
  if (c.n * vec_elems * n_acc <= kMaxAccFloats) return c;
  const int V = hidden / vec_elems;
  for (int g : {64, 128}) {
    int n = (V + g - 1) / g;
    if (n == 7) n = 8;
    if (n < 2) n = 2;
    if (n * vec_elems * n_acc <= kMaxAccFloats) return {3, g, n};
  }
  return c;
}

// Vectors per consumer thread when the 256 consumers of a pipelined CTA
// share one row (rows of more than 256 vectors).
inline int bulk_cta_n(int hidden, int vec_elems) {
  const int V = hidden / vec_elems;
  int n = (V + kBulkThreads - 1) / kBulkThreads;
  if (n == 7) n = 8;
  return n < 2 ? 2 : n;
}

// The kernel tables of one dtype.
template <typename T> struct Tables;
#define NF_TABLES(T, NAME)                                                          \
  template <> struct Tables<T> {                                                    \
    static const void* fwd_bulk(int k, int g, int n) { return fwd_bulk_table_##NAME(k, g, n); } \
    static const void* fwd_reg(int k, int g, int n) { return fwd_reg_table_##NAME(k, g, n); }   \
    static const void* bwd_bulk(int k, int g, int n, bool rms, bool dbias) {        \
      if (dbias) return rms ? bwd_bulk_rms_dbias_table_##NAME(k, g, n)              \
                            : bwd_bulk_ln_dbias_table_##NAME(k, g, n);              \
      return rms ? bwd_bulk_rms_table_##NAME(k, g, n) : bwd_bulk_ln_table_##NAME(k, g, n); \
    }                                                                               \
    static const void* bwd_reg(int k, int g, int n) { return bwd_reg_table_##NAME(k, g, n); }   \
    static const void* softmax(int k, int g, int n) { return softmax_table_##NAME(k, g, n); }   \
  };
NF_TABLES(float, f32)
NF_TABLES(bf16, bf16)
NF_TABLES(f16, f16)
#undef NF_TABLES

// Ring sizing: the slots of one CTA should fill about `target` bytes (so two
// or three pipelined CTAs fit on an SM); never fewer than 2 nor more than 8
// slots. The lane-group forward (<= 74 registers) runs three CTAs per SM.
constexpr size_t kRingTarget = 104 * 1024;
constexpr size_t kRingTargetFwdGroup = 68 * 1024;
constexpr size_t kMaxDynSmem = 200 * 1024;
constexpr size_t kRingTargetSmx = 48 * 1024;

// Ring targets may be overridden (in KiB) through NORMFUSE_RING_KB_FWD /
// NORMFUSE_RING_KB_BWD for tuning; read once.
inline size_t ring_target_kb_env(const char* name) {
  const char* e = getenv(name);
  if (e == nullptr) return 0;
  const long v = strtol(e, nullptr, 10);
  return (v >= 16 && v <= 200) ? (size_t)v * 1024 : 0;
}
// three_ctas: kernels built for three CTAs per SM (the lane-group forward)
// get the smaller ring. (For the CTA-per-row RMSNorm backward, 2 CTAs with
// 3 slots measured 167 us at 16384 x 8192 against 176 us for 3 CTAs with 2.)
inline size_t ring_target(bool bwd, bool three_ctas) {
  static const size_t fwd_env = ring_target_kb_env("NORMFUSE_RING_KB_FWD");
  static const size_t bwd_env = ring_target_kb_env("NORMFUSE_RING_KB_BWD");
  if (bwd && bwd_env) return bwd_env;
  if (!bwd && fwd_env) return fwd_env;
  return three_ctas ? kRingTargetFwdGroup : kRingTarget;
}

// Fill in a pipelined plan; false when the ring does not fit. `extra`:
// shared bytes after the ring's barriers (the backward's fp32 weight row).
inline bool fill_bulk(Plan* p, const Choice& c, int64_t rows, int hidden, size_t esize, int n_in,
                      size_t extra, size_t target) {
  const int tile_rows = c.kind == 0 ? kConsumerWarps * (32 / c.group)
                                    : (c.kind == 3 ? kBulkThreads / c.group : 1);
  const size_t slot = (size_t)n_in * tile_rows * hidden * esize;
  const size_t room = target > extra ? target - extra : 0;
  int stages = (int)std::min<size_t>(8, std::max<size_t>(2, room / slot));
  size_t smem = (size_t)stages * slot + ring_aux_bytes(stages) + extra;
  if (smem > kMaxDynSmem) return false;
  p->bulk = true;
  p->kind = c.kind;
  p->group = (c.kind == 0 || c.kind == 3) ? c.group : kBulkThreads;
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
inline int64_t fill_shape(Plan* p, const Choice& c, int hidden, bool bwd, bool dbias) {
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
  p->smem = (size_t)hidden * sizeof(float) * (bwd ? (dbias ? 5 : 4) : 1);
  return 1;
}

// Persistent grid: every CTA resident at once, never more CTAs than row steps.
inline cudaError_t size_grid(Plan* p, int64_t steps) {
  if (p->fn == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = (cudaError_t)allow_dyn_smem(p->fn, p->smem);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = (cudaError_t)device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  e = (cudaError_t)resident_blocks(p->fn, p->block, p->smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  p->grid = (int)std::max<int64_t>(1, std::min<int64_t>(steps, (int64_t)per_sm * sms));
  return cudaSuccess;
}

// Plan shared by both directions. n_in: streamed [rows, hidden] inputs;
// n_params: [hidden] parameter rows the pipelined kernels stage in shared
// memory as fp32.
// Forward: rows straight into registers with one CTA per row tile (kind 4,
// lane groups) or per row (kind 5, rows of more than 256 vectors), the
// default; NORMFUSE_FWD_PATH=ring selects the bulk-copy ring kernels.
inline bool fwd_tile_path() {
  static const bool v = [] {
    const char* e = getenv("NORMFUSE_FWD_PATH");
    return !(e && strcmp(e, "ring") == 0);
  }();
  return v;
}

// Backward rows of more than 256 vectors run from registers with a CTA per
// row (kind 5) when its accumulators (n * VEC floats per reduction: dgamma;
// dbeta for LayerNorm; dbias) and the row's two inputs (8n registers) fit in
// 64 registers' worth (56 for LayerNorm, which also keeps the mean and a
// second row sum live), so the kernel keeps three CTAs per SM without
// spilling; NORMFUSE_BWD_PATH=ring keeps the pipelined kernel for them.
inline bool bwd_reg_cta_path() {
  static const bool v = [] {
    const char* e = getenv("NORMFUSE_BWD_PATH");
    return !(e && strcmp(e, "ring") == 0);
  }();
  return v;
}
inline bool bwd_row_cta_fits(int n, int vec_elems, bool rms, bool dbias) {
  const int acc = n * vec_elems * (1 + (rms ? 0 : 1) + (dbias ? 1 : 0));
  return n <= 4 && acc + 8 * n <= (rms ? 64 : 56);
}

template <typename T>
cudaError_t make_plan(int64_t rows, int hidden, bool vec, bool bwd, bool rms, bool dbias,
                      int n_in, int n_params, Plan* p) {
  Choice c = choose(hidden, Vec<T>::N, vec);
  if (bwd && vec && c.kind == 1 && path_override() != kPathRegisters && bwd_reg_cta_path()) {
    const int n = bulk_cta_n(hidden, Vec<T>::N);
    if (bwd_row_cta_fits(n, Vec<T>::N, rms, dbias)) {
      p->bulk = false;
      p->kind = 5;
      p->group = kBulkThreads;
      p->n = n;
      p->block = kBulkThreads;
      p->smem = 0;
      p->fn = Tables<T>::bwd_bulk(5, kBulkThreads, n, rms, dbias);
      return size_grid(p, rows);
    }
  }
  if (!bwd && vec && c.kind == 1 && path_override() != kPathRegisters && fwd_tile_path()) {
    p->bulk = false;
    p->kind = 5;
    p->group = kBulkThreads;
    p->n = bulk_cta_n(hidden, Vec<T>::N);
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::fwd_bulk(5, kBulkThreads, p->n);
    cudaError_t e = size_grid(p, 1);
    if (e != cudaSuccess) return e;
    if (rows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)rows;
    return cudaSuccess;
  }
  if (!bwd && vec && c.kind == 0 && path_override() != kPathRegisters && fwd_tile_path()) {
    p->bulk = false;
    p->kind = 4;
    p->group = c.group;
    p->n = c.n;
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::fwd_bulk(4, c.group, c.n);
    cudaError_t e = size_grid(p, 1);   // occupancy check and attributes
    if (e != cudaSuccess) return e;
    const int64_t rpc = (int64_t)kConsumerWarps * (32 / c.group);
    const int64_t ctas = (rows + rpc - 1) / rpc;
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)ctas;
    return cudaSuccess;
  }
  bool want_bulk = vec && path_override() != kPathRegisters;
  // The register kernels do not accumulate dbias: in register mode a dbias
  // call takes the scalar kernel when the row fits it, else the pipelined one.
  if (bwd && dbias && vec && !want_bulk) {
    if (hidden <= kMaxHiddenScalar) {
      c = choose(hidden, 1, false);
    } else {
      want_bulk = true;
    }
  }
  if (want_bulk) {
    Choice b = bwd ? bwd_choice(c, hidden, Vec<T>::N, rms, dbias) : c;
    if (c.kind == 1) b.n = bulk_cta_n(hidden, Vec<T>::N);
    // Lane-group and row-group kernels stage the parameter rows in shared
    // memory as fp32; CTA-per-row kernels read them from global memory.
    const size_t extra = (b.kind == 0 || b.kind == 3) ? (size_t)n_params * hidden * sizeof(float) : 0;
    const bool three = !bwd && b.kind == 0 && b.n <= 4;
    const size_t target = ring_target(bwd, three);
    if (fill_bulk(p, b, rows, hidden, sizeof(T), n_in, extra, target)) {
      p->fn = bwd ? Tables<T>::bwd_bulk(b.kind, b.group, b.n, rms, dbias)
                  : Tables<T>::fwd_bulk(b.kind, b.group, b.n);
      return size_grid(p, p->cfg.num_tiles);
    }
  }
  p->fn = bwd ? Tables<T>::bwd_reg(c.kind, c.group, c.n) : Tables<T>::fwd_reg(c.kind, c.group, c.n);
  const int64_t rpc = fill_shape(p, c, hidden, bwd, dbias);
  return size_grid(p, (rows + rpc - 1) / rpc);
}

template <typename T>
cudaError_t fwd_plan(int64_t rows, int hidden, bool vec, bool has_residual, int n_params,
                     Plan* p) {
  return make_plan<T>(rows, hidden, vec, false, false, false, has_residual ? 2 : 1, n_params, p);
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

template <typename T>
cudaError_t bwd_plan(int64_t rows, int hidden, bool rms, bool dbias, bool vec, Plan* p) {
  cudaError_t e = make_plan<T>(rows, hidden, vec, true, rms, dbias, 2, 1, p);
  p->ws_cols = hidden * (1 + (rms ? 0 : 1) + (dbias ? 1 : 0));
  return e;
}

template <typename T>
cudaError_t bwd_launch(const BwdArgs& a, const Plan& p, void* dgamma, void* dbeta, void* dbias,
                       int grad_dtype, cudaStream_t st) {
  cudaError_t e = launch_plan(p, const_cast<BwdArgs*>(&a), st);
  if (e != cudaSuccess) return e;
  return launch_bwd_finalize(a.ws, p.grid, p.ws_cols, a.hidden, !a.rms, dgamma,
                             a.rms ? nullptr : dbeta, a.has_dbias ? dbias : nullptr, grad_dtype,
                             st);
}

// Row softmax: the pipelined kernels for aligned rows (one streamed input, no
// parameter rows), the scalar kernel otherwise. Softmax kernels of up to 4
// vectors per thread are built for three or four CTAs per SM and take a
// 48 KiB ring: at 16384 x 8192 bf16, 3 CTAs x 3 slots ran 90 us against
// 98 us for 2 CTAs x 6 slots; at 576000 x 384 the two were within 2 %.
// Wider rows (more registers, two CTAs per SM) keep the 104 KiB ring.
template <typename T> cudaError_t softmax_plan(int64_t rows, int hidden, bool vec, Plan* p) {
  const Choice c = choose(hidden, Vec<T>::N, vec);
  static const int smx_path = [] {
    const char* e = getenv("NORMFUSE_SMX_PATH");   // "ring": the pipelined kernels
    return (e && strcmp(e, "ring") == 0) ? 1 : 0;
  }();
  if (smx_path == 0 && c.kind == 1) {
    // Rows of more than 256 vectors: one CTA per row from registers.
    p->bulk = false;
    p->kind = 5;
    p->group = kBulkThreads;
    p->n = bulk_cta_n(hidden, Vec<T>::N);
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::softmax(5, kBulkThreads, p->n);
    cudaError_t e = size_grid(p, 1);
    if (e != cudaSuccess) return e;
    if (rows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)rows;
    return cudaSuccess;
  }
  if (smx_path == 0 && c.kind == 0) {
    // Lane groups of up to 4 vectors: rows straight into registers, one CTA
    // per 8 * (32 / lanes) rows, as many CTAs as the rows need.
    p->bulk = false;
    p->kind = 4;
    p->group = c.group;
    p->n = c.n;
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::softmax(4, c.group, c.n);
    cudaError_t e = size_grid(p, 1);   // occupancy check and attributes
    if (e != cudaSuccess) return e;
    const int64_t rpc = (int64_t)kConsumerWarps * (32 / c.group);
    const int64_t ctas = (rows + rpc - 1) / rpc;
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)ctas;
    return cudaSuccess;
  }
  if (c.kind == 0 || c.kind == 1) {
    Choice b = c;
    if (c.kind == 1) b.n = bulk_cta_n(hidden, Vec<T>::N);
    static const size_t env = ring_target_kb_env("NORMFUSE_RING_KB_SMX");
    const size_t target = env ? env : (b.n <= 4 ? kRingTargetSmx : kRingTarget);
    if (fill_bulk(p, b, rows, hidden, sizeof(T), 1, 0, target)) {
      p->fn = Tables<T>::softmax(b.kind, b.group, b.n);
      return size_grid(p, p->cfg.num_tiles);
    }
    return cudaErrorInvalidConfiguration;
  }
  if (c.kind != 2) return cudaErrorInvalidConfiguration;
  p->fn = Tables<T>::softmax(2, 0, 0);
  fill_shape(p, c, hidden, false, false);
  return size_grid(p, rows);
}

cudaError_t softmax_launch(const SmxArgs& a, const Plan& p, cudaStream_t st) {
  return launch_plan(p, const_cast<SmxArgs*>(&a), st);
}

}  // namespace nf

template cudaError_t nf::softmax_plan<float>(int64_t, int, bool, nf::Plan*);
template cudaError_t nf::softmax_plan<nf::bf16>(int64_t, int, bool, nf::Plan*);
template cudaError_t nf::softmax_plan<nf::f16>(int64_t, int, bool, nf::Plan*);
template cudaError_t nf::fwd_plan<float>(int64_t, int, bool, bool, int, nf::Plan*);
template cudaError_t nf::fwd_plan<nf::bf16>(int64_t, int, bool, bool, int, nf::Plan*);
template cudaError_t nf::fwd_plan<nf::f16>(int64_t, int, bool, bool, int, nf::Plan*);
template cudaError_t nf::bwd_plan<float>(int64_t, int, bool, bool, bool, nf::Plan*);
template cudaError_t nf::bwd_plan<nf::bf16>(int64_t, int, bool, bool, bool, nf::Plan*);
template cudaError_t nf::bwd_plan<nf::f16>(int64_t, int, bool, bool, bool, nf::Plan*);
template cudaError_t nf::fwd_launch<float>(const nf::FwdArgs&, const nf::Plan&, cudaStream_t);
template cudaError_t nf::fwd_launch<nf::bf16>(const nf::FwdArgs&, const nf::Plan&, cudaStream_t);
template cudaError_t nf::fwd_launch<nf::f16>(const nf::FwdArgs&, const nf::Plan&, cudaStream_t);
template cudaError_t nf::bwd_launch<float>(const nf::BwdArgs&, const nf::Plan&, void*, void*,
                                           void*, int, cudaStream_t);
template cudaError_t nf::bwd_launch<nf::bf16>(const nf::BwdArgs&, const nf::Plan&, void*, void*,
                                           void*, int, cudaStream_t);
template cudaError_t nf::bwd_launch<nf::f16>(const nf::BwdArgs&, const nf::Plan&, void*, void*,
                                           void*, int, cudaStream_t);
