// Kernel tables: (family, lanes or threads, vectors per thread) -> kernel.
// Included by the kernel translation units, each of which instantiates one
// family for one dtype (so the instantiations compile in parallel) and
// exposes it through a plain function declared in launch.h.
#pragma once

#include "bwd_kernels.cuh"
#include "fwd_kernels.cuh"
#include "launch.h"

namespace nf {

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
#define NF_BULK_WARP_CASES_M(KERNEL, T, L, M, B, E)      \
  switch (n) {                                           \
    case 1: return (const void*)KERNEL<T, L, 1, M, B, E>; \
    case 2: return (const void*)KERNEL<T, L, 2, M, B, E>; \
    case 3: return (const void*)KERNEL<T, L, 3, M, B, E>; \
    case 4: return (const void*)KERNEL<T, L, 4, M, B, E>; \
    case 5: return (const void*)KERNEL<T, L, 5, M, B, E>; \
    case 6: return (const void*)KERNEL<T, L, 6, M, B, E>; \
    case 8: return (const void*)KERNEL<T, L, 8, M, B, E>; \
    default: return nullptr;                             \
  }
#define NF_BULK_CTA_CASES_M(KERNEL, T, M, B)          \
  switch (n) {                                        \
    case 2: return (const void*)KERNEL<T, 2, M, B>;   \
    case 3: return (const void*)KERNEL<T, 3, M, B>;   \
    case 4: return (const void*)KERNEL<T, 4, M, B>;   \
    case 5: return (const void*)KERNEL<T, 5, M, B>;   \
    case 6: return (const void*)KERNEL<T, 6, M, B>;   \
    case 8: return (const void*)KERNEL<T, 8, M, B>;   \
    default: return nullptr;                          \
  }
#define NF_BULK_GROUP_CASES_M(KERNEL, T, G, M, B)     \
  switch (n) {                                        \
    case 2: return (const void*)KERNEL<T, G, 2, M, B>; \
    case 3: return (const void*)KERNEL<T, G, 3, M, B>; \
    case 4: return (const void*)KERNEL<T, G, 4, M, B>; \
    case 5: return (const void*)KERNEL<T, G, 5, M, B>; \
    case 6: return (const void*)KERNEL<T, G, 6, M, B>; \
    case 8: return (const void*)KERNEL<T, G, 8, M, B>; \
    default: return nullptr;                          \
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

template <typename T> const void* fwd_bulk_table_impl(int kind, int group, int n) {
  if (kind == 0) {
    if (group == 8) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 8) }
    if (group == 16) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 16) }
    if (group == 32) { NF_WARP_CASES(fwd_bulk_warp_kernel, T, 32) }
  } else if (kind == 5) {
    NF_BULK_CTA_CASES(fwd_tile_cta_kernel, T)
  } else if (kind == 4) {
    if (group == 8) { NF_WARP_CASES(fwd_tile_kernel, T, 8) }
    if (group == 16) { NF_WARP_CASES(fwd_tile_kernel, T, 16) }
    if (group == 32) { NF_WARP_CASES(fwd_tile_kernel, T, 32) }
  } else if (kind == 1) {
    NF_BULK_CTA_CASES(fwd_bulk_cta_kernel, T)
  }
  return nullptr;
}

// The scalar forward (any width and alignment); `group` and `n` are unused.
template <typename T> const void* fwd_reg_table_impl(int kind, int group, int n) {
  (void)group;
  (void)n;
  return kind == 2 ? (const void*)fwd_scalar_kernel<T> : nullptr;
}

// exact (lane groups only): the row has exactly group * n vectors.
template <typename T, bool kRms, bool kBias>
const void* bwd_bulk_table_impl(int kind, int group, int n, bool exact) {
  if (kind == 0 && exact) {
    if (group == 8) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 8, kRms, kBias, true) }
    if (group == 16) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 16, kRms, kBias, true) }
    if (group == 32) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 32, kRms, kBias, true) }
  } else if (kind == 0) {
    if (group == 8) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 8, kRms, kBias, false) }
    if (group == 16) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 16, kRms, kBias, false) }
    if (group == 32) { NF_BULK_WARP_CASES_M(bwd_bulk_warp_kernel, T, 32, kRms, kBias, false) }
  } else if (kind == 1) {
    NF_BULK_CTA_CASES_M(bwd_bulk_cta_kernel, T, kRms, kBias)
  } else if (kind == 3) {
    if (group == 64) { NF_BULK_GROUP_CASES_M(bwd_bulk_group_kernel, T, 64, kRms, kBias) }
    if (group == 128) { NF_BULK_GROUP_CASES_M(bwd_bulk_group_kernel, T, 128, kRms, kBias) }
  } else if (kind == 5) {
    switch (n) {
      case 2: return (const void*)bwd_row_cta_kernel<T, 2, kRms, kBias>;
      case 3: return (const void*)bwd_row_cta_kernel<T, 3, kRms, kBias>;
      case 4: return (const void*)bwd_row_cta_kernel<T, 4, kRms, kBias>;
      default: return nullptr;
    }
  } else if (kind >= 6 && kind <= 8 && group > kBulkThreads) {
    // one row group of `group` threads per CTA: 16-bit LayerNorm rows of
    // exactly 1024 vectors at two vectors a thread, rows of more than 1024
    // vectors at four
    if constexpr (!kRms && !kBias && sizeof(T) == 2) {
      if (kind == 7 && group == 512 && n == 2)
        return (const void*)bwd_row_pf_kernel<T, 2, kRms, kBias, 1, 512, 1>;
    }
    if (n != 4) return nullptr;
#define NF_PF_WIDE(GTV)                                                                    \
  if (group == GTV) {                                                                      \
    if constexpr (kRms && !kBias) {                                                        \
      if (kind == 6) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 0, GTV, 1>;  \
    } else if constexpr (!kRms && !kBias) {                                                \
      if (kind == 8) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 2, GTV, 1>;  \
      if constexpr (GTV >= 448) {                                                          \
        if (kind == 7) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 1, GTV, 1>; \
      }                                                                                    \
    } else {                                                                               \
      if (kind == 7) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 1, GTV, 1>;  \
    }                                                                                      \
    return nullptr;                                                                        \
  }
    NF_PF_WIDE(320)
    NF_PF_WIDE(384)
    NF_PF_WIDE(448)
    NF_PF_WIDE(512)
#undef NF_PF_WIDE
  } else if (kind == 6 && (group == 64 || group == 128)) {
    // two 64- or 128-thread row groups (RMSNorm rows of up to 256 or 512 vectors)
    if constexpr (kRms && !kBias) {
      if (group == 64 && n == 3) return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias, 0, 64>;
      if (group == 64 && n == 4) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 0, 64>;
      if (group == 128 && n == 3) return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias, 0, 128>;
      if (group == 128 && n == 4) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 0, 128>;
    }
  } else if (kind == 6) {
    switch (n) {
      case 2: return (const void*)bwd_row_pf_kernel<T, 2, kRms, kBias>;
      case 3: return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias>;
      case 4: return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias>;
      default: return nullptr;
    }
  } else if (kind == 7 && (group == 64 || group == 128)) {
    if constexpr (!kRms || kBias) {
      if (group == 64 && n == 3) return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias, 1, 64>;
      if (group == 128 && n == 3) return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias, 1, 128>;
    }
  } else if (kind == 7) {
    // dbeta / dbias sums in shared memory (RMSNorm without dbias has none)
    if constexpr (!kRms || kBias) {
      if (n == 3) return (const void*)bwd_row_pf_kernel<T, 3, kRms, kBias, 1>;
      if (n == 4) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 1>;
    }
  } else if (kind == 8 && n == 4) {
    // every column sum in shared memory (LayerNorm rows of four vectors)
    if constexpr (!kRms && !kBias) return (const void*)bwd_row_pf_kernel<T, 4, kRms, kBias, 2>;
  }
  return nullptr;
}

// The scalar backward (any width and alignment); `group` and `n` are unused.
template <typename T> const void* bwd_reg_table_impl(int kind, int group, int n) {
  (void)group;
  (void)n;
  return kind == 2 ? (const void*)bwd_scalar_kernel<T> : nullptr;
}

}  // namespace nf
