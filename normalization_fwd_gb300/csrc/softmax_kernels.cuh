// Row softmax kernels: y[r, :] = exp(x[r, :] - max_j x[r, j]) / sum_j exp(...).
//
// Definition (iree-org/iree issue 9139, the softmax IR and its single
// dispatch form): per row, a max reduction, the exponential of the shifted
// row, a sum reduction, and a division. Like the normalization forward the
// whole row stays on chip between the reductions, so each element is read
// from HBM once and written once.
//
//  * smx_bulk_warp_kernel / smx_bulk_cta_kernel (16-byte aligned rows): tiles
//    of rows stream into a shared-memory ring by cp.async.bulk (the ring and
//    refill scheme of the normalization kernels) and 8 warps work on them
//    from shared memory: a lane group of LANES lanes per row, or all 256
//    threads per row for rows of more than 256 vectors.
//  * smx_scalar_kernel: any hidden size and alignment; element-wise loads,
//    the row staged in shared memory as fp32.
//
// Arithmetic: fp32 throughout. m = max (fmaxf), e = expf(x - m), s = sum of
// e, y = e * (1/s) with a correctly rounded reciprocal. A row whose entries
// are all -inf, or that holds a NaN or +inf, comes out as NaN, as the
// definition gives.
#pragma once

#include <math.h>

#include "bulk.cuh"
#include "common.cuh"

namespace nf {

// One row from shared memory. `G` threads share the row, this one is `t`;
// `xrow` is the shared-memory address of the row. `rmax` / `rsum` reduce a
// float over the G threads.
template <typename T, int G, int N, typename RMax, typename RSum>
__device__ __forceinline__ void smx_row_smem(const SmxArgs& a, int64_t row, bool row_ok, int t,
                                             uint32_t xrow, RMax rmax, RSum rsum) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int V = a.hidden / VEC;
  T* y_row = static_cast<T*>(a.y) + row * (int64_t)a.hidden;

  float2 v[N][P];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * G + t;
    if (row_ok && i < V) {
      unpack2<T>(lds_u4(xrow + i * 16), v[k]);
#pragma unroll
      for (int p = 0; p < P; ++p) m = fmaxf(m, fmaxf(v[k][p].x, v[k][p].y));
    }
  }
  m = rmax(m);

  float2 acc = splat2(0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (row_ok && (k * G + t) < V) {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        v[k][p].x = expf(v[k][p].x - m);
        v[k][p].y = expf(v[k][p].y - m);
        acc = add2(acc, v[k][p]);
      }
    }
  }
  const float2 inv = splat2(__frcp_rn(rsum(acc.x + acc.y)));

#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * G + t;
    if (row_ok && i < V) {
      float2 o[P];
#pragma unroll
      for (int p = 0; p < P; ++p) o[p] = mul2(v[k][p], inv);
      st_vec(y_row + i * VEC, pack2<T>(o));
    }
  }
}

template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads, N <= 4 ? 3 : 2) smx_bulk_warp_kernel(const SmxArgs a,
                                                                         const BulkCfg c) {
  constexpr int RPW = 32 / LANES;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const Ring ring = make_ring(smem, (uint32_t)c.tile_rows * H * sizeof(T), c.stages);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  ring_init(ring);

  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int local = (threadIdx.x >> 5) * RPW + lane / LANES;   // row within the tile
  bool aborted = false;
  const int64_t taken = run_pipeline<false, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.x), static_cast<const T*>(nullptr), aborted,
      [&](int64_t tile, unsigned char* slot) {
        const int64_t row = tile * c.tile_rows + local;
        const uint32_t xs = smem_addr(slot) + (uint32_t)(local * H * sizeof(T));
        smx_row_smem<T, LANES, N>(a, row, row < a.rows, l, xs,
                                  [](float v) { return group_max<LANES>(v); },
                                  [](float v) { return group_sum<LANES>(v); });
      });
  pipeline_finish(ring, aborted, taken, &s_abort, &s_taken);
}

template <typename T, int N>
__global__ void __launch_bounds__(kBulkThreads, 2) smx_bulk_cta_kernel(const SmxArgs a,
                                                                        const BulkCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[2][kConsumerWarps];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const Ring ring = make_ring(smem, (uint32_t)H * sizeof(T), c.stages);   // one row per tile
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  ring_init(ring);

  bool aborted = false;
  int parity = 0;
  const int64_t taken = run_pipeline<true, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.x), static_cast<const T*>(nullptr), aborted,
      [&](int64_t row, unsigned char* slot) {
        smx_row_smem<T, kBulkThreads, N>(
            a, row, true, threadIdx.x, smem_addr(slot),
            [&](float v) { return cta_max_db<kBulkThreads>(v, red, parity); },
            [&](float v) { return cta_sum_db<kBulkThreads>(v, red, parity); });
      });
  pipeline_finish(ring, aborted, taken, &s_abort, &s_taken);
}

// Any hidden size and alignment. Dynamic shared memory: hidden floats.
// Each thread only ever reads back the entries of srow it wrote itself.
template <typename T>
__global__ void __launch_bounds__(kScalarCta) smx_scalar_kernel(const SmxArgs a) {
  extern __shared__ float srow[];
  __shared__ float red[2][kScalarCta / 32];
  const int H = a.hidden;
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(a.y);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t off = row * (int64_t)H;
    float m = -INFINITY;
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float v = to_f(x[off + j]);
      srow[j] = v;
      m = fmaxf(m, v);
    }
    m = cta_max_db<kScalarCta>(m, red, parity);
    float s = 0.f;
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float e = expf(srow[j] - m);
      srow[j] = e;
      s += e;
    }
    const float inv = __frcp_rn(cta_sum_db<kScalarCta>(s, red, parity));
    for (int j = threadIdx.x; j < H; j += kScalarCta) y[off + j] = from_f<T>(srow[j] * inv);
  }
}

// (kind, lanes, vectors per thread) -> kernel: kind 0 lane group per row,
// 1 CTA per row, 2 scalar.
template <typename T> const void* smx_table_impl(int kind, int group, int n) {
#define NF_SMX_WARP(L)                                                  \
  switch (n) {                                                          \
    case 1: return (const void*)smx_bulk_warp_kernel<T, L, 1>;          \
    case 2: return (const void*)smx_bulk_warp_kernel<T, L, 2>;          \
    case 3: return (const void*)smx_bulk_warp_kernel<T, L, 3>;          \
    case 4: return (const void*)smx_bulk_warp_kernel<T, L, 4>;          \
    case 5: return (const void*)smx_bulk_warp_kernel<T, L, 5>;          \
    case 6: return (const void*)smx_bulk_warp_kernel<T, L, 6>;          \
    case 8: return (const void*)smx_bulk_warp_kernel<T, L, 8>;          \
    default: return nullptr;                                            \
  }
  if (kind == 0) {
    if (group == 8) { NF_SMX_WARP(8) }
    if (group == 16) { NF_SMX_WARP(16) }
    if (group == 32) { NF_SMX_WARP(32) }
  } else if (kind == 1) {
    switch (n) {
      case 2: return (const void*)smx_bulk_cta_kernel<T, 2>;
      case 3: return (const void*)smx_bulk_cta_kernel<T, 3>;
      case 4: return (const void*)smx_bulk_cta_kernel<T, 4>;
      case 5: return (const void*)smx_bulk_cta_kernel<T, 5>;
      case 6: return (const void*)smx_bulk_cta_kernel<T, 6>;
      case 8: return (const void*)smx_bulk_cta_kernel<T, 8>;
      default: return nullptr;
    }
  } else if (kind == 2) {
    return (const void*)smx_scalar_kernel<T>;
  }
#undef NF_SMX_WARP
  return nullptr;
}

}  // namespace nf
