// Normalize from partial statistics (NVIDIA/cutlass discussion 874, the
// reply pointing at example 37's gemm_with_layernorm): the GEMM that
// produced the row already summed it per column tile in its epilogue, so the
// row's mean and variance are combined from those per-tile partials instead
// of taken by a reduction over the row. One read of the row, one write of y.
//
// Partials, per row r and column tile t (tile_cols wide from column 0; the
// last tile holds what is left, last_cols):
//   kind 0 (sum, sum of squares):  psum = sum_j s_j, psq = sum_j s_j^2;
//     LayerNorm: mean = S / H, var = max(Q / H - mean^2, 0); RMSNorm: Q / H.
//   kind 1 (sum, centred M2):      psum as above, psq = sum_j (s_j - m_t)^2
//     with m_t = psum / n_t; the tiles combine by the parallel-variance
//     identity M2 = sum psq_t + sum (psum_t - n_t mean)^2 / n_t, var = M2 / H;
//     RMSNorm: mean square = sum (psq_t + psum_t^2 / n_t) / H.
// The tile sums are fp32, each thread adding its own tiles in increasing t,
// then the threads of a row in a fixed butterfly (a CTA exchange for long
// rows). rstd = 1 / sqrt(var + eps); y = (s - mean) * rstd * w + beta
// (RMSNorm: s * rstd * w), w = gamma or 1 + gamma; amax as ln_fwd's.
//
//  * fwdp_tile_kernel: rows of up to 256 16-byte vectors, a lane group of
//    LANES lanes per row, one CTA per tile of 8 * (32 / LANES) rows.
//  * fwdp_cta_kernel: longer rows, one CTA per row, its size fitted to the
//    row at launch.
//  * fwdp_scalar_kernel: any width and alignment, one CTA per row.
#pragma once

#include "common.cuh"

namespace nf {

struct PartialsArgs {
  const void* x;         // [rows, hidden] the stored row
  const float* psum;     // [rows, n_tiles]
  const float* psq;      // [rows, n_tiles]
  const void* gamma;
  const void* beta;      // nullable (always null for RMSNorm)
  void* y;
  float* mean;           // nullable (always null for RMSNorm)
  float* rstd;           // nullable
  unsigned* amax;        // nullable; fp32 bit pattern, zeroed before launch
  int64_t rows;
  int hidden;
  int n_tiles;
  int tile_cols;
  float inv_tile;        // 1 / tile_cols and 1 / last_cols, fp32
  float inv_last;
  float eps;
  float inv_hidden;
  int kind;              // 0 sum + sum of squares, 1 sum + centred M2
  int rms;
  int zero_centered;
};

// This thread's share of the first pass over its tiles t = t0, t0 + step,
// ... in increasing t: x = the sum of psum; y = the sum of psq for kind 0.
// For kind 1 the psq of those tiles are prefetched into L1 for the second
// pass, so both passes' loads leave together and the second pass, which
// needs the row mean, finds them on chip.
__device__ __forceinline__ float2 partial_first(const PartialsArgs& a, int64_t row, int t0,
                                                int step) {
  const float* ps = a.psum + row * (int64_t)a.n_tiles;
  const float* pq = a.psq + row * (int64_t)a.n_tiles;
  float s = 0.f, q = 0.f;
  for (int t = t0; t < a.n_tiles; t += step) {
    s += ps[t];
    if (a.kind == 0) {
      q += pq[t];
    } else {
      asm volatile("prefetch.global.L1 [%0];" ::"l"(pq + t));
    }
  }
  return make_float2(s, q);
}

// Kind 1's second pass over the same tiles: psq_t + (psum_t - n_t mean)^2
// / n_t for LayerNorm (the row mean from the first pass), psq_t +
// psum_t^2 / n_t for RMSNorm.
__device__ __forceinline__ float partial_second(const PartialsArgs& a, int64_t row, int t0,
                                                int step, float mean) {
  const float* ps = a.psum + row * (int64_t)a.n_tiles;
  const float* pq = a.psq + row * (int64_t)a.n_tiles;
  float q = 0.f;
  for (int t = t0; t < a.n_tiles; t += step) {
    const bool last = t == a.n_tiles - 1;
    const float n = last ? (float)(a.hidden - (a.n_tiles - 1) * a.tile_cols)
                         : (float)a.tile_cols;
    const float inv_n = last ? a.inv_last : a.inv_tile;
    const float d = a.rms ? ps[t] : fmaf(-n, mean, ps[t]);
    q += fmaf(d * d, inv_n, pq[t]);
  }
  return q;
}

// (mean, rstd) of the row from the two reduced quantities.
__device__ __forceinline__ float2 partial_stats(const PartialsArgs& a, float S, float Q) {
  const float mean = a.rms ? 0.f : S * a.inv_hidden;
  float v = Q * a.inv_hidden;
  if (!a.rms && a.kind == 0) v = fmaxf(fmaf(-mean, mean, v), 0.f);
  return make_float2(mean, 1.0f / sqrtf(v + a.eps));
}

// y of one 16-byte vector of the row, with its amax update.
template <typename T>
__device__ __forceinline__ void partial_store(const PartialsArgs& a, T* yrow, int v,
                                              const uint4& xr, float mean, float rstd,
                                              unsigned& amax_acc) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  float2 s[P], w[P], o[P];
  unpack2<T>(xr, s);
  unpack2<T>(ld_vec_param(static_cast<const T*>(a.gamma) + v * VEC), w);
  if (a.beta) {
    unpack2<T>(ld_vec_param(static_cast<const T*>(a.beta) + v * VEC), o);
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) o[i] = splat2(0.f);
  }
  const float2 r2 = splat2(rstd), nm = splat2(-mean);
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (a.zero_centered) w[i] = add2(w[i], splat2(1.f));
    o[i] = fma2(mul2(add2(s[i], nm), r2), w[i], o[i]);
  }
  const uint4 packed = pack2<T>(o);
  st_vec(yrow + v * VEC, packed);
  if (a.amax) amax_update<T>(amax_acc, packed);
}

// The CTA's amax: one atomicMax, skipped unless it beats the stored value.
template <typename T>
__device__ __forceinline__ void partial_amax_commit(const PartialsArgs& a, unsigned amax_acc,
                                                    unsigned* red) {
  unsigned m = __reduce_max_sync(0xffffffffu, amax_bits<T>(amax_acc));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = max(m, red[i]);
    if (m > *(volatile unsigned*)a.amax) atomicMax(a.amax, m);
  }
}

template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads) fwdp_tile_kernel(const PartialsArgs a) {
  constexpr int RPW = 32 / LANES;
  constexpr int VEC = Vec<T>::N;
  __shared__ unsigned red_amax[kConsumerWarps];
  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int64_t row =
      ((int64_t)blockIdx.x * kConsumerWarps + (threadIdx.x >> 5)) * RPW + lane / LANES;
  const bool row_ok = row < a.rows;
  const int V = a.hidden / VEC;
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)a.hidden;
  uint4 xr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * LANES + l;
    if (row_ok && v < V) xr[k] = ld_vec(x + v * VEC);
  }
  // Statistics: every lane group runs its butterflies (whole warps take
  // part in the shuffles); a group past the last row reads no partials.
  float2 sq;
  float Q;
  if (a.n_tiles <= LANES) {
    // At most one tile per lane: lane l holds tile l's (psum, psq) in
    // registers for both passes, loaded together with no loop. The sums
    // are those of the general path below (one term per lane).
    const bool has = row_ok && l < a.n_tiles;
    float ps = 0.f, pq = 0.f;
    if (has) {
      ps = a.psum[row * (int64_t)a.n_tiles + l];
      pq = a.psq[row * (int64_t)a.n_tiles + l];
    }
    sq = group_sum2<LANES>(make_float2(ps, a.kind == 0 ? pq : 0.f));
    Q = sq.y;
    if (a.kind == 1) {
      const bool last = l == a.n_tiles - 1;
      const float n = last ? (float)(a.hidden - (a.n_tiles - 1) * a.tile_cols)
                           : (float)a.tile_cols;
      const float inv_n = last ? a.inv_last : a.inv_tile;
      const float d = a.rms ? ps : fmaf(-n, sq.x * a.inv_hidden, ps);
      Q = group_sum<LANES>(has ? fmaf(d * d, inv_n, pq) : 0.f);
    }
  } else {
    sq = group_sum2<LANES>(row_ok ? partial_first(a, row, l, LANES) : make_float2(0.f, 0.f));
    Q = sq.y;
    if (a.kind == 1) {
      const float mean0 = a.rms ? 0.f : sq.x * a.inv_hidden;
      Q = group_sum<LANES>(row_ok ? partial_second(a, row, l, LANES, mean0) : 0.f);
    }
  }
  const float2 st = partial_stats(a, sq.x, Q);
  if (row_ok && l == 0) {
    if (a.mean) a.mean[row] = st.x;
    if (a.rstd) a.rstd[row] = st.y;
  }
  unsigned amax_acc = 0;
  T* yrow = static_cast<T*>(a.y) + row * (int64_t)a.hidden;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * LANES + l;
    if (row_ok && v < V) partial_store<T>(a, yrow, v, xr[k], st.x, st.y, amax_acc);
  }
  if (a.amax) partial_amax_commit<T>(a, amax_acc, red_amax);
}

// The CTA's size is fitted to the row at launch (blockDim.x, a whole number
// of warps up to kMaxFitThreads).
template <typename T, int N>
__global__ void __launch_bounds__(kMaxFitThreads) __maxnreg__(N <= 4 ? 48 : 80) fwdp_cta_kernel(const PartialsArgs a) {
  constexpr int VEC = Vec<T>::N;
  __shared__ float2 red[2][kMaxFitWarps];
  __shared__ float red1[2][kMaxFitWarps];
  int parity1 = 0;
  __shared__ unsigned red_amax[kMaxFitWarps];
  const int nt = blockDim.x;
  const int64_t row = blockIdx.x;
  const int V = a.hidden / VEC;
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)a.hidden;
  uint4 xr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * nt + threadIdx.x;
    if (v < V) xr[k] = ld_vec(x + v * VEC);
  }
  int parity = 0;
  const float2 sq = cta_sum2_db_fit(partial_first(a, row, threadIdx.x, nt), red, parity);
  float Q = sq.y;
  if (a.kind == 1) {
    const float mean0 = a.rms ? 0.f : sq.x * a.inv_hidden;
    Q = cta_sum_db_fit(partial_second(a, row, threadIdx.x, nt, mean0), red1, parity1);
  }
  const float2 st = partial_stats(a, sq.x, Q);
  if (threadIdx.x == 0) {
    if (a.mean) a.mean[row] = st.x;
    if (a.rstd) a.rstd[row] = st.y;
  }
  unsigned amax_acc = 0;
  T* yrow = static_cast<T*>(a.y) + row * (int64_t)a.hidden;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * nt + threadIdx.x;
    if (v < V) partial_store<T>(a, yrow, v, xr[k], st.x, st.y, amax_acc);
  }
  if (a.amax) partial_amax_commit<T>(a, amax_acc, red_amax);
}

// Any width and alignment: one CTA per row, element-wise.
template <typename T>
__global__ void __launch_bounds__(kScalarCta) fwdp_scalar_kernel(const PartialsArgs a) {
  __shared__ float2 red[2][kScalarCta / 32];
  __shared__ float red1[2][kScalarCta / 32];
  __shared__ unsigned red_amax[kScalarCta / 32];
  const int64_t row = blockIdx.x;
  const int H = a.hidden;
  int parity = 0, parity1 = 0;
  const float2 sq = cta_sum2_db<kScalarCta>(partial_first(a, row, threadIdx.x, kScalarCta), red,
                                            parity);
  float Q = sq.y;
  if (a.kind == 1) {
    const float mean0 = a.rms ? 0.f : sq.x * a.inv_hidden;
    Q = cta_sum_db<kScalarCta>(partial_second(a, row, threadIdx.x, kScalarCta, mean0), red1,
                               parity1);
  }
  const float2 st = partial_stats(a, sq.x, Q);
  if (threadIdx.x == 0) {
    if (a.mean) a.mean[row] = st.x;
    if (a.rstd) a.rstd[row] = st.y;
  }
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)H;
  const T* gamma = static_cast<const T*>(a.gamma);
  const T* beta = static_cast<const T*>(a.beta);
  T* y = static_cast<T*>(a.y) + row * (int64_t)H;
  unsigned amax_acc = 0;
  for (int j = threadIdx.x; j < H; j += kScalarCta) {
    const float w = a.zero_centered ? 1.0f + to_f(gamma[j]) : to_f(gamma[j]);
    const float b = beta ? to_f(beta[j]) : 0.f;
    const T o = from_f<T>(fmaf((to_f(x[j]) - st.x) * st.y, w, b));
    y[j] = o;
    amax_acc = max(amax_acc, abs_bits(to_f(o)));
  }
  if (a.amax) {
    unsigned m = __reduce_max_sync(0xffffffffu, amax_acc);
    if ((threadIdx.x & 31) == 0) red_amax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < kScalarCta / 32; ++i) m = max(m, red_amax[i]);
      if (m > *(volatile unsigned*)a.amax) atomicMax(a.amax, m);
    }
  }
}

template <typename T> const void* partials_table_impl(int kind, int group, int n) {
#define NF_FWDP_TILE(L)                                               \
  switch (n) {                                                        \
    case 1: return (const void*)fwdp_tile_kernel<T, L, 1>;            \
    case 2: return (const void*)fwdp_tile_kernel<T, L, 2>;            \
    case 3: return (const void*)fwdp_tile_kernel<T, L, 3>;            \
    case 4: return (const void*)fwdp_tile_kernel<T, L, 4>;            \
    case 5: return (const void*)fwdp_tile_kernel<T, L, 5>;            \
    case 6: return (const void*)fwdp_tile_kernel<T, L, 6>;            \
    case 8: return (const void*)fwdp_tile_kernel<T, L, 8>;            \
    default: return nullptr;                                          \
  }
  if (kind == 4) {
    if (group == 8) { NF_FWDP_TILE(8) }
    if (group == 16) { NF_FWDP_TILE(16) }
    if (group == 32) { NF_FWDP_TILE(32) }
  } else if (kind == 5) {
    switch (n) {
      case 2: return (const void*)fwdp_cta_kernel<T, 2>;
      case 3: return (const void*)fwdp_cta_kernel<T, 3>;
      case 4: return (const void*)fwdp_cta_kernel<T, 4>;
      case 5: return (const void*)fwdp_cta_kernel<T, 5>;
      case 6: return (const void*)fwdp_cta_kernel<T, 6>;
      case 8: return (const void*)fwdp_cta_kernel<T, 8>;
      default: return nullptr;
    }
  } else if (kind == 2) {
    return (const void*)fwdp_scalar_kernel<T>;
  }
#undef NF_FWDP_TILE
  return nullptr;
}

}  // namespace nf
