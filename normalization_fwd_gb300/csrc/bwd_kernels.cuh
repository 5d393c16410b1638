// Backward kernels of the fused block (pytorch/pytorch PR 165370).
//
// An RMS/Layer norm backward has two kinds of reduction over the same inputs
// (dy, x_sum and the per-row statistics): dx reduces over the hidden
// dimension of one row, dgamma/dbeta over all rows. Here one persistent
// kernel does both in a single read of the inputs: each row is loaded once
// and kept in registers (the "persistent reduction" the PR requires) while
// its dx is formed, and the row's dy * xhat and dy are added into per-thread
// fp32 accumulators (the outer reduction turned into a partial accumulation).
// At the end each CTA writes its partial dgamma/dbeta row to the workspace,
// and bwd_finalize_kernel adds the partials of all CTAs in a fixed order.
//
// The row -> CTA assignment is a grid-stride loop over a grid sized from the
// SM count, so the partials, and the finalize's fixed-order fp64 sum over
// them, are the same on every run.
#pragma once

#include "common.cuh"
#include "fwd_kernels.cuh"

namespace nf {

// One row for the vector kernels: loads dy and x_sum, computes dx, and adds
// the row into acc_g (dy * xhat) and acc_b (dy). G threads share the row.
template <typename T, int G, int N, typename Reduce2>
__device__ __forceinline__ void bwd_row(const BwdArgs& a, int64_t row, bool row_ok, int t,
                                        Reduce2 reduce2, float (&acc_g)[N][Vec<T>::N],
                                        float (&acc_b)[N][Vec<T>::N]) {
  constexpr int VEC = Vec<T>::N;
  const int H = a.hidden;
  const int V = H / VEC;
  const int64_t off = row * (int64_t)H;
  const T* dy = static_cast<const T*>(a.dy) + off;
  const T* xs = static_cast<const T*>(a.x_sum) + off;
  const T* gamma = static_cast<const T*>(a.gamma);

  uint4 dr[N], xr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (row_ok && v < V) {
      dr[k] = ld_vec(dy + v * VEC);
      xr[k] = ld_vec(xs + v * VEC);
    }
  }
  float mean = 0.f, rstd = 0.f;
  if (row_ok) {
    rstd = a.rstd[row];
    if (!a.rms) mean = a.mean[row];
  }

  // xhat, g = dy * w, the two row sums, and the outer-reduction partials.
  float xh[N][VEC], g[N][VEC];
  float2 sums = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
#pragma unroll
    for (int e = 0; e < VEC; ++e) { xh[k][e] = 0.f; g[k][e] = 0.f; }
    if (row_ok && v < V) {
      float d[VEC], xv[VEC], w[VEC];
      unpack<T>(dr[k], d);
      unpack<T>(xr[k], xv);
      unpack<T>(ld_vec_param(gamma + v * VEC), w);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float we = a.zero_centered ? 1.0f + w[e] : w[e];
        xh[k][e] = (xv[e] - mean) * rstd;
        g[k][e] = d[e] * we;
        sums.x += g[k][e];
        sums.y = fmaf(g[k][e], xh[k][e], sums.y);
        acc_g[k][e] = fmaf(d[e], xh[k][e], acc_g[k][e]);
        acc_b[k][e] += d[e];
      }
    }
  }
  sums = reduce2(sums);
  const float c1 = a.rms ? 0.f : sums.x / (float)H;
  const float c2 = sums.y / (float)H;

  T* dx = static_cast<T*>(a.dx) + off;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (row_ok && v < V) {
      float o[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[e] = rstd * (g[k][e] - c1 - xh[k][e] * c2);
      st_vec(dx + v * VEC, pack<T>(o));
    }
  }
}

template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kWarpCta) bwd_warp_kernel(const BwdArgs a) {
  constexpr int VEC = Vec<T>::N;
  constexpr int RPW = 32 / LANES;
  constexpr int W = kWarpCta / 32;
  constexpr int SLOT = LANES * VEC;   // columns covered by one vector slot
  __shared__ float red[W][SLOT];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane / LANES;
  const int l = lane % LANES;

  float acc_g[N][VEC], acc_b[N][VEC];
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int e = 0; e < VEC; ++e) { acc_g[k][e] = 0.f; acc_b[k][e] = 0.f; }

  const int64_t step = (int64_t)gridDim.x * W * RPW;
  for (int64_t base = ((int64_t)blockIdx.x * W + warp) * RPW; base < a.rows; base += step) {
    const int64_t row = base + sub;
    bwd_row<T, LANES, N>(a, row, row < a.rows, l,
                         [](float2 v) { return group_sum2<LANES>(v); }, acc_g, acc_b);
  }

  // Groups of one warp that share columns: fixed butterfly.
#pragma unroll
  for (int o = LANES; o < 32; o <<= 1)
#pragma unroll
    for (int k = 0; k < N; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        acc_g[k][e] += __shfl_xor_sync(0xffffffffu, acc_g[k][e], o);
        acc_b[k][e] += __shfl_xor_sync(0xffffffffu, acc_b[k][e], o);
      }

  // Warps of the CTA: one vector slot at a time through shared memory, then
  // a fixed-order sum over the warps. Slot k covers columns
  // [k * SLOT, (k + 1) * SLOT), lane l holding l * VEC .. l * VEC + VEC - 1.
  const int H = a.hidden;
  const int C = a.rms ? H : 2 * H;
  float* ws = a.ws + (int64_t)blockIdx.x * C;
  const int nacc = a.rms ? 1 : 2;
  for (int which = 0; which < nacc; ++which) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (sub == 0) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) red[warp][l * VEC + e] = which ? acc_b[k][e] : acc_g[k][e];
      }
      __syncthreads();
      for (int c = threadIdx.x; c < SLOT; c += kWarpCta) {
        const int col = k * SLOT + c;
        if (col < H) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) t += red[w][c];
          ws[which * H + col] = t;
        }
      }
      __syncthreads();
    }
  }
}

template <typename T, int THREADS, int N>
__global__ void __launch_bounds__(THREADS) bwd_cta_kernel(const BwdArgs a) {
  constexpr int VEC = Vec<T>::N;
  __shared__ float2 red[THREADS / 32];
  float acc_g[N][VEC], acc_b[N][VEC];
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int e = 0; e < VEC; ++e) { acc_g[k][e] = 0.f; acc_b[k][e] = 0.f; }

  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    bwd_row<T, THREADS, N>(a, row, true, threadIdx.x,
                           [&](float2 v) { return cta_sum2<THREADS>(v, red); }, acc_g, acc_b);
  }
  // Each column belongs to exactly one thread of the CTA.
  const int H = a.hidden;
  const int V = H / VEC;
  const int C = a.rms ? H : 2 * H;
  float* ws = a.ws + (int64_t)blockIdx.x * C;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * THREADS + threadIdx.x;
    if (v < V) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        ws[v * VEC + e] = acc_g[k][e];
        if (!a.rms) ws[H + v * VEC + e] = acc_b[k][e];
      }
    }
  }
}

// Any hidden size and alignment. Dynamic shared memory: 4 * hidden floats
// (two per-row staging arrays and the two column accumulators); column j
// belongs to thread j % kScalarCta throughout, so no barrier guards them.
template <typename T>
__global__ void __launch_bounds__(kScalarCta) bwd_scalar_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  __shared__ float2 red[kScalarCta / 32];
  const int H = a.hidden;
  float* acc_g = sm;
  float* acc_b = sm + H;
  float* sxh = sm + 2 * H;
  float* sg = sm + 3 * H;
  const T* dy = static_cast<const T*>(a.dy);
  const T* xs = static_cast<const T*>(a.x_sum);
  const T* gamma = static_cast<const T*>(a.gamma);
  T* dx = static_cast<T*>(a.dx);
  for (int j = threadIdx.x; j < H; j += kScalarCta) { acc_g[j] = 0.f; acc_b[j] = 0.f; }
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t off = row * (int64_t)H;
    const float rstd = a.rstd[row];
    const float mean = a.rms ? 0.f : a.mean[row];
    float2 sums = make_float2(0.f, 0.f);
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float d = to_f(dy[off + j]);
      const float xh = (to_f(xs[off + j]) - mean) * rstd;
      const float w = a.zero_centered ? 1.0f + to_f(gamma[j]) : to_f(gamma[j]);
      const float g = d * w;
      sxh[j] = xh;
      sg[j] = g;
      sums.x += g;
      sums.y = fmaf(g, xh, sums.y);
      acc_g[j] = fmaf(d, xh, acc_g[j]);
      acc_b[j] += d;
    }
    sums = cta_sum2<kScalarCta>(sums, red);
    const float c1 = a.rms ? 0.f : sums.x / (float)H;
    const float c2 = sums.y / (float)H;
    for (int j = threadIdx.x; j < H; j += kScalarCta)
      dx[off + j] = from_f<T>(rstd * (sg[j] - c1 - sxh[j] * c2));
  }
  const int C = a.rms ? H : 2 * H;
  float* ws = a.ws + (int64_t)blockIdx.x * C;
  for (int j = threadIdx.x; j < H; j += kScalarCta) {
    ws[j] = acc_g[j];
    if (!a.rms) ws[H + j] = acc_b[j];
  }
}

}  // namespace nf
