// Forward kernels of the fused block: bias + residual add, LayerNorm or
// RMSNorm, amax of |y| (NVIDIA/Fuser issue 1660, the layernorm + amax
// snippet; iree-org/iree issue 9139, mean / variance / normalize over one read
// of the input).
//
// Every kernel keeps a row on chip between the statistics and the normalize
// step, so each input element is read from HBM once and each output written
// once; the amax partial is committed once per CTA.
//
//  * fwd_tile_kernel / fwd_tile_cta_kernel (default for 16-byte aligned
//    rows): one CTA per tile of rows (a lane group of LANES lanes per row) or
//    per row (rows of more than 256 vectors), as many CTAs as that takes;
//    rows go straight from global memory into registers and the CTA
//    scheduler keeps loads in flight as CTAs end and start.
//  * fwd_bulk_warp_kernel / fwd_bulk_cta_kernel (selected by a test through
//    ln_testing_select_kernels):
//    persistent CTAs; tiles of rows stream into a shared-memory ring by
//    cp.async.bulk (every slot in flight, each refilled by the warp that
//    frees it last) and 8 warps normalize them from shared memory.
//  * fwd_scalar_kernel: any hidden size and alignment; element-wise loads,
//    the row staged in shared memory.
#pragma once

#include "bulk.cuh"
#include "common.cuh"

namespace nf {

// ---- bulk-copy pipelined kernels ------------------------------------------

// Per-column parameters of the forward: w = gamma (+1 for zero-centered
// gamma), bias and beta (absent ones have a null global pointer). The lane
// group kernels stage them in shared memory once per CTA; the CTA-per-row
// kernels read them from global memory, leaving shared memory to the ring.
template <typename T>
struct FwdParams {
  ParamRow<T> w, bias, beta;
  float fp8_scale;     // loaded once per CTA when y_fp8 is written
};

template <typename T>
__device__ __forceinline__ FwdParams<T> fwd_params(const FwdArgs& a, float* p_s) {
  const int H = a.hidden;
  const T* bias = static_cast<const T*>(a.bias);
  const T* beta = static_cast<const T*>(a.beta);
  FwdParams<T> p;
  p.fp8_scale = a.y_fp8 ? *a.fp8_scale : 0.f;
  p.w = {p_s, static_cast<const T*>(a.gamma), H, a.zero_centered != 0};
  p.bias = {p_s && bias ? p_s + H : nullptr, bias, H, false};
  p.beta = {p_s && beta ? p_s + (bias ? 2 : 1) * H : nullptr, beta, H, false};
  if (p_s) {
    stage_param_row<T>(p.w.g, H, p.w.plus_one, p_s);
    if (bias) stage_param_row<T>(bias, H, false, const_cast<float*>(p.bias.s));
    if (beta) stage_param_row<T>(beta, H, false, const_cast<float*>(p.beta.s));
    __syncthreads();
  }
  return p;
}

// The row body: `xr` / `rr` hold the thread's 16-byte vectors k * G + t of
// the x and residual rows (those below V; rr only with a residual),
// parameters staged in shared memory (kStaged) or read from global memory.
// Values are kept as fp32 pairs (packed fp32 math). G = 0: the row's
// threads are the whole CTA, blockDim.x of them.
template <typename T, int G0, int N, bool kStaged, typename Reduce>
__device__ __forceinline__ void fwd_row_regs(const FwdArgs& a, int64_t row, bool row_ok, int t,
                                             const uint4 (&xr)[N], const uint4 (&rr)[N],
                                             bool has_res, const FwdParams<T>& p, Reduce reduce,
                                             unsigned& amax_acc, bool write_stats) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int G = G0 > 0 ? G0 : (int)blockDim.x;
  const int H = a.hidden;
  const int V = H / VEC;
  T* sum_row = a.out_sum ? static_cast<T*>(a.out_sum) + row * (int64_t)H : nullptr;
  T* y_row = static_cast<T*>(a.y) + row * (int64_t)H;
  const uint32_t wa = kStaged ? p.w.saddr() : 0u;
  const uint32_t ba = (kStaged && p.beta.g) ? p.beta.saddr() : 0u;
  const uint32_t bia = (kStaged && p.bias.g) ? p.bias.saddr() : 0u;

  // F1: s = (x + bias) + residual in fp32, stored rounded; the statistics
  // see the stored value.
  float2 s[N][P];
  float2 t1 = splat2(0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
#pragma unroll
    for (int i = 0; i < P; ++i) s[k][i] = splat2(0.f);
    if (row_ok && v < V) {
      unpack2<T>(xr[k], s[k]);
      if (p.bias.g) {
        float2 b[P];
        p.bias.template load2<kStaged>(v, b, bia);
#pragma unroll
        for (int i = 0; i < P; ++i) s[k][i] = add2(s[k][i], b[i]);
      }
      if (has_res) {
        float2 r[P];
        unpack2<T>(rr[k], r);
#pragma unroll
        for (int i = 0; i < P; ++i) s[k][i] = add2(s[k][i], r[i]);
      }
      const uint4 packed = pack2<T>(s[k]);
      if (sum_row) st_vec(sum_row + v * VEC, packed);
      unpack2<T>(packed, s[k]);
#pragma unroll
      for (int i = 0; i < P; ++i) t1 = add2(t1, s[k][i]);
    }
  }

  // F2: mean, then the centred sum of squares (RMSNorm: mean 0).
  const float mean = a.rms ? 0.f : reduce(t1.x + t1.y) / (float)H;
  const float2 neg_mean = splat2(-mean);
  float2 t2 = splat2(0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (row_ok && (k * G + t) < V) {
#pragma unroll
      for (int i = 0; i < P; ++i) {
        s[k][i] = add2(s[k][i], neg_mean);
        t2 = fma2(s[k][i], s[k][i], t2);
      }
    }
  }
  const float rstd = 1.0f / sqrtf(reduce(t2.x + t2.y) / (float)H + a.eps);
  if (row_ok && write_stats) {
    if (a.mean) a.mean[row] = mean;
    if (a.rstd) a.rstd[row] = rstd;
  }

  // F3: y = (s - mean) * rstd * w + beta; F4: amax of the stored y.
  const float2 r2 = splat2(rstd);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (row_ok && v < V) {
      float2 w[P], o[P];
      p.w.template load2<kStaged>(v, w, wa);
      if (p.beta.g) {
        p.beta.template load2<kStaged>(v, o, ba);
      } else {
#pragma unroll
        for (int i = 0; i < P; ++i) o[i] = splat2(0.f);
      }
#pragma unroll
      for (int i = 0; i < P; ++i) o[i] = fma2(mul2(s[k][i], r2), w[i], o[i]);
      const uint4 packed = pack2<T>(o);
      if (a.y) st_vec(y_row + v * VEC, packed);
      if (a.amax) amax_update<T>(amax_acc, packed);
      if (a.y_fp8) {           // FP8 of the stored (rounded) y
        unpack2<T>(packed, o);
        store_fp8<VEC>(a.y_fp8 + row * (int64_t)H + v * VEC, o, p.fp8_scale);
      }
    }
  }
}

// The same row with its vectors read from shared memory (the ring slot).
template <typename T, int G, int N, bool kStaged, typename Reduce>
__device__ __forceinline__ void fwd_row_smem(const FwdArgs& a, int64_t row, bool row_ok, int t,
                                             uint32_t xrow, uint32_t rrow, bool has_res,
                                             const FwdParams<T>& p, Reduce reduce,
                                             unsigned& amax_acc, bool write_stats) {
  const int V = a.hidden / Vec<T>::N;
  uint4 xr[N], rr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (row_ok && v < V) {
      xr[k] = lds_u4(xrow + v * 16);
      if (has_res) rr[k] = lds_u4(rrow + v * 16);
    }
  }
  fwd_row_regs<T, G, N, kStaged>(a, row, row_ok, t, xr, rr, has_res, p, reduce, amax_acc,
                                 write_stats);
}

// One CTA per tile of 8 * (32 / LANES) rows, as many CTAs as tiles: rows go
// straight from global memory into registers (no ring) and the CTA scheduler
// keeps loads in flight as CTAs end and start. Parameters come from global
// memory (L1/L2-resident). amax: a CTA issues its atomicMax only when its
// maximum beats the value already there.
template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads, N <= 3 ? 4 : 2) fwd_tile_kernel(const FwdArgs a) {
  constexpr int RPW = 32 / LANES;
  constexpr int VEC = Vec<T>::N;
  __shared__ unsigned red_amax[kConsumerWarps];
  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int64_t row =
      ((int64_t)blockIdx.x * kConsumerWarps + (threadIdx.x >> 5)) * RPW + lane / LANES;
  const bool row_ok = row < a.rows;
  const int H = a.hidden;
  const int V = H / VEC;
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)H;
  const T* res = a.residual ? static_cast<const T*>(a.residual) + row * (int64_t)H : nullptr;
  uint4 xr[N], rr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * LANES + l;
    if (row_ok && v < V) {
      xr[k] = ld_vec(x + v * VEC);
      if (res) rr[k] = ld_vec(res + v * VEC);
    }
  }
  const FwdParams<T> p = fwd_params<T>(a, nullptr);
  unsigned amax_acc = 0;
  fwd_row_regs<T, LANES, N, false>(a, row, row_ok, l, xr, rr, res != nullptr, p,
                                   [](float v) { return group_sum<LANES>(v); }, amax_acc, l == 0);
  if (a.amax) {
    unsigned m = __reduce_max_sync(0xffffffffu, amax_bits<T>(amax_acc));
    if (lane == 0) red_amax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < kConsumerWarps; ++i) m = max(m, red_amax[i]);
      if (m > *(volatile unsigned*)a.amax) atomicMax(a.amax, m);
    }
  }
}

// Rows of more than 256 vectors from registers: one CTA per row, as many
// CTAs as rows; the row sums go through the CTA (double-buffered, one
// barrier each).
// One CTA per row, its size fitted to the row at launch (blockDim.x = NT,
// a whole number of warps up to kMaxFitThreads, NT * N >= the row's
// vectors): small CTAs of a few vectors per thread keep more rows in flight
// per SM than a fixed 256 threads that leave vector slots idle (2560 bf16,
// 52428 rows: 157 us as 64 x 5 against 228 as 256 x 2).
template <typename T, int N>
__global__ void __launch_bounds__(kMaxFitThreads) __maxnreg__(N <= 4 ? 56 : 128) fwd_tile_cta_kernel(const FwdArgs a) {
  constexpr int VEC = Vec<T>::N;
  __shared__ float red[2][kMaxFitWarps];
  __shared__ unsigned red_amax[kMaxFitWarps];
  const int nt = blockDim.x;
  const int64_t row = blockIdx.x;
  const int H = a.hidden;
  const int V = H / VEC;
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)H;
  const T* res = a.residual ? static_cast<const T*>(a.residual) + row * (int64_t)H : nullptr;
  uint4 xr[N], rr[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * nt + threadIdx.x;
    if (v < V) {
      xr[k] = ld_vec(x + v * VEC);
      if (res) rr[k] = ld_vec(res + v * VEC);
    }
  }
  const FwdParams<T> p = fwd_params<T>(a, nullptr);
  unsigned amax_acc = 0;
  int parity = 0;
  fwd_row_regs<T, 0, N, false>(
      a, row, true, threadIdx.x, xr, rr, res != nullptr, p,
      [&](float v) { return cta_sum_db_fit(v, red, parity); }, amax_acc, threadIdx.x == 0);
  if (a.amax) {
    unsigned m = __reduce_max_sync(0xffffffffu, amax_bits<T>(amax_acc));
    if ((threadIdx.x & 31) == 0) red_amax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < (nt >> 5); ++i) m = max(m, red_amax[i]);
      if (m > *(volatile unsigned*)a.amax) atomicMax(a.amax, m);
    }
  }
}

template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads, N <= 4 ? 3 : 2) fwd_bulk_warp_kernel(const FwdArgs a,
                                                                         const BulkCfg c) {
  constexpr int RPW = 32 / LANES;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ unsigned red_amax[kConsumerWarps];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const int n_in = a.residual ? 2 : 1;
  const uint32_t in_bytes = (uint32_t)c.tile_rows * H * sizeof(T);
  const Ring ring = make_ring(smem, n_in * in_bytes, c.stages);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  const FwdParams<T> p = fwd_params<T>(a, reinterpret_cast<float*>(ring.after));
  ring_init(ring);

  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int local = (threadIdx.x >> 5) * RPW + lane / LANES;   // row within the tile
  bool aborted = false;
  unsigned amax_acc = 0;
  const int64_t taken = run_pipeline<false, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.x), static_cast<const T*>(a.residual), aborted,
      [&](int64_t tile, unsigned char* slot) {
        const int64_t row = tile * c.tile_rows + local;
        const uint32_t xs = smem_addr(slot) + (uint32_t)(local * H * sizeof(T));
        fwd_row_smem<T, LANES, N, true>(a, row, row < a.rows, l, xs, xs + in_bytes,
                                        a.residual != nullptr, p,
                                  [](float v) { return group_sum<LANES>(v); }, amax_acc, l == 0);
      });
  if (pipeline_finish(ring, aborted, taken, &s_abort, &s_taken)) return;
  if (a.amax) cta_amax_commit(amax_bits<T>(amax_acc), a.amax, red_amax);
}

template <typename T, int N>
__global__ void __launch_bounds__(kBulkThreads, 2) fwd_bulk_cta_kernel(const FwdArgs a,
                                                                        const BulkCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[2][kConsumerWarps];
  __shared__ unsigned red_amax[kConsumerWarps];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const int n_in = a.residual ? 2 : 1;
  const uint32_t in_bytes = (uint32_t)H * sizeof(T);   // one row per tile
  const Ring ring = make_ring(smem, n_in * in_bytes, c.stages);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  const FwdParams<T> p = fwd_params<T>(a, nullptr);
  ring_init(ring);

  bool aborted = false;
  unsigned amax_acc = 0;
  int parity = 0;
  const int64_t taken = run_pipeline<true, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.x), static_cast<const T*>(a.residual), aborted,
      [&](int64_t row, unsigned char* slot) {
        const uint32_t xs = smem_addr(slot);
        fwd_row_smem<T, kBulkThreads, N, false>(a, row, true, threadIdx.x, xs, xs + in_bytes,
                                                a.residual != nullptr, p,
                                         [&](float v) { return cta_sum_db<kBulkThreads>(v, red, parity); },
                                         amax_acc, threadIdx.x == 0);
      });
  if (pipeline_finish(ring, aborted, taken, &s_abort, &s_taken)) return;
  if (a.amax) cta_amax_commit(amax_bits<T>(amax_acc), a.amax, red_amax);
}

// ---- scalar kernel ----------------------------------------------------------

// Any hidden size and alignment. Dynamic shared memory: hidden floats.
template <typename T>
__global__ void __launch_bounds__(kScalarCta) fwd_scalar_kernel(const FwdArgs a) {
  extern __shared__ float srow[];
  __shared__ float red[kScalarCta / 32];
  __shared__ unsigned red_amax[kScalarCta / 32];
  const int H = a.hidden;
  const T* x = static_cast<const T*>(a.x);
  const T* res = static_cast<const T*>(a.residual);
  const T* bias = static_cast<const T*>(a.bias);
  const T* gamma = static_cast<const T*>(a.gamma);
  const T* beta = static_cast<const T*>(a.beta);
  T* out_sum = static_cast<T*>(a.out_sum);
  T* y = static_cast<T*>(a.y);
  unsigned amax_u = 0;
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t off = row * (int64_t)H;
    float t1 = 0.f;
    // Each thread only ever reads back the srow entries it wrote itself.
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      float s = to_f(x[off + j]);
      if (bias) s += to_f(bias[j]);
      if (res) s += to_f(res[off + j]);
      const T st = from_f<T>(s);
      if (out_sum) out_sum[off + j] = st;
      s = to_f(st);
      srow[j] = s;
      t1 += s;
    }
    const float mean = a.rms ? 0.f : cta_sum<kScalarCta>(t1, red) / (float)H;
    float t2 = 0.f;
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float d = srow[j] - mean;
      t2 = fmaf(d, d, t2);
    }
    const float var = cta_sum<kScalarCta>(t2, red) / (float)H;
    const float rstd = 1.0f / sqrtf(var + a.eps);
    if (threadIdx.x == 0) {
      if (a.mean) a.mean[row] = mean;
      if (a.rstd) a.rstd[row] = rstd;
    }
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float w = a.zero_centered ? 1.0f + to_f(gamma[j]) : to_f(gamma[j]);
      const float b = beta ? to_f(beta[j]) : 0.f;
      const T o = from_f<T>(fmaf((srow[j] - mean) * rstd, w, b));
      if (y) y[off + j] = o;
      amax_u = max(amax_u, abs_bits(to_f(o)));
      if (a.y_fp8) a.y_fp8[off + j] = fp8_one(to_f(o), *a.fp8_scale);
    }
  }
  if (a.amax) cta_amax_commit(amax_u, a.amax, red_amax);
}

}  // namespace nf
