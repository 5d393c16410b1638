// Row softmax kernels: y[r, :] = exp(x[r, :] - max_j x[r, j]) / sum_j exp(...).
//
// Definition (iree-org/iree issue 9139, the softmax IR and its single
// dispatch form): per row, a max reduction, the exponential of the shifted
// row, a sum reduction, and a division. Like the normalization forward the
// whole row stays on chip between the reductions, so each element is read
// from HBM once and written once.
//
//  * smx_reg_kernel / smx_reg_cta_kernel (default for 16-byte aligned rows):
//    one CTA per tile of rows (lane groups) or per row, rows straight from
//    global memory into registers.
//  * smx_bulk_warp_kernel / smx_bulk_cta_kernel (selected by a test through
//    ln_testing_select_kernels):
//    tiles of rows stream into a shared-memory ring by cp.async.bulk (the
//    ring and refill scheme of the normalization kernels) and 8 warps work on
//    them from shared memory: a lane group of LANES lanes per row, or all 256
//    threads per row for rows of more than 256 vectors.
//  * smx_scalar_kernel: any hidden size and alignment; element-wise loads,
//    the row staged in shared memory as fp32.
//
// Arithmetic: fp32 throughout. m = max, e = exp2f((x - m) * log2 e) (one fma
// and one exp2f per element), s = sum of e, y = e * (1/s) with a correctly
// rounded reciprocal. A row whose entries are all -inf, or that holds a NaN
// or +inf, comes out as NaN, as the definition gives.
#pragma once

#include <math.h>

#include "bulk.cuh"
#include "common.cuh"

namespace nf {

// exp(v) = 2^(v * log2(e)): the exponential of the shifted row is taken as
// exp2f(fma(x, log2e, -m * log2e)). The rounding of m * log2e multiplies every
// e_j of the row by the same factor, which the division by their sum removes.
constexpr float kLog2e = 1.4426950408889634f;

// Running max over a row's 16-byte vectors. For bf16/fp16 the max is taken
// on the packed pairs (exact: no rounding is involved) and widened at the end.
template <typename T> struct RowMax;
template <> struct RowMax<float> {
  float m = -INFINITY;
  __device__ __forceinline__ void add(const uint4& u) {
    m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                       fmaxf(__uint_as_float(u.z), __uint_as_float(u.w))));
  }
  __device__ __forceinline__ float value() const { return m; }
};
template <> struct RowMax<bf16> {
  __nv_bfloat162 m = __nv_bfloat162(__ushort_as_bfloat16(0xff80u), __ushort_as_bfloat16(0xff80u));
  static __device__ __forceinline__ __nv_bfloat162 h(unsigned w) {
    return *reinterpret_cast<__nv_bfloat162*>(&w);
  }
  __device__ __forceinline__ void add(const uint4& u) {
    m = __hmax2(m, __hmax2(__hmax2(h(u.x), h(u.y)), __hmax2(h(u.z), h(u.w))));
  }
  __device__ __forceinline__ float value() const {
    return fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
  }
};
template <> struct RowMax<f16> {
  __half2 m = __half2(__ushort_as_half(0xfc00u), __ushort_as_half(0xfc00u));
  static __device__ __forceinline__ __half2 h(unsigned w) { return *reinterpret_cast<__half2*>(&w); }
  __device__ __forceinline__ void add(const uint4& u) {
    m = __hmax2(m, __hmax2(__hmax2(h(u.x), h(u.y)), __hmax2(h(u.z), h(u.w))));
  }
  __device__ __forceinline__ float value() const {
    return fmaxf(__half2float(m.x), __half2float(m.y));
  }
};

// e = 2^(x * log2e + nml) for one vector, added into acc; nml = -shift * log2e.
template <typename T>
__device__ __forceinline__ void exp_vec(const uint4& u, float nml, float2* e, float2& acc) {
  constexpr int P = Vec<T>::N / 2;
  unpack2<T>(u, e);
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float2 t = fma2(e[p], splat2(kLog2e), splat2(nml));
    e[p].x = exp2f(t.x);
    e[p].y = exp2f(t.y);
    acc = add2(acc, e[p]);
  }
}

// Lane-group rows: `G` lanes share the row, this one is `t`; `raw` holds
// the lane's 16-byte vectors k * G + t of the row (those below V).
// Reductions: max over the row, then the sum.
template <typename T, int G, int N, typename RMax, typename RSum>
__device__ __forceinline__ void smx_row_regs(const SmxArgs& a, int64_t row, bool row_ok, int t,
                                             const uint4 (&raw)[N], RMax rmax, RSum rsum) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int V = a.hidden / VEC;
  T* y_row = static_cast<T*>(a.y) + row * (int64_t)a.hidden;

  RowMax<T> rm;
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (row_ok && k * G + t < V) rm.add(raw[k]);
  const float nml = -rmax(rm.value()) * kLog2e;

  float2 e[N][P];
  float2 acc = splat2(0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (row_ok && (k * G + t) < V) exp_vec<T>(raw[k], nml, e[k], acc);
  }
  const float2 inv = splat2(__frcp_rn(rsum(acc.x + acc.y)));

#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * G + t;
    if (row_ok && i < V) {
      float2 o[P];
#pragma unroll
      for (int p = 0; p < P; ++p) o[p] = mul2(e[k][p], inv);
      st_vec(y_row + i * VEC, pack2<T>(o));
    }
  }
}

// The same row with its vectors read from shared memory (row address `xrow`).
template <typename T, int G, int N, typename RMax, typename RSum>
__device__ __forceinline__ void smx_row_smem(const SmxArgs& a, int64_t row, bool row_ok, int t,
                                             uint32_t xrow, RMax rmax, RSum rsum) {
  const int V = a.hidden / Vec<T>::N;
  uint4 raw[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * G + t;
    if (row_ok && i < V) raw[k] = lds_u4(xrow + i * 16);
  }
  smx_row_regs<T, G, N>(a, row, row_ok, t, raw, rmax, rsum);
}

// Lane groups, rows straight from global memory into registers, one CTA per
// 8 * (32 / LANES) rows and as many CTAs as that takes: no ring, the CTA
// scheduler keeps loads in flight by starting a new CTA whenever one ends.
// At 576000 x 384 bf16 this ran 127 us against 159 us for the ring kernel
// and 131 us for a device-to-device cudaMemcpy of the same bytes.
template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads, N <= 3 ? 6 : (N <= 4 ? 4 : 2))
    smx_reg_kernel(const SmxArgs a) {
  constexpr int RPW = 32 / LANES;
  constexpr int VEC = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int64_t row = ((int64_t)blockIdx.x * kConsumerWarps + (threadIdx.x >> 5)) * RPW + lane / LANES;
  const bool row_ok = row < a.rows;
  const int V = a.hidden / VEC;
  const T* x = static_cast<const T*>(a.x) + row * (int64_t)a.hidden;
  uint4 raw[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * LANES + l;
    if (row_ok && i < V) raw[k] = ld_vec(x + i * VEC);
  }
  smx_row_regs<T, LANES, N>(a, row, row_ok, l, raw, [](float v) { return group_max<LANES>(v); },
                            [](float v) { return group_sum<LANES>(v); });
}

// CTA rows (all the CTA's threads on one row), with one barrier per row: each warp
// takes the exponentials against its own max m_w and sums them to s_w; the
// warps' (m_w, s_w) pairs meet in shared memory, where every warp forms the
// row max M and s = sum_w s_w * exp(m_w - M); thread scale exp(m_w - M) / s
// (all in log2 units: L = m * log2 e).
// This is the online normalizer of Milakov and Gimelshein ("Online normalizer
// calculation for softmax", 2018) applied across the CTA's warps. A warp
// whose entries are all -inf shifts by 0 instead (its e are 0 either way)
// and contributes 0; a row that is all -inf stays NaN.
template <typename T, int N>
__device__ __forceinline__ void smx_row_cta_regs(const SmxArgs& a, int64_t row,
                                                 const uint4 (&raw)[N],
                                                 float2 (*red)[kMaxFitWarps], int& parity) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int V = a.hidden / VEC;
  const int nt = blockDim.x;
  const int t = threadIdx.x;
  const int lane = t & 31;
  T* y_row = static_cast<T*>(a.y) + row * (int64_t)a.hidden;

  RowMax<T> rm;
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k * nt + t < V) rm.add(raw[k]);
  // Lw: this warp's shift in log2 units, rounded once. The warps exchange Lw
  // itself, so the factor 2^(Lw - L) that moves a warp's e onto the row max
  // carries exactly the rounding its exponentials were taken with.
  const float Lw = group_max<32>(rm.value()) * kLog2e;
  float2 e[N][P];
  float2 acc = splat2(0.f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (k * nt + t < V) exp_vec<T>(raw[k], Lw == -INFINITY ? 0.f : -Lw, e[k], acc);
  }
  const float sw = group_sum<32>(acc.x + acc.y);
  if (lane == 0) red[parity][t >> 5] = make_float2(Lw, sw);
  __syncthreads();
  // Lane w of each 16-lane half takes warp w's pair; lanes past the CTA's
  // warps hold (-inf, 0), which change neither the max nor the sum.
  const int w = lane & (kMaxFitWarps - 1);
  const float2 q = w < (nt >> 5) ? red[parity][w] : make_float2(-INFINITY, 0.f);
  parity ^= 1;
  const float L = group_max<kMaxFitWarps>(q.x);
  const float S = group_sum<kMaxFitWarps>(q.y * exp2f(q.x - L));
  const float2 f = splat2(exp2f(Lw - L) * __frcp_rn(S));

#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * nt + t;
    if (i < V) {
      float2 o[P];
#pragma unroll
      for (int p = 0; p < P; ++p) o[p] = mul2(e[k][p], f);
      st_vec(y_row + i * VEC, pack2<T>(o));
    }
  }
}

template <typename T, int N>
__device__ __forceinline__ void smx_row_cta(const SmxArgs& a, int64_t row, uint32_t xrow,
                                            float2 (*red)[kMaxFitWarps], int& parity) {
  const int V = a.hidden / Vec<T>::N;
  uint4 raw[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int i = k * (int)blockDim.x + threadIdx.x;
    if (i < V) raw[k] = lds_u4(xrow + i * 16);
  }
  smx_row_cta_regs<T, N>(a, row, raw, red, parity);
}

// Rows a CTA of the CTA-per-row softmax takes: two while a thread's row
// share is at most four vectors (64 registers: still four CTAs per SM, so an
// SM has eight rows' loads in flight instead of four; 16384 x 8192 bf16:
// 80.3 against 82.8 us), one beyond.
template <int N>
constexpr int kSmxRowsPerCta = N <= 4 ? 2 : 1;

// Rows of more than 256 vectors straight from global memory into registers:
// a CTA loads all of its rows' vectors at once, then finishes each row in
// turn (as many CTAs as the rows need). The CTA's size is fitted to the row
// at launch (blockDim.x, a whole number of warps up to kMaxFitThreads).
template <typename T, int N>
__global__ void __launch_bounds__(kMaxFitThreads, N <= 4 ? 2 : 1) smx_reg_cta_kernel(const SmxArgs a) {
  constexpr int R = kSmxRowsPerCta<N>;
  __shared__ float2 red[2][kMaxFitWarps];
  constexpr int VEC = Vec<T>::N;
  const int V = a.hidden / VEC;
  uint4 raw[R][N];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = (int64_t)blockIdx.x * R + r;
    const T* x = static_cast<const T*>(a.x) + row * (int64_t)a.hidden;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int i = k * (int)blockDim.x + threadIdx.x;
      if (row < a.rows && i < V) raw[r][k] = ld_vec(x + i * VEC);
    }
  }
  int parity = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = (int64_t)blockIdx.x * R + r;
    if (row < a.rows) smx_row_cta_regs<T, N>(a, row, raw[r], red, parity);
  }
}

// CTAs of smx_reg_cta_kernel for `rows` rows of N vectors per thread.
inline int64_t smx_cta_grid(int64_t rows, int n) {
  const int r = n <= 4 ? 2 : 1;
  return (rows + r - 1) / r;
}

template <typename T, int LANES, int N>
__global__ void __launch_bounds__(kBulkThreads, N <= 3 ? 4 : (N == 4 ? 3 : 2)) smx_bulk_warp_kernel(const SmxArgs a,
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
__global__ void __launch_bounds__(kBulkThreads, N <= 4 ? 3 : 2) smx_bulk_cta_kernel(const SmxArgs a,
                                                                        const BulkCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float2 red[2][kMaxFitWarps];
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
        smx_row_cta<T, N>(a, row, smem_addr(slot), red, parity);
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
    const float nml = -cta_max_db<kScalarCta>(m, red, parity) * kLog2e;
    float s = 0.f;
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float e = exp2f(fmaf(srow[j], kLog2e, nml));
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
#define NF_SMX_REG(L)                                                   \
  switch (n) {                                                          \
    case 1: return (const void*)smx_reg_kernel<T, L, 1>;                \
    case 2: return (const void*)smx_reg_kernel<T, L, 2>;                \
    case 3: return (const void*)smx_reg_kernel<T, L, 3>;                \
    case 4: return (const void*)smx_reg_kernel<T, L, 4>;                \
    case 5: return (const void*)smx_reg_kernel<T, L, 5>;                \
    case 6: return (const void*)smx_reg_kernel<T, L, 6>;                \
    case 8: return (const void*)smx_reg_kernel<T, L, 8>;                \
    default: return nullptr;                                            \
  }
  if (kind == 0) {
    if (group == 8) { NF_SMX_WARP(8) }
    if (group == 16) { NF_SMX_WARP(16) }
    if (group == 32) { NF_SMX_WARP(32) }
  } else if (kind == 5) {
    switch (n) {
      case 2: return (const void*)smx_reg_cta_kernel<T, 2>;
      case 3: return (const void*)smx_reg_cta_kernel<T, 3>;
      case 4: return (const void*)smx_reg_cta_kernel<T, 4>;
      case 5: return (const void*)smx_reg_cta_kernel<T, 5>;
      case 6: return (const void*)smx_reg_cta_kernel<T, 6>;
      case 8: return (const void*)smx_reg_cta_kernel<T, 8>;
      default: return nullptr;
    }
  } else if (kind == 4) {
    if (group == 8) { NF_SMX_REG(8) }
    if (group == 16) { NF_SMX_REG(16) }
    if (group == 32) { NF_SMX_REG(32) }
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
#undef NF_SMX_REG
  return nullptr;
}

}  // namespace nf
