// Shared device helpers for the normalization kernels: 128-bit vector
// load/store, dtype <-> fp32 conversion, warp and CTA reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace nf {

using bf16 = __nv_bfloat16;
using f16 = __half;

// Block shapes shared by the kernels and the host-side planner.
constexpr int kScalarCta = 256;        // threads per CTA of the scalar kernels
constexpr int kConsumerWarps = 8;      // warps of a pipelined CTA
constexpr int kBulkThreads = kConsumerWarps * 32;
constexpr int kMaxFitThreads = 512;   // largest CTA of the row-fitted kernels
constexpr int kMaxFitWarps = kMaxFitThreads / 32;
// Threads of the prefetching CTA-per-row backward: two row groups of 256.
constexpr int kPfGroups = 2;
constexpr int kPfThreads = kPfGroups * kBulkThreads;

// Elements per 16-byte vector.
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<bf16> { static constexpr int N = 8; };
template <> struct Vec<f16> { static constexpr int N = 8; };

// Arguments of the forward kernels (validated on the host).
struct FwdArgs {
  const void* x;
  const void* bias;      // nullable
  const void* residual;  // nullable
  const void* gamma;
  const void* beta;      // nullable (always null for RMSNorm)
  void* out_sum;         // nullable
  void* y;
  float* mean;           // nullable (always null for RMSNorm)
  float* rstd;           // nullable
  unsigned* amax;        // nullable; fp32 bit pattern, zeroed before launch
  unsigned char* y_fp8;  // nullable; E4M3 codes of y * fp8_scale
  const float* fp8_scale;  // device scalar, required with y_fp8
  int64_t rows;
  int hidden;
  float eps;
  float inv_hidden;
  int rms;
  int zero_centered;
};

// Arguments of the backward kernels.
struct BwdArgs {
  const void* dy;
  const void* x_sum;
  const void* gamma;
  const float* mean;     // null for RMSNorm
  const float* rstd;
  void* dx;
  float* ws;             // [gridDim.x][ws_cols] partials: dgamma, then dbeta
                         // (LayerNorm), then dbias (when has_dbias), hidden each
  int64_t rows;
  int hidden;
  float inv_hidden;
  int rms;
  int zero_centered;
  int has_dbias;         // also accumulate dbias = sum over rows of dx
  int ws_cols;
};

// Arguments of the row softmax kernels.
struct SmxArgs {
  const void* x;
  void* y;               // may equal x (in place); no other overlap
  int64_t rows;
  int hidden;
};

// Launch parameters of the pipelined (bulk-copy) kernels.
struct BulkCfg {
  int stages;          // ring slots
  int tile_rows;       // rows per tile
  int64_t num_tiles;   // ceil(rows / tile_rows)
};

// ---- scalar conversions --------------------------------------------------
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(f16 v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ f16 from_f<f16>(float v) { return __float2half_rn(v); }

// ---- 16-byte vectors -----------------------------------------------------
// Read-only streaming load of 16 bytes (non-coherent path; inputs are never
// written by the same kernel).
__device__ __forceinline__ uint4 ld_vec(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
// L1-cached load for the small per-column vectors (gamma, beta, bias).
__device__ __forceinline__ uint4 ld_vec_param(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_vec(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Unpack a 16-byte vector of T into fp32.
template <typename T> __device__ __forceinline__ void unpack(const uint4& u, float* f);
template <> __device__ __forceinline__ void unpack<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
__device__ __forceinline__ void unpack_bf16x2(unsigned w, float* f) {
  f[0] = __uint_as_float(w << 16);
  f[1] = __uint_as_float(w & 0xffff0000u);
}
template <> __device__ __forceinline__ void unpack<bf16>(const uint4& u, float* f) {
  unpack_bf16x2(u.x, f); unpack_bf16x2(u.y, f + 2);
  unpack_bf16x2(u.z, f + 4); unpack_bf16x2(u.w, f + 6);
}
__device__ __forceinline__ void unpack_f16x2(unsigned w, float* f) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 v = __half22float2(h);
  f[0] = v.x; f[1] = v.y;
}
template <> __device__ __forceinline__ void unpack<f16>(const uint4& u, float* f) {
  unpack_f16x2(u.x, f); unpack_f16x2(u.y, f + 2);
  unpack_f16x2(u.z, f + 4); unpack_f16x2(u.w, f + 6);
}

// Pack fp32 values into a 16-byte vector of T, rounding to nearest even.
template <typename T> __device__ __forceinline__ uint4 pack(const float* f);
template <> __device__ __forceinline__ uint4 pack<float>(const float* f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                    __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ unsigned pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<unsigned*>(&h);
}
template <> __device__ __forceinline__ uint4 pack<bf16>(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ unsigned pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<unsigned*>(&h);
}
template <> __device__ __forceinline__ uint4 pack<f16>(const float* f) {
  return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]),
                    pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
}

// |v| as an fp32 bit pattern. For v >= 0 (and NaN with the sign cleared)
// unsigned order equals float order, so an unsigned max is an exact amax
// that also lets a NaN win, as torch.amax does.
__device__ __forceinline__ unsigned abs_bits(float v) {
  return __float_as_uint(v) & 0x7fffffffu;
}

// ---- fp32 pairs -------------------------------------------------------------
// sm_100-class GPUs issue two IEEE round-to-nearest fp32 adds, multiplies or
// fmas in one instruction on a register pair; the row bodies of the pipelined
// kernels keep their values as float2 pairs to use them.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// Unpack a 16-byte vector of T into Vec<T>::N / 2 fp32 pairs.
template <typename T> __device__ __forceinline__ void unpack2(const uint4& u, float2* f);
template <> __device__ __forceinline__ void unpack2<float>(const uint4& u, float2* f) {
  f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
  f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}
__device__ __forceinline__ float2 bf16x2_to_f2(unsigned w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ void unpack2<bf16>(const uint4& u, float2* f) {
  f[0] = bf16x2_to_f2(u.x); f[1] = bf16x2_to_f2(u.y);
  f[2] = bf16x2_to_f2(u.z); f[3] = bf16x2_to_f2(u.w);
}
__device__ __forceinline__ float2 f16x2_to_f2(unsigned w) {
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}
template <> __device__ __forceinline__ void unpack2<f16>(const uint4& u, float2* f) {
  f[0] = f16x2_to_f2(u.x); f[1] = f16x2_to_f2(u.y);
  f[2] = f16x2_to_f2(u.z); f[3] = f16x2_to_f2(u.w);
}

// Pack fp32 pairs into a 16-byte vector of T (round to nearest even).
template <typename T> __device__ __forceinline__ uint4 pack2(const float2* f);
template <> __device__ __forceinline__ uint4 pack2<float>(const float2* f) {
  return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                    __float_as_uint(f[1].x), __float_as_uint(f[1].y));
}
__device__ __forceinline__ unsigned f2_to_bf16x2(float2 v) {
  __nv_bfloat162 h = __float22bfloat162_rn(v);
  return *reinterpret_cast<unsigned*>(&h);
}
template <> __device__ __forceinline__ uint4 pack2<bf16>(const float2* f) {
  return make_uint4(f2_to_bf16x2(f[0]), f2_to_bf16x2(f[1]), f2_to_bf16x2(f[2]),
                    f2_to_bf16x2(f[3]));
}
__device__ __forceinline__ unsigned f2_to_f16x2(float2 v) {
  __half2 h = __float22half2_rn(v);
  return *reinterpret_cast<unsigned*>(&h);
}
template <> __device__ __forceinline__ uint4 pack2<f16>(const float2* f) {
  return make_uint4(f2_to_f16x2(f[0]), f2_to_f16x2(f[1]), f2_to_f16x2(f[2]), f2_to_f16x2(f[3]));
}

// FP8 E4M3 codes of VEC fp32 values times `scale` (fp32 product, round to
// nearest even, finite values saturate to +-448): VEC bytes at `dst`.
__device__ __forceinline__ unsigned short fp8x2(float2 v, float2 scale) {
  return __nv_cvt_float2_to_fp8x2(__fmul2_rn(v, scale), __NV_SATFINITE, __NV_E4M3);
}
template <int VEC>
__device__ __forceinline__ void store_fp8(unsigned char* dst, const float2* v, float scale);
template <>
__device__ __forceinline__ void store_fp8<8>(unsigned char* dst, const float2* v, float scale) {
  const float2 s2 = make_float2(scale, scale);
  const uint2 q = make_uint2((unsigned)fp8x2(v[0], s2) | ((unsigned)fp8x2(v[1], s2) << 16),
                             (unsigned)fp8x2(v[2], s2) | ((unsigned)fp8x2(v[3], s2) << 16));
  *reinterpret_cast<uint2*>(dst) = q;
}
template <>
__device__ __forceinline__ void store_fp8<4>(unsigned char* dst, const float2* v, float scale) {
  const float2 s2 = make_float2(scale, scale);
  *reinterpret_cast<unsigned*>(dst) = (unsigned)fp8x2(v[0], s2) | ((unsigned)fp8x2(v[1], s2) << 16);
}
// One value (scalar kernels).
__device__ __forceinline__ unsigned char fp8_one(float v, float scale) {
  return (unsigned char)(fp8x2(make_float2(v, 0.f), make_float2(scale, 1.f)) & 0xffu);
}

// Running amax over stored 16-byte vectors. For 16-bit types the
// accumulator holds two halves (|y| bit patterns compared as unsigned 16-bit
// lanes, which orders non-negative bf16/fp16 values like the values and lets
// NaN win); amax_bits<T>() turns it into the fp32 bit pattern of the max.
template <typename T> __device__ __forceinline__ void amax_update(unsigned& acc, const uint4& u);
template <> __device__ __forceinline__ void amax_update<float>(unsigned& acc, const uint4& u) {
  acc = max(acc, u.x & 0x7fffffffu);
  acc = max(acc, u.y & 0x7fffffffu);
  acc = max(acc, u.z & 0x7fffffffu);
  acc = max(acc, u.w & 0x7fffffffu);
}
__device__ __forceinline__ void amax_update_16(unsigned& acc, const uint4& u) {
  acc = __vmaxu2(acc, u.x & 0x7fff7fffu);
  acc = __vmaxu2(acc, u.y & 0x7fff7fffu);
  acc = __vmaxu2(acc, u.z & 0x7fff7fffu);
  acc = __vmaxu2(acc, u.w & 0x7fff7fffu);
}
template <> __device__ __forceinline__ void amax_update<bf16>(unsigned& acc, const uint4& u) {
  amax_update_16(acc, u);
}
template <> __device__ __forceinline__ void amax_update<f16>(unsigned& acc, const uint4& u) {
  amax_update_16(acc, u);
}
template <typename T> __device__ __forceinline__ unsigned amax_bits(unsigned acc);
template <> __device__ __forceinline__ unsigned amax_bits<float>(unsigned acc) { return acc; }
template <> __device__ __forceinline__ unsigned amax_bits<bf16>(unsigned acc) {
  return max(acc & 0xffffu, acc >> 16) << 16;   // bf16 bits are the top half of fp32 bits
}
template <> __device__ __forceinline__ unsigned amax_bits<f16>(unsigned acc) {
  const unsigned short m = (unsigned short)max(acc & 0xffffu, acc >> 16);
  return __float_as_uint(__half2float(__ushort_as_half(m)));
}

// ---- reductions ----------------------------------------------------------
// Butterfly sum over aligned groups of LANES lanes (LANES a power of two
// <= 32). Every lane of the warp must call it; each group gets its own sum.
template <int LANES> __device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int LANES> __device__ __forceinline__ float2 group_sum2(float2 v) {
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  return v;
}

// Butterfly max over aligned groups of LANES lanes (fmaxf: a NaN operand
// loses to a number, so a NaN in a row is caught later by exp(x - m) instead).
template <int LANES> __device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the CTA, same fixed order in every thread; returns the total to
// all threads. `red` holds one float per warp. Two barriers: the second one
// lets the caller reuse `red` right away.
template <int THREADS> __device__ __forceinline__ float cta_sum(float v, float* red) {
  constexpr int W = THREADS / 32;
  v = group_sum<32>(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < W; ++i) t += red[i];
  __syncthreads();
  return t;
}
template <int THREADS> __device__ __forceinline__ float2 cta_sum2(float2 v, float2* red) {
  constexpr int W = THREADS / 32;
  v = group_sum2<32>(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < W; ++i) { t.x += red[i].x; t.y += red[i].y; }
  __syncthreads();
  return t;
}

// The same sums with one barrier: `red` holds two buffers of one entry per
// warp and `parity` picks the buffer, flipping each call. A warp can write a
// buffer again only after the barrier of the call in between, which every
// warp reaches after it has read the buffer, so no second barrier is needed.
template <int THREADS>
__device__ __forceinline__ float cta_sum_db(float v, float (*red)[THREADS / 32], int& parity) {
  constexpr int W = THREADS / 32;
  v = group_sum<32>(v);
  if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < W; ++i) t += red[parity][i];
  parity ^= 1;
  return t;
}
template <int THREADS>
__device__ __forceinline__ float2 cta_sum2_db(float2 v, float2 (*red)[THREADS / 32], int& parity) {
  constexpr int W = THREADS / 32;
  v = group_sum2<32>(v);
  if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < W; ++i) {
    t.x += red[parity][i].x;
    t.y += red[parity][i].y;
  }
  parity ^= 1;
  return t;
}

// cta_sum_db for a CTA of any whole number of warps up to kMaxFitWarps
// (blockDim.x chosen at launch): the warps' sums added in warp order.
__device__ __forceinline__ float cta_sum_db_fit(float v, float (*red)[kMaxFitWarps], int& parity) {
  const int W = blockDim.x >> 5;
  v = group_sum<32>(v);
  if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll 4
  for (int i = 0; i < W; ++i) t += red[parity][i];
  parity ^= 1;
  return t;
}

__device__ __forceinline__ float2 cta_sum2_db_fit(float2 v, float2 (*red)[kMaxFitWarps],
                                                  int& parity) {
  const int W = blockDim.x >> 5;
  v = group_sum2<32>(v);
  if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int i = 0; i < W; ++i) {
    t.x += red[parity][i].x;
    t.y += red[parity][i].y;
  }
  parity ^= 1;
  return t;
}

// Max over the CTA with one barrier (double buffer and parity as above).
template <int THREADS>
__device__ __forceinline__ float cta_max_db(float v, float (*red)[THREADS / 32], int& parity) {
  constexpr int W = THREADS / 32;
  v = group_max<32>(v);
  if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[parity][0];
#pragma unroll
  for (int i = 1; i < W; ++i) t = fmaxf(t, red[parity][i]);
  parity ^= 1;
  return t;
}

// Max of per-thread amax bits over the CTA, then one atomicMax per CTA on
// the fp32 bit pattern in global memory (the partial-then-final split of the
// amax reduction). Must be called by all threads of the CTA.
__device__ __forceinline__ void cta_amax_commit(unsigned bits, unsigned* amax, unsigned* red) {
  bits = __reduce_max_sync(0xffffffffu, bits);
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = bits;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned m = 0;
    for (int i = 0; i < nw; ++i) m = max(m, red[i]);
    atomicMax(amax, m);
  }
}

}  // namespace nf
