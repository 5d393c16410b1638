// Backward kernels of the fused block (pytorch/pytorch PR 165370).
//
// An RMS/Layer norm backward has two kinds of reduction over the same inputs
// (dy, x_sum and the per-row statistics): dx reduces over the hidden
// dimension of one row, dgamma/dbeta over all rows. Here one persistent
// kernel does both in a single read of the inputs: each row stays on chip
// (the "persistent reduction" the PR requires) while its dx is formed, and
// the row's dy * xhat and dy are added into per-thread fp32 accumulators (the
// outer reduction turned into a partial accumulation). At the end each CTA
// writes its partial dgamma/dbeta row to the workspace, and the finalize
// kernel adds the partials of all CTAs in a fixed order.
//
// The row -> CTA assignment is a grid-stride loop over a grid sized from the
// SM count, so the partials, and the finalize's fixed-order compensated sum
// over them, are the same on every run.
//
//  * bwd_row_cta_kernel (default for rows of more than 256 vectors whose
//    accumulators and row fit in registers at three CTAs per SM: bf16/fp16
//    RMSNorm up to 8192, LayerNorm up to 4096): the row straight from global
//    memory into registers, a CTA per row.
//  * bwd_bulk_warp_kernel / bwd_bulk_group_kernel / bwd_bulk_cta_kernel
//    (the other 16-byte aligned rows, and all of them when a test selects the
//    ring family through ln_testing_select_kernels):
//    dy and x_sum tiles stream into a shared-memory ring by
//    cp.async.bulk; the row is read from shared memory twice (sums, then dx)
//    instead of being held in registers, and w = gamma (+1) sits in shared
//    memory as fp32.
//  * bwd_scalar_kernel: any hidden size and alignment.
#pragma once

#include "bulk.cuh"
#include "common.cuh"
#include "fwd_kernels.cuh"

namespace nf {

// The row body of the pipelined kernels: dy and x_sum rows in shared memory,
// w = gamma (+1) staged in shared memory (kStaged), read from global, or
// (kWReg) held in registers: a thread covers the same columns in every row,
// so `wreg` is loaded once per kernel. The second pass reads shared memory
// again, so only the accumulators (and wreg) stay in registers across the
// reduction, except that the first kKeep vectors keep their (x - mean) and
// g = dy * w from the first pass (registers the kernel has to spare; the same
// values either way). Values are fp32 pairs (packed fp32 math). kRms drops
// the mean, c1 and the dbeta accumulators at compile time; kBias adds the
// row's fp32 dx into the dbias accumulators. The row means c1 and c2 are the
// row sums times the fp32 reciprocal of the width (a multiply instead of a
// division per row). Each vector slot of either pass is skipped as a whole
// when it lies past the row (or the tile has no row for this group), so the
// compiler keeps a slot's loads next to their use. kExact: the row has
// exactly G * N vectors, so no slot lies past it.
template <typename T, int G, int N, bool kRms, bool kBias, bool kStaged, bool kWReg, int kKeep,
          bool kExact, typename Reduce2>
__device__ __forceinline__ void bwd_row_smem(const BwdArgs& a, int64_t row, bool row_ok, int t,
                                             uint32_t dyrow, uint32_t xsrow, const ParamRow<T>& wr,
                                             const float2 (&wreg)[N][Vec<T>::N / 2],
                                             float mean, float rstd, Reduce2 reduce2,
                                             float2 (&acc_g)[N][Vec<T>::N / 2],
                                             float2 (&acc_b)[N][Vec<T>::N / 2],
                                             float2 (&acc_d)[N][Vec<T>::N / 2]) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int H = kExact ? G * N * VEC : a.hidden;
  const int V = kExact ? G * N : H / VEC;
  const float2 neg_mean = splat2(-mean);
  const float2 r2 = splat2(rstd);
  const uint32_t wa = kStaged ? wr.saddr() : 0u;
  float2 sx = splat2(0.f), sy = splat2(0.f);
  constexpr int KK = kKeep > 0 ? kKeep : 1;
  float2 keep_xm[KK][P], keep_g[KK][P];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (!row_ok || (!kExact && v >= V)) continue;
    float2 d[P], xv[P], w[P];
    unpack2<T>(lds_u4(dyrow + v * 16), d);
    unpack2<T>(lds_u4(xsrow + v * 16), xv);
    if (kWReg) {
#pragma unroll
      for (int i = 0; i < P; ++i) w[i] = wreg[k][i];
    } else {
      wr.template load2<kStaged>(v, w, wa);
    }
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float2 xm = kRms ? xv[i] : add2(xv[i], neg_mean);
      const float2 xh = mul2(xm, r2);
      const float2 g = mul2(d[i], w[i]);
      if (k < kKeep) {
        keep_xm[k < kKeep ? k : 0][i] = xm;
        keep_g[k < kKeep ? k : 0][i] = g;
      }
      if (!kRms) sx = add2(sx, g);
      sy = fma2(g, xh, sy);
      acc_g[k][i] = fma2(d[i], xh, acc_g[k][i]);
      if (!kRms) acc_b[k][i] = add2(acc_b[k][i], d[i]);
    }
  }
  const float2 sums = reduce2(make_float2(sx.x + sx.y, sy.x + sy.y));
  // dx = rstd * (g - c1 - xhat * c2) = (x - mean) * b2 + (g * rstd + a1)
  const float c2 = sums.y * a.inv_hidden;
  const float2 a1 = splat2(kRms ? 0.f : -rstd * (sums.x * a.inv_hidden));
  const float2 b2 = splat2(-rstd * rstd * c2);
  asm volatile("" ::: "memory");   // the second pass reads shared memory again

  T* dx = static_cast<T*>(a.dx) + row * (int64_t)H;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (!row_ok || (!kExact && v >= V)) continue;
    float2 o[P];
    if (k < kKeep) {
#pragma unroll
      for (int i = 0; i < P; ++i)
        o[i] = fma2(keep_xm[k < kKeep ? k : 0][i], b2, fma2(keep_g[k < kKeep ? k : 0][i], r2, a1));
    } else {
      float2 d[P], xv[P], w[P];
      unpack2<T>(lds_u4(dyrow + v * 16), d);
      unpack2<T>(lds_u4(xsrow + v * 16), xv);
      if (kWReg) {
#pragma unroll
        for (int i = 0; i < P; ++i) w[i] = wreg[k][i];
      } else {
        wr.template load2<kStaged>(v, w, wa);
      }
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float2 xm = kRms ? xv[i] : add2(xv[i], neg_mean);
        o[i] = fma2(xm, b2, fma2(mul2(d[i], w[i]), r2, a1));
      }
    }
    if (kBias) {
#pragma unroll
      for (int i = 0; i < P; ++i) acc_d[k][i] = add2(acc_d[k][i], o[i]);
    }
    st_vec(dx + v * VEC, pack2<T>(o));
  }
}

template <typename T, int N>
__device__ __forceinline__ void zero_acc2(float2 (&acc)[N][Vec<T>::N / 2]) {
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int i = 0; i < Vec<T>::N / 2; ++i) acc[k][i] = splat2(0.f);
}

// The pipelined kernels' partials: the pair accumulators as plain floats.
template <typename T, int N>
__device__ __forceinline__ void unpair_acc(const float2 (&p)[N][Vec<T>::N / 2],
                                           float (&f)[N][Vec<T>::N]) {
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int i = 0; i < Vec<T>::N / 2; ++i) {
      f[k][2 * i] = p[k][i].x;
      f[k][2 * i + 1] = p[k][i].y;
    }
}

// Column offset of each partial row in the workspace: dgamma at 0, dbeta
// at hidden (LayerNorm), dbias after them.
__device__ __forceinline__ int partial_offset(const BwdArgs& a, int which) {
  if (which == 0) return 0;
  if (which == 1) return a.hidden;
  return a.rms ? a.hidden : 2 * a.hidden;
}

// Partials of a lane-group kernel: W warps, each with 32 / LANES groups that
// hold the same columns. Groups of a warp are added by a fixed butterfly,
// then the warps through shared memory in warp order. Slot k of a warp covers
// columns [k * LANES * VEC, (k + 1) * LANES * VEC). When `buf` (the ring's
// slots, idle once the pipeline has drained) holds every warp's N slots, a
// sum goes through it in one step, two barriers per sum; otherwise one slot
// at a time through `red` (two barriers per slot and sum). Both add the same
// values in the same order. All threads of the CTA call this (threads of
// warps >= W only pass barriers). Accumulators: 0 = dgamma, 1 = dbeta
// (LayerNorm), 2 = dbias (kBias).
template <typename T, int LANES, int N, int W, bool kRms, bool kBias>
__device__ __forceinline__ void store_group_partials(const BwdArgs& a,
                                                     float (&acc_g)[N][Vec<T>::N],
                                                     float (&acc_b)[N][Vec<T>::N],
                                                     float (&acc_d)[N][Vec<T>::N],
                                                     float (*red)[LANES * Vec<T>::N],
                                                     float* buf, size_t buf_bytes) {
  constexpr int VEC = Vec<T>::N;
  constexpr int SLOT = LANES * VEC;
  constexpr int NS = N * SLOT;   // columns a warp holds
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane / LANES;
  const int l = lane % LANES;
  const bool rms = kRms || a.rms;
  if (warp < W) {
#pragma unroll
    for (int o = LANES; o < 32; o <<= 1)
#pragma unroll
      for (int k = 0; k < N; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          acc_g[k][e] += __shfl_xor_sync(0xffffffffu, acc_g[k][e], o);
          if (!kRms) acc_b[k][e] += __shfl_xor_sync(0xffffffffu, acc_b[k][e], o);
          if (kBias) acc_d[k][e] += __shfl_xor_sync(0xffffffffu, acc_d[k][e], o);
        }
  }
  const int H = a.hidden;
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  const bool whole = (size_t)W * NS * sizeof(float) <= buf_bytes;
  for (int which = 0; which < 3; ++which) {
    if (which == 1 && (kRms || rms)) continue;
    if (which == 2 && !kBias) continue;
    const int off = partial_offset(a, which);
    if (whole) {
      if (warp < W && sub == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            buf[warp * NS + k * SLOT + l * VEC + e] =
                which == 0 ? acc_g[k][e] : (which == 1 ? acc_b[k][e] : acc_d[k][e]);
      }
      __syncthreads();
      for (int col = threadIdx.x; col < H; col += blockDim.x) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) t += buf[w * NS + col];
        ws[off + col] = t;
      }
      __syncthreads();
      continue;
    }
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (warp < W && sub == 0) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          red[warp][l * VEC + e] = which == 0 ? acc_g[k][e] : (which == 1 ? acc_b[k][e] : acc_d[k][e]);
      }
      __syncthreads();
      for (int c = threadIdx.x; c < SLOT; c += blockDim.x) {
        const int col = k * SLOT + c;
        if (col < H) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) t += red[w][c];
          ws[off + col] = t;
        }
      }
      __syncthreads();
    }
  }
}

// Partials of a CTA-per-row kernel: every column belongs to one thread.
template <typename T, int G, int N, bool kRms, bool kBias>
__device__ __forceinline__ void store_thread_partials(const BwdArgs& a, int t,
                                                      float (&acc_g)[N][Vec<T>::N],
                                                      float (&acc_b)[N][Vec<T>::N],
                                                      float (&acc_d)[N][Vec<T>::N]) {
  constexpr int VEC = Vec<T>::N;
  const bool rms = kRms || a.rms;
  const int H = a.hidden;
  const int V = H / VEC;
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  const int off_d = partial_offset(a, 2);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int v = k * G + t;
    if (v < V) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        ws[v * VEC + e] = acc_g[k][e];
        if (!rms) ws[H + v * VEC + e] = acc_b[k][e];
        if (kBias) ws[off_d + v * VEC + e] = acc_d[k][e];
      }
    }
  }
}

// Partials of a row-group kernel: 256 / G groups of G threads (G = 64 or
// 128), thread t of every group holding the same columns (vectors k * G + t).
// The groups are added through shared memory in group order: through `buf`
// (the drained ring's slots) in one step per sum when it holds every group's
// N slots, else one vector slot (G * VEC columns) at a time through `red`;
// the same values in the same order either way. All threads of the CTA call
// this.
template <typename T, int G, int N, bool kRms, bool kBias>
__device__ __forceinline__ void store_rowgroup_partials(const BwdArgs& a,
                                                        float (&acc_g)[N][Vec<T>::N],
                                                        float (&acc_b)[N][Vec<T>::N],
                                                        float (&acc_d)[N][Vec<T>::N],
                                                        float (*red)[G * Vec<T>::N],
                                                        float* buf, size_t buf_bytes) {
  constexpr int VEC = Vec<T>::N;
  constexpr int SLOT = G * VEC;
  constexpr int NS = N * SLOT;   // columns a group holds
  constexpr int NG = kBulkThreads / G;
  const int grp = threadIdx.x / G;
  const int t = threadIdx.x % G;
  const bool rms = kRms || a.rms;
  const int H = a.hidden;
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  const bool whole = (size_t)NG * NS * sizeof(float) <= buf_bytes;
  for (int which = 0; which < 3; ++which) {
    if (which == 1 && rms) continue;
    if (which == 2 && !kBias) continue;
    const int off = partial_offset(a, which);
    if (whole) {
#pragma unroll
      for (int k = 0; k < N; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          buf[grp * NS + k * SLOT + t * VEC + e] =
              which == 0 ? acc_g[k][e] : (which == 1 ? acc_b[k][e] : acc_d[k][e]);
      __syncthreads();
      for (int col = threadIdx.x; col < H; col += kBulkThreads) {
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) s += buf[g * NS + col];
        ws[off + col] = s;
      }
      __syncthreads();
      continue;
    }
#pragma unroll
    for (int k = 0; k < N; ++k) {
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        red[grp][t * VEC + e] = which == 0 ? acc_g[k][e] : (which == 1 ? acc_b[k][e] : acc_d[k][e]);
      __syncthreads();
      for (int c = threadIdx.x; c < SLOT; c += kBulkThreads) {
        const int col = k * SLOT + c;
        if (col < H) {
          float s = 0.f;
#pragma unroll
          for (int g = 0; g < NG; ++g) s += red[g][c];
          ws[off + col] = s;
        }
      }
      __syncthreads();
    }
  }
}

// ---- bulk-copy pipelined kernels ------------------------------------------

// Vectors per lane whose first-pass values the lane-group backward keeps for
// the second pass: one for 16-bit LayerNorm rows of three vectors per lane
// (384 wide with 16 lanes: 106 -> 118 registers, still two CTAs per SM;
// 228 -> 221 us at 576000 rows; keeping two vectors, 125 registers, took
// 253 us), none for the shapes where it was not measured.
template <typename T, int N, bool kRms, bool kBias>
constexpr int kKeepWarp = (sizeof(T) == 2 && !kRms && !kBias && N == 3) ? 1 : 0;

// kExact: the row has exactly LANES * N vectors (the planner's usual fit).
template <typename T, int LANES, int N, bool kRms, bool kBias, bool kExact>
__global__ void __launch_bounds__(kBulkThreads, 2) bwd_bulk_warp_kernel(const BwdArgs a,
                                                                         const BulkCfg c) {
  constexpr int RPW = 32 / LANES;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[kConsumerWarps][LANES * Vec<T>::N];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const uint32_t in_bytes = (uint32_t)c.tile_rows * H * sizeof(T);
  const Ring ring = make_ring(smem, 2 * in_bytes, c.stages);
  float* w_s = reinterpret_cast<float*>(ring.after);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  const ParamRow<T> wr = {w_s, static_cast<const T*>(a.gamma), H, a.zero_centered != 0};
  stage_param_row<T>(wr.g, H, wr.plus_one, w_s);
  ring_init(ring);

  const int lane = threadIdx.x & 31;
  const int l = lane % LANES;
  const int local = (threadIdx.x >> 5) * RPW + lane / LANES;   // row within the tile
  float2 wreg[N][Vec<T>::N / 2];   // unused: w is staged in shared memory
  float2 acc_g[N][Vec<T>::N / 2], acc_b[N][Vec<T>::N / 2], acc_d[N][Vec<T>::N / 2];
  zero_acc2<T, N>(acc_g);
  zero_acc2<T, N>(acc_b);
  zero_acc2<T, N>(acc_d);
  // Statistics of this group's row in a tile, loaded one tile ahead (a
  // tile past the last one has no row below a.rows).
  auto load_stats = [&](int64_t tile, float& m, float& r) {
    const int64_t row = tile * c.tile_rows + local;
    m = 0.f;
    r = 0.f;
    if (row < a.rows) {
      r = a.rstd[row];
      if (!kRms) m = a.mean[row];
    }
  };
  float nm, nr;
  load_stats(blockIdx.x, nm, nr);
  bool aborted = false;
  const int64_t taken = run_pipeline<false, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.dy), static_cast<const T*>(a.x_sum), aborted,
      [&](int64_t tile, unsigned char* slot) {
        const float mean = nm, rstd = nr;
        load_stats(tile + gridDim.x, nm, nr);
        const int64_t row = tile * c.tile_rows + local;
        const uint32_t dys = smem_addr(slot) + (uint32_t)(local * H * sizeof(T));
        const uint32_t xss = dys + in_bytes;
        bwd_row_smem<T, LANES, N, kRms, kBias, true, false, kKeepWarp<T, N, kRms, kBias>, kExact>(
            a, row, row < a.rows, l, dys, xss, wr, wreg, mean, rstd,
            [](float2 v) { return group_sum2<LANES>(v); }, acc_g, acc_b, acc_d);
      });
  allow_dependent_launch();
  if (pipeline_finish(ring, aborted, taken, &s_abort, &s_taken)) return;
  float fg[N][Vec<T>::N], fb[N][Vec<T>::N], fd[N][Vec<T>::N];
  unpair_acc<T, N>(acc_g, fg);
  unpair_acc<T, N>(acc_b, fb);
  unpair_acc<T, N>(acc_d, fd);
  // The ring's slots are idle now: every issued copy has landed and been
  // consumed (an aborted pipeline returned above).
  store_group_partials<T, LANES, N, kConsumerWarps, kRms, kBias>(
      a, fg, fb, fd, red, reinterpret_cast<float*>(ring.base),
      (size_t)ring.stages * ring.slot_bytes);
}

// Whether the CTA-per-row backward keeps w in registers: its accumulators
// take N * VEC floats per reduction (dgamma; dbeta for LayerNorm; dbias).
template <typename T, int N, bool kRms, bool kBias>
constexpr bool kWRegCta = N * Vec<T>::N * (1 + (kRms ? 0 : 1) + (kBias ? 1 : 0)) <= 32;

// Rows of two or four warps (G = 64 or 128 threads per row; 256 / G rows
// per tile): for widths whose lane-group accumulators would not fit in
// registers (LayerNorm from 6 vectors per lane, with dbias from 4), without
// the one-row-per-CTA-step latency of the CTA-per-row kernel. The row sums
// are added across the group's warps through shared memory behind a named
// barrier of the group's threads; w is staged in shared memory as fp32.
// Bodies synchronise within groups, so the loop runs in the uniform mode
// (a thread whose wait timed out still runs the body; its group leaves
// together after it, and every other group at its own next check).
template <typename T, int G, int N, bool kRms, bool kBias>
__global__ void __launch_bounds__(kBulkThreads, 2) bwd_bulk_group_kernel(const BwdArgs a,
                                                                          const BulkCfg c) {
  static_assert(G == 64 || G == 128, "row groups of two or four warps");
  constexpr int WPR = G / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[kBulkThreads / G][G * Vec<T>::N];
  __shared__ float2 xch[2][kConsumerWarps];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const uint32_t in_bytes = (uint32_t)c.tile_rows * H * sizeof(T);
  const Ring ring = make_ring(smem, 2 * in_bytes, c.stages);
  float* w_s = reinterpret_cast<float*>(ring.after);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  const ParamRow<T> wr = {w_s, static_cast<const T*>(a.gamma), H, a.zero_centered != 0};
  stage_param_row<T>(wr.g, H, wr.plus_one, w_s);
  ring_init(ring);

  const int local = threadIdx.x / G;   // row within the tile
  const int t = threadIdx.x % G;
  const int warp = threadIdx.x >> 5;
  float2 wreg[N][Vec<T>::N / 2];   // unused: w is staged in shared memory
  float2 acc_g[N][Vec<T>::N / 2], acc_b[N][Vec<T>::N / 2], acc_d[N][Vec<T>::N / 2];
  zero_acc2<T, N>(acc_g);
  zero_acc2<T, N>(acc_b);
  zero_acc2<T, N>(acc_d);
  auto load_stats = [&](int64_t tile, float& m, float& r) {
    const int64_t row = tile * c.tile_rows + local;
    m = 0.f;
    r = 0.f;
    if (row < a.rows) {
      r = a.rstd[row];
      if (!kRms) m = a.mean[row];
    }
  };
  // Sum of a float2 over the group: warp butterfly, then the group's warps
  // in order through a double-buffered exchange (one barrier per call).
  int parity = 0;
  auto row_sum = [&](float2 v) {
    v = group_sum2<32>(v);
    if ((threadIdx.x & 31) == 0) xch[parity][warp] = v;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + local), "r"(G) : "memory");
    float2 s = xch[parity][local * WPR];
#pragma unroll
    for (int i = 1; i < WPR; ++i) {
      s.x += xch[parity][local * WPR + i].x;
      s.y += xch[parity][local * WPR + i].y;
    }
    parity ^= 1;
    return s;
  };
  float nm, nr;
  load_stats(blockIdx.x, nm, nr);
  bool aborted = false;
  const int64_t taken = run_pipeline<true, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.dy), static_cast<const T*>(a.x_sum), aborted,
      [&](int64_t tile, unsigned char* slot) {
        const float mean = nm, rstd = nr;
        load_stats(tile + gridDim.x, nm, nr);
        const int64_t row = tile * c.tile_rows + local;
        const uint32_t dys = smem_addr(slot) + (uint32_t)(local * H * sizeof(T));
        const uint32_t xss = dys + in_bytes;
        bwd_row_smem<T, G, N, kRms, kBias, true, false, 0, false>(a, row, row < a.rows, t, dys, xss, wr,
                                                        wreg, mean, rstd, row_sum, acc_g,
                                                        acc_b, acc_d);
      });
  allow_dependent_launch();
  if (pipeline_finish(ring, aborted, taken, &s_abort, &s_taken)) return;
  float fg[N][Vec<T>::N], fb[N][Vec<T>::N], fd[N][Vec<T>::N];
  unpair_acc<T, N>(acc_g, fg);
  unpair_acc<T, N>(acc_b, fb);
  unpair_acc<T, N>(acc_d, fd);
  store_rowgroup_partials<T, G, N, kRms, kBias>(a, fg, fb, fd, red,
                                                reinterpret_cast<float*>(ring.base),
                                                (size_t)ring.stages * ring.slot_bytes);
}

template <typename T, int N, bool kRms, bool kBias>
__global__ void __launch_bounds__(kBulkThreads, 2)
    bwd_bulk_cta_kernel(const BwdArgs a, const BulkCfg c) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float2 red[2][kConsumerWarps];
  __shared__ int s_abort;
  __shared__ long long s_taken;
  const int H = a.hidden;
  const uint32_t in_bytes = (uint32_t)H * sizeof(T);   // one row per tile
  const Ring ring = make_ring(smem, 2 * in_bytes, c.stages);
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_taken = 0x7fffffffffffffffll;
  }
  const ParamRow<T> wr = {nullptr, static_cast<const T*>(a.gamma), H, a.zero_centered != 0};
  // w in registers when the accumulators leave room for it.
  constexpr bool kWReg = kWRegCta<T, N, kRms, kBias>;
  float2 wreg[N][Vec<T>::N / 2];
  if (kWReg) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * kBulkThreads + threadIdx.x;
      if (v < H / Vec<T>::N) wr.template load2<false>(v, wreg[k]);
    }
  }
  ring_init(ring);

  float2 acc_g[N][Vec<T>::N / 2], acc_b[N][Vec<T>::N / 2], acc_d[N][Vec<T>::N / 2];
  zero_acc2<T, N>(acc_g);
  zero_acc2<T, N>(acc_b);
  zero_acc2<T, N>(acc_d);
  auto load_stats = [&](int64_t row, float& m, float& r) {
    m = 0.f;
    r = 0.f;
    if (row < a.rows) {
      r = a.rstd[row];
      if (!kRms) m = a.mean[row];
    }
  };
  float nm, nr;
  load_stats(blockIdx.x, nm, nr);
  bool aborted = false;
  int parity = 0;
  const int64_t taken = run_pipeline<true, T>(
      ring, c, a.rows, H, static_cast<const T*>(a.dy), static_cast<const T*>(a.x_sum), aborted,
      [&](int64_t row, unsigned char* slot) {
        const float mean = nm, rstd = nr;
        load_stats(row + gridDim.x, nm, nr);
        const uint32_t dys = smem_addr(slot);
        const uint32_t xss = dys + in_bytes;
        bwd_row_smem<T, kBulkThreads, N, kRms, kBias, false, kWReg, 0, false>(
            a, row, true, threadIdx.x, dys, xss, wr, wreg, mean, rstd,
            [&](float2 v) { return cta_sum2_db<kBulkThreads>(v, red, parity); }, acc_g, acc_b,
            acc_d);
      });
  allow_dependent_launch();
  if (pipeline_finish(ring, aborted, taken, &s_abort, &s_taken)) return;
  float fg[N][Vec<T>::N], fb[N][Vec<T>::N], fd[N][Vec<T>::N];
  unpair_acc<T, N>(acc_g, fg);
  unpair_acc<T, N>(acc_b, fb);
  unpair_acc<T, N>(acc_d, fd);
  store_thread_partials<T, kBulkThreads, N, kRms, kBias>(a, threadIdx.x, fg, fb, fd);
}

// ---- register backward, one CTA per row ------------------------------------

// An empty asm statement that claims to rewrite N 16-byte vectors held in
// registers, so the compiler re-unpacks them where they are used instead of
// keeping the fp32 values live across the row sum (twice the registers).
template <int N>
__device__ __forceinline__ void vec_fence(uint4 (&q)[N]) {
#pragma unroll
  for (int k = 0; k < N; ++k)
    asm volatile("" : "+r"(q[k].x), "+r"(q[k].y), "+r"(q[k].z), "+r"(q[k].w));
}

// The row loop of bwd_row_cta_kernel; kZc adds 1 to gamma (zero-centered
// gamma) at compile time, so the loop carries no per-element branch.
template <typename T, int N, bool kRms, bool kBias, bool kZc>
__device__ __forceinline__ void row_cta_rows(const BwdArgs& a, float2 (*red)[kConsumerWarps],
                                             float2 (&acc_g)[N][Vec<T>::N / 2],
                                             float2 (&acc_b)[N][Vec<T>::N / 2],
                                             float2 (&acc_d)[N][Vec<T>::N / 2]) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  const int t = threadIdx.x;
  const int H = a.hidden;
  const int V = H / VEC;
  const T* gamma = static_cast<const T*>(a.gamma);
  const T* dy = static_cast<const T*>(a.dy);
  const T* xs = static_cast<const T*>(a.x_sum);
  T* dx = static_cast<T*>(a.dx);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t off = row * (int64_t)H;
    uint4 dr[N], xr[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * kBulkThreads + t;
      if (v < V) {
        dr[k] = ld_vec(dy + off + v * VEC);
        xr[k] = ld_vec(xs + off + v * VEC);
      }
    }
    const float rstd = a.rstd[row];
    const float mean = kRms ? 0.f : a.mean[row];
    const float2 neg_mean = splat2(-mean);
    const float2 r2 = splat2(rstd);
    float2 sx = splat2(0.f), sy = splat2(0.f);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * kBulkThreads + t;
      if (v < V) {
        float2 d[P], xv[P], w[P];
        unpack2<T>(dr[k], d);
        unpack2<T>(xr[k], xv);
        unpack2<T>(ld_vec_param(gamma + v * VEC), w);
#pragma unroll
        for (int i = 0; i < P; ++i) {
          if (kZc) w[i] = add2(w[i], splat2(1.f));
          const float2 xh = mul2(kRms ? xv[i] : add2(xv[i], neg_mean), r2);
          const float2 g = mul2(d[i], w[i]);
          if (!kRms) sx = add2(sx, g);
          sy = fma2(g, xh, sy);
          acc_g[k][i] = fma2(d[i], xh, acc_g[k][i]);
          if (!kRms) acc_b[k][i] = add2(acc_b[k][i], d[i]);
        }
      }
    }
    const float2 sums = cta_sum2_db<kBulkThreads>(
        make_float2(kRms ? 0.f : sx.x + sx.y, sy.x + sy.y), red, parity);
    // dx = rstd * (g - c1 - xhat * c2) = (x - mean) * b2 + (g * rstd + a1)
    const float c2 = sums.y * a.inv_hidden;
    const float2 a1 = splat2(kRms ? 0.f : -rstd * (sums.x * a.inv_hidden));
    const float2 b2 = splat2(-rstd * rstd * c2);
    vec_fence<N>(dr);
    vec_fence<N>(xr);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * kBulkThreads + t;
      if (v < V) {
        float2 d[P], xv[P], w[P], o[P];
        unpack2<T>(dr[k], d);
        unpack2<T>(xr[k], xv);
        unpack2<T>(ld_vec_param(gamma + v * VEC), w);
#pragma unroll
        for (int i = 0; i < P; ++i) {
          if (kZc) w[i] = add2(w[i], splat2(1.f));
          const float2 gr = kRms ? mul2(mul2(d[i], w[i]), r2)
                                 : fma2(mul2(d[i], w[i]), r2, a1);
          o[i] = fma2(kRms ? xv[i] : add2(xv[i], neg_mean), b2, gr);
          if (kBias) acc_d[k][i] = add2(acc_d[k][i], o[i]);
        }
        st_vec(dx + off + v * VEC, pack2<T>(o));
      }
    }
  }
}

// Rows of more than 256 vectors, straight from global memory into registers
// (N 16-byte vectors per thread, 256 threads per row): the CTAs of one wave
// step through the rows (row blockIdx.x + k * gridDim.x), so the partial row
// of CTA b sums a fixed set of rows and the sums depend only on the grid.
// gamma is read through L1 in both passes (it is the same for every row),
// the row sums go through a double-buffered CTA exchange with one barrier,
// and each thread owns the same columns in every row, so its dgamma / dbeta
// / dbias sums stay in registers until the end.
template <typename T, int N, bool kRms, bool kBias>
__global__ void __launch_bounds__(kBulkThreads, 3) bwd_row_cta_kernel(const BwdArgs a) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  __shared__ float2 red[2][kConsumerWarps];
  float2 acc_g[N][P], acc_b[N][P], acc_d[N][P];
  zero_acc2<T, N>(acc_g);
  zero_acc2<T, N>(acc_b);
  zero_acc2<T, N>(acc_d);
  if (a.zero_centered) {
    row_cta_rows<T, N, kRms, kBias, true>(a, red, acc_g, acc_b, acc_d);
  } else {
    row_cta_rows<T, N, kRms, kBias, false>(a, red, acc_g, acc_b, acc_d);
  }
  allow_dependent_launch();
  // Partials: every column belongs to one thread; fp32 pairs go out as
  // 16-byte stores (dgamma at 0, dbeta at H, dbias after them).
  const int H = a.hidden;
  const int V = H / VEC;
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  auto put = [&](const float2 (&acc)[N][P], int off) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * kBulkThreads + threadIdx.x;
      if (v < V) {
        float4* q = reinterpret_cast<float4*>(ws + off + v * VEC);
#pragma unroll
        for (int i = 0; i < P / 2; ++i)
          q[i] = make_float4(acc[k][2 * i].x, acc[k][2 * i].y, acc[k][2 * i + 1].x,
                             acc[k][2 * i + 1].y);
      }
    }
  };
  put(acc_g, 0);
  if (!kRms) put(acc_b, H);
  if (kBias) put(acc_d, kRms ? H : 2 * H);
}

// The same rows with the next row's dy and x_sum (and statistics) loaded
// into registers while this row is worked on. A CTA holds G row groups of
// GT threads: two groups of 256, or of 128 or 64 for rows of up to 512 or
// 256 vectors (two or four CTAs per SM); one group of 320 to 512 for wider
// rows (and for 16-bit LayerNorm rows of 1024 vectors, at two vectors a
// thread). Group g of CTA b takes rows G b + g, G b + g + G C, ... (C
// CTAs), so each group keeps two rows in flight.
// Each group sums its row behind a named barrier of its own threads, so the
// groups never wait for each other inside the row loop. w = gamma (+1 for
// zero-centered gamma) is staged once per kernel in shared memory as fp32
// ([k][pair of float2][thread] float4: no bank conflicts), which saves the
// per-row unpacking of gamma. At the end two groups' column sums are added
// (group 0's plus group 1's) through shared memory, so the CTA writes one
// partial row: half as many partials for the finalize to read as two
// single-group CTAs would leave. Per-row results are those of bwd_row_cta_kernel
// (the same operations in the same order). Taken when the accumulators and
// both rows fit in registers (the planner's bwd_row_pf_fits).
//
// kSmem: where the column sums live. 0: registers. 1: dbeta (LayerNorm) and
// dbias in shared memory after w, [N][Q][thread] float4 per sum, each thread
// its own slots (no barrier guards them inside the row loop), dgamma in
// registers. 2: dgamma in shared memory too. Moving the sums out of
// registers is what lets rows of four vectors per thread keep both rows in
// registers without spilling; the same sums in the same order as the
// register form, one 16-byte shared load and store per two pairs and sum.
template <typename T, int N, bool kRms, bool kBias, int kSmem = 0, int GT = kBulkThreads,
          int G = kPfGroups>
__global__ void __launch_bounds__(G * GT, G * GT < kPfThreads ? kPfThreads / (G * GT) : 1)
    bwd_row_pf_kernel(const BwdArgs a) {
  constexpr int VEC = Vec<T>::N;
  constexpr int P = VEC / 2;
  constexpr int Q = P / 2;   // float4 per vector of w
  extern __shared__ __align__(16) float4 w_s[];   // [N][Q][gt], then the kSmem slots
  // Threads of a row group (GT: 256; 128 for rows of up to 512 vectors; 320
  // to 512, one group per CTA, for rows of more than 1024) and of the CTA.
  constexpr int gt = GT;
  constexpr int ct = G * GT;
  // Shared-memory sums in order: dgamma (kSmem 2), dbeta (LayerNorm), dbias.
  constexpr bool kGS = kSmem == 2;
  constexpr bool kBS = kSmem >= 1 && !kRms;
  constexpr bool kDS = kSmem >= 1 && kBias;
  constexpr int kSlotB = kGS ? 1 : 0;
  constexpr int kSlotD = kSlotB + (kBS ? 1 : 0);
  constexpr int kAccS = (kGS ? 1 : 0) + (kBS ? 1 : 0) + (kDS ? 1 : 0);
  float4* acc_s = w_s + N * Q * gt;
  auto acc_slot = [&](int which, int k, int q) -> float4& {
    return acc_s[((which * N + k) * Q + q) * ct + threadIdx.x];
  };
  auto acc_add = [&](int which, int k, const float2 (&v)[P]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      float4& s = acc_slot(which, k, q);
      const float2 lo = add2(make_float2(s.x, s.y), v[2 * q]);
      const float2 hi = add2(make_float2(s.z, s.w), v[2 * q + 1]);
      s = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
  };
  auto acc_fma = [&](int which, int k, const float2 (&u)[P], const float2 (&v)[P]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      float4& s = acc_slot(which, k, q);
      const float2 lo = fma2(u[2 * q], v[2 * q], make_float2(s.x, s.y));
      const float2 hi = fma2(u[2 * q + 1], v[2 * q + 1], make_float2(s.z, s.w));
      s = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
  };
#pragma unroll
  for (int which = 0; which < kAccS; ++which)
#pragma unroll
    for (int k = 0; k < N; ++k)
#pragma unroll
      for (int q = 0; q < Q; ++q) acc_slot(which, k, q) = make_float4(0.f, 0.f, 0.f, 0.f);
  __shared__ float2 red[G][2][GT / 32];
  const int grp = threadIdx.x / gt;
  const int t = threadIdx.x % gt;
  const int H = a.hidden;
  const int V = H / VEC;
  const T* dy = static_cast<const T*>(a.dy);
  const T* xs = static_cast<const T*>(a.x_sum);
  T* dx = static_cast<T*>(a.dx);
  if (grp == 0) {
    const T* gamma = static_cast<const T*>(a.gamma);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * gt + t;
      if (v < V) {
        float2 w[P];
        unpack2<T>(ld_vec_param(gamma + v * VEC), w);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          float2 w0 = w[2 * q], w1 = w[2 * q + 1];
          if (a.zero_centered) {
            w0 = add2(w0, splat2(1.f));
            w1 = add2(w1, splat2(1.f));
          }
          w_s[(k * Q + q) * gt + t] = make_float4(w0.x, w0.y, w1.x, w1.y);
        }
      }
    }
  }
  __syncthreads();
  auto load_w = [&](int k, float2 (&w)[P]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 f = w_s[(k * Q + q) * gt + t];
      w[2 * q] = make_float2(f.x, f.y);
      w[2 * q + 1] = make_float2(f.z, f.w);
    }
  };
  // Sum of a float2 over the group: warp butterfly, then the group's 8 warps
  // in order through a double-buffered exchange behind the group's barrier.
  int parity = 0;
  auto group_row_sum = [&](float2 v) {
    v = group_sum2<32>(v);
    if ((t & 31) == 0) red[grp][parity][t >> 5] = v;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(gt) : "memory");
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < gt / 32; ++i) {
      s.x += red[grp][parity][i].x;
      s.y += red[grp][parity][i].y;
    }
    parity ^= 1;
    return s;
  };
  float2 acc_g[N][P], acc_b[N][P], acc_d[N][P];
  zero_acc2<T, N>(acc_g);
  zero_acc2<T, N>(acc_b);
  zero_acc2<T, N>(acc_d);
  uint4 nd[N], nx[N];
  float nr = 0.f, nm = 0.f;
  auto load_row = [&](int64_t row) {
    const int64_t off = row * (int64_t)H;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * gt + t;
      if (v < V) {
        nd[k] = ld_vec(dy + off + v * VEC);
        nx[k] = ld_vec(xs + off + v * VEC);
      }
    }
    nr = a.rstd[row];
    if (!kRms) nm = a.mean[row];
  };
  const int64_t first = (int64_t)blockIdx.x * G + grp;
  const int64_t stride = (int64_t)gridDim.x * G;
  if (first < a.rows) load_row(first);
  for (int64_t row = first; row < a.rows; row += stride) {
    uint4 dr[N], xr[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      dr[k] = nd[k];
      xr[k] = nx[k];
    }
    const float rstd = nr, mean = nm;
    if (row + stride < a.rows) load_row(row + stride);
    const int64_t off = row * (int64_t)H;
    const float2 neg_mean = splat2(-mean);
    const float2 r2 = splat2(rstd);
    float2 sx = splat2(0.f), sy = splat2(0.f);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * gt + t;
      if (v < V) {
        float2 d[P], xv[P], w[P];
        unpack2<T>(dr[k], d);
        unpack2<T>(xr[k], xv);
        load_w(k, w);
        float2 xh[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
          xh[i] = mul2(kRms ? xv[i] : add2(xv[i], neg_mean), r2);
          const float2 g = mul2(d[i], w[i]);
          if (!kRms) sx = add2(sx, g);
          sy = fma2(g, xh[i], sy);
          if (!kGS) acc_g[k][i] = fma2(d[i], xh[i], acc_g[k][i]);
          if (!kRms && !kBS) acc_b[k][i] = add2(acc_b[k][i], d[i]);
        }
        if (kGS) acc_fma(0, k, d, xh);
        if (kBS) acc_add(kSlotB, k, d);
      }
    }
    const float2 sums = group_row_sum(make_float2(kRms ? 0.f : sx.x + sx.y, sy.x + sy.y));
    // dx = rstd * (g - c1 - xhat * c2) = (x - mean) * b2 + (g * rstd + a1)
    const float c2 = sums.y * a.inv_hidden;
    const float2 a1 = splat2(kRms ? 0.f : -rstd * (sums.x * a.inv_hidden));
    const float2 b2 = splat2(-rstd * rstd * c2);
    vec_fence<N>(dr);
    vec_fence<N>(xr);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int v = k * gt + t;
      if (v < V) {
        float2 d[P], xv[P], w[P], o[P];
        unpack2<T>(dr[k], d);
        unpack2<T>(xr[k], xv);
        load_w(k, w);
#pragma unroll
        for (int i = 0; i < P; ++i) {
          const float2 gr = kRms ? mul2(mul2(d[i], w[i]), r2)
                                 : fma2(mul2(d[i], w[i]), r2, a1);
          o[i] = fma2(kRms ? xv[i] : add2(xv[i], neg_mean), b2, gr);
          if (kBias && !kDS) acc_d[k][i] = add2(acc_d[k][i], o[i]);
        }
        if (kDS) acc_add(kSlotD, k, o);
        st_vec(dx + off + v * VEC, pack2<T>(o));
      }
    }
  }
  allow_dependent_launch();
  // One partial row per CTA: with two groups, group 1's sums go through
  // shared memory (the staged w is no longer needed) and group 0 adds them
  // to its own.
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  auto put = [&](float2 (&acc)[N][P], int off) {
    __syncthreads();
    if (G == 2 && grp == 1) {
#pragma unroll
      for (int k = 0; k < N; ++k)
#pragma unroll
        for (int q = 0; q < Q; ++q)
          w_s[(k * Q + q) * gt + t] =
              make_float4(acc[k][2 * q].x, acc[k][2 * q].y, acc[k][2 * q + 1].x, acc[k][2 * q + 1].y);
    }
    __syncthreads();
    if (grp == 0) {
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const int v = k * gt + t;
        if (v < V) {
          float4* dst = reinterpret_cast<float4*>(ws + off + v * VEC);
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            if (G == 2) {
              const float4 o = w_s[(k * Q + q) * gt + t];
              const float2 lo = add2(acc[k][2 * q], make_float2(o.x, o.y));
              const float2 hi = add2(acc[k][2 * q + 1], make_float2(o.z, o.w));
              dst[q] = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
              dst[q] = make_float4(acc[k][2 * q].x, acc[k][2 * q].y, acc[k][2 * q + 1].x,
                                   acc[k][2 * q + 1].y);
            }
          }
        }
      }
    }
  };
  // Shared-memory sums: group 0 adds group 1's slots (thread t + gt) to its
  // own, after a barrier that orders the row loop's last shared stores.
  auto put_s = [&](int which, int off) {
    __syncthreads();
    if (grp == 0) {
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const int v = k * gt + t;
        if (v < V) {
          float4* dst = reinterpret_cast<float4*>(ws + off + v * VEC);
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            const float4 m = acc_slot(which, k, q);
            if (G == 2) {
              const float4 o = acc_s[((which * N + k) * Q + q) * ct + gt + t];
              const float2 lo = add2(make_float2(m.x, m.y), make_float2(o.x, o.y));
              const float2 hi = add2(make_float2(m.z, m.w), make_float2(o.z, o.w));
              dst[q] = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
              dst[q] = m;
            }
          }
        }
      }
    }
  };
  if (kGS) put_s(0, 0); else put(acc_g, 0);
  if (kBS) put_s(kSlotB, H); else if (!kRms) put(acc_b, H);
  if (kDS) put_s(kSlotD, kRms ? H : 2 * H); else if (kBias) put(acc_d, kRms ? H : 2 * H);
}

// ---- scalar kernel ----------------------------------------------------------

// Any hidden size and alignment. Dynamic shared memory: 4 * hidden floats
// (two per-row staging arrays and the dgamma/dbeta accumulators) plus hidden
// floats of dbias accumulators when has_dbias; column j belongs to thread
// j % kScalarCta throughout, so no barrier guards them.
template <typename T>
__global__ void __launch_bounds__(kScalarCta) bwd_scalar_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  __shared__ float2 red[kScalarCta / 32];
  const int H = a.hidden;
  float* acc_g = sm;
  float* acc_b = sm + H;
  float* sxh = sm + 2 * H;
  float* sg = sm + 3 * H;
  float* acc_d = sm + 4 * H;   // only with has_dbias
  const T* dy = static_cast<const T*>(a.dy);
  const T* xs = static_cast<const T*>(a.x_sum);
  const T* gamma = static_cast<const T*>(a.gamma);
  T* dx = static_cast<T*>(a.dx);
  for (int j = threadIdx.x; j < H; j += kScalarCta) {
    acc_g[j] = 0.f;
    acc_b[j] = 0.f;
    if (a.has_dbias) acc_d[j] = 0.f;
  }
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
    const float c1 = a.rms ? 0.f : sums.x * a.inv_hidden;
    const float c2 = sums.y * a.inv_hidden;
    for (int j = threadIdx.x; j < H; j += kScalarCta) {
      const float o = rstd * (sg[j] - c1 - sxh[j] * c2);
      dx[off + j] = from_f<T>(o);
      if (a.has_dbias) acc_d[j] += o;
    }
  }
  float* ws = a.ws + (int64_t)blockIdx.x * a.ws_cols;
  const int off_d = partial_offset(a, 2);
  for (int j = threadIdx.x; j < H; j += kScalarCta) {
    ws[j] = acc_g[j];
    if (!a.rms) ws[H + j] = acc_b[j];
    if (a.has_dbias) ws[off_d + j] = acc_d[j];
  }
}

}  // namespace nf
