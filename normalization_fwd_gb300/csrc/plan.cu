// Host-side planning and launching: which kernel runs a call, its grid,
// block and shared memory, and the launch itself. Kernels come from the
// per-family tables of the kernel translation units (tables.cuh).
#include <algorithm>

#include "bulk.cuh"
#include "launch.h"
#include "softmax_kernels.cuh"

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

// Backward lane groups: four vectors a lane, else three, five, two or one,
// where the row splits exactly over 8, 16 or 32 lanes and the accumulators
// (n * VEC floats per reduction: dgamma; dbeta for LayerNorm; dbias) fit.
// A lane group whose accumulators would not fit, or whose lanes would hold
// more than 40 floats of each input row (more than five 16-byte vectors of
// a 16-bit type), moves to a row group of 64 or 128 threads (kind 3), the
// smallest that fits. Measured at 268 MB per tensor, bf16, kernel alone:
// 256 wide LayerNorm 127 us as 8 x 4 against 208 as 32 x 1 (RMSNorm 138
// against 190); 512 wide LayerNorm 131 as 16 x 4 against 160 as 32 x 2;
// 1536 wide RMSNorm 127 as a 64 x 3 row group against 139 as 32 x 6 lanes;
// 2048 wide RMSNorm 137 as 64 x 4 against 149 as 32 x 8.
constexpr int kMaxLaneRowFloats = 40;
inline Choice bwd_choice(const Choice& c, int hidden, int vec_elems, bool rms, bool dbias) {
  if (c.kind != 0) return c;
  const int n_acc = 1 + (rms ? 0 : 1) + (dbias ? 1 : 0);
  const int V = hidden / vec_elems;
  for (int n : {4, 3, 5, 2, 1}) {
    if (V % n) continue;
    const int lanes = V / n;
    if ((lanes == 8 || lanes == 16 || lanes == 32) && n * vec_elems * n_acc <= kMaxAccFloats &&
        n * vec_elems <= kMaxLaneRowFloats)
      return {0, lanes, n};
  }
  if (c.n * vec_elems * n_acc <= kMaxAccFloats && c.n * vec_elems <= kMaxLaneRowFloats) return c;
  for (int g : {64, 128}) {
    int n = (V + g - 1) / g;
    if (n == 7) n = 8;
    if (n < 2) n = 2;
    if (n * vec_elems * n_acc <= kMaxAccFloats) return {3, g, n};
  }
  return c;
}

// CTA size (a whole number of warps, 64 to kMaxFitThreads) and vectors per
// thread of the row-fitted CTA-per-row kernels, for rows of V > 256
// vectors: four vectors per thread where that splits the row into whole
// warps, else five, three, six, eight or two; failing all, the split of
// four, five, three or six per thread that leaves the fewest vector slots
// idle. (Forward at 268 MB per tensor, bf16: 2560 wide 157 us as 64 x 5,
// 228 as 256 x 2; 3072 156 as 96 x 4, 199 as 256 x 2; 4096 157 as
// 128 x 4, 176 as 256 x 2; 5120 156 as 160 x 4, 168 as 256 x 3.)
struct Fit {
  int threads, n;
};
inline Fit cta_fit(int V) {
  for (int n : {4, 5, 3, 6, 8, 2}) {
    if (V % n) continue;
    const int nt = V / n;
    if (nt % 32 == 0 && nt >= 64 && nt <= kMaxFitThreads) return {nt, n};
  }
  Fit best = {0, 0};
  int idle = 1 << 30;
  for (int n : {4, 5, 3, 6}) {
    const int nt = std::max(64, (V + 32 * n - 1) / (32 * n) * 32);
    if (nt > kMaxFitThreads) continue;
    if (nt * n - V < idle) {
      idle = nt * n - V;
      best = {nt, n};
    }
  }
  if (best.n == 0) best = {kMaxFitThreads, std::max(2, (V + kMaxFitThreads - 1) / kMaxFitThreads)};
  return best;
}

// The register forward's lane groups: four, then three, five, two or one
// vectors per lane where the row splits exactly over 8, 16 or 32 lanes; rows
// of more than kFwdGroupMaxV vectors take the row-fitted CTA kernel instead.
// (268 MB per tensor, bf16 with residual: 256 wide 159 us as 8 x 4, 189 as
// 32 x 1; 512 wide 160 as 16 x 4, 172 as 32 x 2; 1536 wide 155 as a 64 x 3
// CTA, 168 as 32 x 6 lanes; 2048 wide 157 as a 64 x 4 CTA, 161 as 32 x 8.)
constexpr int kFwdGroupMaxV = 160;
inline Choice fwd_group_choice(const Choice& c, int V) {
  for (int n : {4, 3, 5, 2, 1}) {
    if (V % n) continue;
    const int lanes = V / n;
    if (lanes == 8 || lanes == 16 || lanes == 32) return {0, lanes, n};
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
    static const void* bwd_bulk(int k, int g, int n, bool rms, bool dbias, bool exact) {  \
      if (dbias) return rms ? bwd_bulk_rms_dbias_table_##NAME(k, g, n, exact)             \
                            : bwd_bulk_ln_dbias_table_##NAME(k, g, n, exact);             \
      return rms ? bwd_bulk_rms_table_##NAME(k, g, n, exact)                              \
                 : bwd_bulk_ln_table_##NAME(k, g, n, exact);                              \
    }                                                                               \
    static const void* bwd_reg(int k, int g, int n) { return bwd_reg_table_##NAME(k, g, n); }   \
    static const void* softmax(int k, int g, int n) { return softmax_table_##NAME(k, g, n); }   \
    static const void* partials(int k, int g, int n) { return partials_table_##NAME(k, g, n); } \
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
// The lane-group backward keeps at most three slots once a slot holds
// 20 KiB or more (three slots of 16 rows at 384 bf16: 199.9 against 201.1 us
// for four at 576000 rows; the smaller ring leaves more of the SM's on-chip
// memory to L1, which serves the statistics).
constexpr size_t kBwdGroupBigSlot = 20 * 1024;
constexpr int kBwdGroupBigSlotStages = 3;
constexpr size_t kMaxDynSmem = 200 * 1024;
constexpr size_t kRingTargetSmx = 48 * 1024;

// three_ctas: kernels built for three CTAs per SM (the lane-group forward)
// get the smaller ring. (For the CTA-per-row RMSNorm backward, 2 CTAs with
// 3 slots measured 167 us at 16384 x 8192 against 176 us for 3 CTAs with 2.)
inline size_t ring_target(bool three_ctas) {
  return three_ctas ? kRingTargetFwdGroup : kRingTarget;
}

// Fill in a pipelined plan; false when the ring does not fit. `extra`:
// shared bytes after the ring's barriers (the backward's fp32 weight row).
inline bool fill_bulk(Plan* p, const Choice& c, int64_t rows, int hidden, size_t esize, int n_in,
                      size_t extra, size_t target, bool bwd_group) {
  const int tile_rows = c.kind == 0 ? kConsumerWarps * (32 / c.group)
                                    : (c.kind == 3 ? kBulkThreads / c.group : 1);
  const size_t slot = (size_t)n_in * tile_rows * hidden * esize;
  const size_t room = target > extra ? target - extra : 0;
  int stages = (int)std::min<size_t>(8, std::max<size_t>(2, room / slot));
  if (bwd_group && slot >= kBwdGroupBigSlot) stages = std::min(stages, kBwdGroupBigSlotStages);
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

// Block and shared memory of the scalar kernels (one row per CTA step).
inline void fill_scalar(Plan* p, int hidden, bool bwd, bool dbias) {
  p->bulk = false;
  p->kind = 2;
  p->group = kScalarCta;
  p->n = 0;
  p->block = kScalarCta;
  p->smem = (size_t)hidden * sizeof(float) * (bwd ? (dbias ? 5 : 4) : 1);
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
//
// Forward: rows straight into registers with one CTA per row tile (kind 4,
// lane groups, up to kFwdGroupMaxV vectors) or per row (kind 5, the CTA
// sized by cta_fit); the ring family selects the bulk-copy ring kernels
// instead.
//
// Backward rows of more than 256 vectors run from registers with a CTA per
// row when the accumulators (n * VEC floats per reduction: dgamma; dbeta for
// LayerNorm; dbias) and the row's two inputs (8n registers) fit in 64
// registers' worth (56 for LayerNorm, which also keeps the mean and a second
// row sum live), so that kernel (kind 5) keeps three or more CTAs per SM
// without spilling. Its variant with the next row prefetched (kind 6, one
// CTA of two 256-thread row groups per SM, both rows' inputs in 16n
// registers) holds four rows per SM in flight; it is taken where it fits in
// 96 registers' worth and the one-row kernel would hold fewer than four
// (measured with two 256-thread CTAs per SM, the same four rows in flight:
// 16384 x 8192 bf16 RMSNorm 121.6 against 127.7 us, 21845 x 6144
// LayerNorm 135.5 against 159.4 us; at 32768 x 4096 RMSNorm, where kind 5
// runs four CTAs per SM, 138.5 against 128.9 us). Where neither fits, kinds
// 7 and 8 (below) keep some or all column sums in shared memory. The other
// aligned rows, and these too under the ring family, stream through the
// bulk-copy ring.
inline int bwd_acc_floats(int n, int vec_elems, bool rms, bool dbias) {
  return n * vec_elems * (1 + (rms ? 0 : 1) + (dbias ? 1 : 0));
}
inline bool bwd_row_pf_fits(int n, int vec_elems, bool rms, bool dbias) {
  return n <= 4 && bwd_acc_floats(n, vec_elems, rms, dbias) + 16 * n <= 96;
}
inline bool bwd_row_cta_fits(int n, int vec_elems, bool rms, bool dbias) {
  return n <= 4 && bwd_acc_floats(n, vec_elems, rms, dbias) + 8 * n <= (rms ? 64 : 56);
}
// Kinds 7 and 8: kind 6 with column sums in shared memory, each thread its
// own slots. Kind 7 moves dbeta and dbias there, so only dgamma's (n * VEC
// floats) count against the registers; kind 8 moves dgamma's too, and is
// taken for LayerNorm without dbias (rows of four vectors: kind 7 spills a
// little there). Measured at 16384 x 8192 bf16, kernel alone: LayerNorm
// 150 us as kind 8 against 166 as kind 7 and 171 on the ring; LayerNorm
// with dbias 189 as kind 7 against 232 as kind 8 (224 KiB of shared memory
// leave L1 little room) and 246 on the ring; RMSNorm with dbias 135 as kind
// 7 against 142 as kind 8; 21845 x 6144 LayerNorm with dbias 146 as kind 7
// against 174 as kind 8 and 189 on the ring.
inline bool bwd_row_pf_smem_fits(int n, int vec_elems, bool rms, bool dbias) {
  return n >= 3 && n <= 4 && (!rms || dbias) && n * vec_elems + 16 * n <= 96;
}
inline bool bwd_row_pf_all_smem(int n, bool rms, bool dbias) {
  return n == 4 && !rms && !dbias;
}
// Dynamic shared memory of kinds 6-8 with row groups of gt threads: w
// staged as fp32 (n vectors of VEC floats per thread of a row group), then
// the shared-memory sums of both row groups (smem_sums: 1 for kind 7, 2 for
// kind 8).
inline size_t bwd_row_pf_smem(int n, int vec_elems, bool rms, bool dbias, int smem_sums,
                              int gt = kBulkThreads, int groups = kPfGroups) {
  const size_t per = (size_t)n * vec_elems * sizeof(float);
  const int n_acc = smem_sums == 0 ? 0
                                   : (smem_sums == 2 ? 1 : 0) + (rms ? 0 : 1) + (dbias ? 1 : 0);
  return per * gt + per * groups * gt * n_acc;
}

// Rows of more than 1024 vectors (wider than 8192 in 16-bit types, than 4096
// in fp32): one row group per CTA of 320 to 512 threads (a multiple of 64,
// the row at four vectors a thread) with the next row prefetched: RMSNorm
// keeps its sums in registers (kind 6); with dbias, dbeta / dbias go to
// shared memory (kind 7); LayerNorm without dbias keeps every sum in shared
// memory (kind 8) up to 384-thread groups and dgamma in registers (kind 7)
// from 448 (16384-wide bf16: 164.5 us as kind 7, 187.1 as kind 8;
// 12288-wide: 178.3 as kind 7, 157.7 as kind 8). Two rows of 40 to 64 KB
// each are in flight per SM. The ring kernel these replace ran 12288-wide
// bf16 LayerNorm at 0.53 of the measured copy rate and 16384-wide at 0.35
// (RMSNorm 0.75 and 0.68).
constexpr int kWideMaxThreads = 512;
inline int bwd_wide_threads(int V) {
  if (V <= 4 * kBulkThreads || V > 4 * kWideMaxThreads) return 0;
  return (V + 255) / 256 * 64;
}
inline int bwd_wide_kind(bool rms, bool dbias, int threads) {
  if (rms && !dbias) return 6;
  if (!rms && !dbias) return threads >= 448 ? 7 : 8;
  return 7;
}

// Rows of 257 to 512 vectors, where 256-thread row groups of two vectors a
// thread leave slots idle or hold too few rows per SM: two 128-thread row
// groups per CTA and two CTAs per SM, three or four vectors a thread.
// RMSNorm keeps its sums in registers (kind 6), LayerNorm and dbias rows of
// three vectors keep dbeta / dbias in shared memory (kind 7). Measured at
// 268 MB per tensor, bf16, kernel alone: RMSNorm 2560 wide 131.5 us against
// 151.0 (256 x 2, kind 5), 3072 125.2 against 141.3, 4096 (four vectors)
// 123.1 against 130.0; LayerNorm 2560 141.3 against 176.6 (256 x 2, kind 6),
// 3072 129.3 against 177.0. LayerNorm at 4096 stays on 256 x 2 (142.7 us;
// 147.6 as 128 x 4 with every sum in shared memory).
//
// The same one size down for rows of 129 to 256 vectors (1032 to 2048 wide
// in 16-bit types): two 64-thread row groups per CTA, four CTAs per SM.
// Kernel alone, bf16: RMSNorm 1280 wide 128.2 us against 134.1 (32 x 5
// lanes), 1536 123.0 against 127.5 (64 x 3 row-group ring), 2048 127.7
// against 139.3 (64 x 4 ring); LayerNorm 1280 130.4 against 144.2, 1536
// 124.9 against 138.9. LayerNorm at 2048 stays on the ring (129.0 against
// 135.3 with every sum in shared memory).
inline Choice bwd_small_group(int V, bool rms, bool dbias) {
  int gt = 0;
  if (V > 128 && V <= 256) {
    gt = 64;
  } else if (V > 256 && V <= 512) {
    gt = 128;
  } else {
    return {0, 0, 0};
  }
  const int n = (V + gt - 1) / gt;
  if (rms && !dbias) return {6, gt, n};
  return n == 3 ? Choice{7, gt, n} : Choice{0, 0, 0};
}
constexpr int kRowsInFlightPf = 4;   // kind 6: two row groups per SM, two rows each

template <typename T>
cudaError_t make_plan(int64_t rows, int hidden, bool vec, bool bwd, bool rms, bool dbias,
                      int n_in, int n_params, Plan* p) {
  const Choice c = choose(hidden, Vec<T>::N, vec);
  const bool ring = kernel_family(bwd ? kFamilyBackward : kFamilyForward) == kFamilyRing;
  if (bwd && vec && (c.kind == 0 || c.kind == 1) && !ring) {
    const Choice sg = bwd_small_group(hidden / Vec<T>::N, rms, dbias);
    if (sg.kind != 0) {
      p->bulk = false;
      p->kind = sg.kind;
      p->group = sg.group;
      p->n = sg.n;
      p->block = kPfGroups * sg.group;
      p->smem = bwd_row_pf_smem(sg.n, Vec<T>::N, rms, dbias, sg.kind - 6, sg.group);
      p->fn = Tables<T>::bwd_bulk(p->kind, sg.group, sg.n, rms, dbias, false);
      return size_grid(p, rows);
    }
  }
  if (bwd && vec && c.kind == 1 && !ring && !rms && !dbias && Vec<T>::N == 8 &&
      hidden / Vec<T>::N == 1024) {
    // 16-bit LayerNorm rows of 1024 vectors (8192 wide): one 512-thread row
    // group per CTA, two vectors a thread, dgamma in registers and dbeta in
    // shared memory (16384 x 8192, with the finalize, back to back: fp16
    // 154.5 us against 160.7 for two 256-thread groups of four vectors with
    // every sum in shared memory, bf16 within 2 us either way; at 6152 to
    // 8184 wide, where 512 x 2 leaves slots idle, the two groups stay).
    p->bulk = false;
    p->kind = 7;
    p->group = 512;
    p->n = 2;
    p->block = 512;
    p->smem = bwd_row_pf_smem(2, Vec<T>::N, rms, dbias, 1, 512, 1);
    p->fn = Tables<T>::bwd_bulk(7, 512, 2, rms, dbias, false);
    return size_grid(p, rows);
  }
  if (bwd && vec && c.kind == 1 && !ring) {
    const int wt = bwd_wide_threads(hidden / Vec<T>::N);
    if (wt != 0) {
      const int kind = bwd_wide_kind(rms, dbias, wt);
      p->bulk = false;
      p->kind = kind;
      p->group = wt;
      p->n = 4;
      p->block = wt;
      p->smem = bwd_row_pf_smem(4, Vec<T>::N, rms, dbias, kind - 6, wt, 1);
      p->fn = Tables<T>::bwd_bulk(kind, wt, 4, rms, dbias, false);
      return size_grid(p, rows);
    }
    const int n = bulk_cta_n(hidden, Vec<T>::N);
    const bool one = bwd_row_cta_fits(n, Vec<T>::N, rms, dbias);
    bool pf = bwd_row_pf_fits(n, Vec<T>::N, rms, dbias);
    if (pf && one) {
      // keep the one-row kernel where it already holds as many rows per SM
      int per_sm = 0;
      cudaError_t e = (cudaError_t)resident_blocks(
          Tables<T>::bwd_bulk(5, kBulkThreads, n, rms, dbias, false), kBulkThreads, 0, &per_sm);
      if (e != cudaSuccess) return e;
      pf = per_sm < kRowsInFlightPf;
    }
    const bool pf_smem = !pf && !one && bwd_row_pf_smem_fits(n, Vec<T>::N, rms, dbias);
    if (pf || one || pf_smem) {
      const int smem_sums = pf_smem ? (bwd_row_pf_all_smem(n, rms, dbias) ? 2 : 1) : 0;
      p->bulk = false;
      p->kind = pf ? 6 : (pf_smem ? 6 + smem_sums : 5);
      p->group = kBulkThreads;
      p->n = n;
      p->block = (pf || pf_smem) ? kPfThreads : kBulkThreads;
      p->smem = (pf || pf_smem) ? bwd_row_pf_smem(n, Vec<T>::N, rms, dbias, smem_sums) : 0;
      p->fn = Tables<T>::bwd_bulk(p->kind, kBulkThreads, n, rms, dbias, false);
      return size_grid(p, rows);
    }
  }
  const int V = vec ? hidden / Vec<T>::N : 0;
  if (!bwd && vec && !ring && (c.kind == 1 || (c.kind == 0 && V > kFwdGroupMaxV))) {
    const Fit f = cta_fit(V);
    p->bulk = false;
    p->kind = 5;
    p->group = f.threads;
    p->n = f.n;
    p->block = f.threads;
    p->smem = 0;
    p->fn = Tables<T>::fwd_bulk(5, f.threads, p->n);
    cudaError_t e = size_grid(p, 1);
    if (e != cudaSuccess) return e;
    if (rows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)rows;
    return cudaSuccess;
  }
  if (!bwd && vec && c.kind == 0 && !ring) {
    const Choice g = fwd_group_choice(c, V);
    p->bulk = false;
    p->kind = 4;
    p->group = g.group;
    p->n = g.n;
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::fwd_bulk(4, g.group, g.n);
    cudaError_t e = size_grid(p, 1);   // occupancy check and attributes
    if (e != cudaSuccess) return e;
    const int64_t rpc = (int64_t)kConsumerWarps * (32 / g.group);
    const int64_t ctas = (rows + rpc - 1) / rpc;
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)ctas;
    return cudaSuccess;
  }
  if (vec) {
    Choice b = bwd ? bwd_choice(c, hidden, Vec<T>::N, rms, dbias) : c;
    if (c.kind == 1) b.n = bulk_cta_n(hidden, Vec<T>::N);
    // Lane-group and row-group kernels stage the parameter rows in shared
    // memory as fp32; CTA-per-row kernels read them from global memory.
    const size_t extra = (b.kind == 0 || b.kind == 3) ? (size_t)n_params * hidden * sizeof(float) : 0;
    const bool three = !bwd && b.kind == 0 && b.n <= 4;
    if (fill_bulk(p, b, rows, hidden, sizeof(T), n_in, extra, ring_target(three),
                  bwd && b.kind == 0)) {
      const bool exact = b.kind == 0 && b.group * b.n * Vec<T>::N == hidden;
      p->fn = bwd ? Tables<T>::bwd_bulk(b.kind, b.group, b.n, rms, dbias, exact)
                  : Tables<T>::fwd_bulk(b.kind, b.group, b.n);
      return size_grid(p, p->cfg.num_tiles);
    }
    // No ring fits (not reached by any supported width): the scalar kernel.
    if (hidden > kMaxHiddenScalar) return cudaErrorInvalidConfiguration;
  }
  p->fn = bwd ? Tables<T>::bwd_reg(2, 0, 0) : Tables<T>::fwd_reg(2, 0, 0);
  fill_scalar(p, hidden, bwd, dbias);
  return size_grid(p, rows);
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
  const int smx_path = kernel_family(kFamilySoftmax);
  const int V = vec ? hidden / Vec<T>::N : 0;
  if (smx_path == 0 && (c.kind == 1 || (c.kind == 0 && V > kFwdGroupMaxV))) {
    // Longer rows: a row-fitted CTA per one or two rows, from registers.
    const Fit f = cta_fit(V);
    p->bulk = false;
    p->kind = 5;
    p->group = f.threads;
    p->n = f.n;
    p->block = f.threads;
    p->smem = 0;
    p->fn = Tables<T>::softmax(5, f.threads, p->n);
    cudaError_t e = size_grid(p, 1);
    if (e != cudaSuccess) return e;
    const int64_t ctas = smx_cta_grid(rows, p->n);
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)ctas;
    return cudaSuccess;
  }
  if (smx_path == 0 && c.kind == 0) {
    // Lane groups (the forward's choice of lanes): rows straight into
    // registers, one CTA per 8 * (32 / lanes) rows, as many CTAs as needed.
    const Choice g = fwd_group_choice(c, V);
    p->bulk = false;
    p->kind = 4;
    p->group = g.group;
    p->n = g.n;
    p->block = kBulkThreads;
    p->smem = 0;
    p->fn = Tables<T>::softmax(4, g.group, g.n);
    cudaError_t e = size_grid(p, 1);   // occupancy check and attributes
    if (e != cudaSuccess) return e;
    const int64_t rpc = (int64_t)kConsumerWarps * (32 / g.group);
    const int64_t ctas = (rows + rpc - 1) / rpc;
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p->grid = (int)ctas;
    return cudaSuccess;
  }
  if (c.kind == 0 || c.kind == 1) {
    Choice b = c;
    if (c.kind == 1) b.n = bulk_cta_n(hidden, Vec<T>::N);
    const size_t target = b.n <= 4 ? kRingTargetSmx : kRingTarget;
    if (fill_bulk(p, b, rows, hidden, sizeof(T), 1, 0, target, false)) {
      p->fn = Tables<T>::softmax(b.kind, b.group, b.n);
      return size_grid(p, p->cfg.num_tiles);
    }
    return cudaErrorInvalidConfiguration;
  }
  if (c.kind != 2) return cudaErrorInvalidConfiguration;
  p->fn = Tables<T>::softmax(2, 0, 0);
  fill_scalar(p, hidden, false, false);
  return size_grid(p, rows);
}

cudaError_t softmax_launch(const SmxArgs& a, const Plan& p, cudaStream_t st) {
  return launch_plan(p, const_cast<SmxArgs*>(&a), st);
}

// Normalize from partials: the forward's register shapes (a lane group per
// row and one CTA per row tile, or one CTA per row beyond 256 vectors), as
// many CTAs as the rows need; unaligned rows take the scalar kernel, one CTA
// per row.
// The normalize-from-partials kernel reads one stream per row (the forward
// reads two), so its lane groups take the exact fit with the fewest lanes:
// more vectors of a row per lane, more bytes in flight per SM (576000 x 384
// bf16: 8 lanes x 6 vectors 135 us against 152 for 16 x 3).
inline Choice partials_choice(const Choice& c, int hidden, int vec_elems) {
  if (c.kind != 0) return c;
  const int V = hidden / vec_elems;
  for (int lanes : {8, 16, 32}) {
    if (V % lanes == 0) {
      const int n = V / lanes;
      if (n <= 8 && n != 7) return {0, lanes, n};
    }
  }
  return c;
}

template <typename T> cudaError_t partials_plan(int64_t rows, int hidden, bool vec, Plan* p) {
  const Choice c = partials_choice(choose(hidden, Vec<T>::N, vec), hidden, Vec<T>::N);
  p->bulk = false;
  p->smem = 0;
  p->block = kBulkThreads;
  int64_t ctas = rows;
  if (c.kind == 0) {
    p->kind = 4;
    p->group = c.group;
    p->n = c.n;
    const int64_t rpc = (int64_t)kConsumerWarps * (32 / c.group);
    ctas = (rows + rpc - 1) / rpc;
  } else if (c.kind == 1) {
    const Fit f = cta_fit(hidden / Vec<T>::N);
    p->kind = 5;
    p->group = f.threads;
    p->n = f.n;
    p->block = f.threads;
  } else {
    p->kind = 2;
    p->group = kScalarCta;
    p->n = 0;
    p->block = kScalarCta;
  }
  p->fn = Tables<T>::partials(p->kind, p->group, p->n);
  cudaError_t e = size_grid(p, 1);   // occupancy check
  if (e != cudaSuccess) return e;
  if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
  p->grid = (int)ctas;
  return cudaSuccess;
}

cudaError_t partials_launch(const PartialsArgs& a, const Plan& p, cudaStream_t st) {
  return launch_plan(p, const_cast<PartialsArgs*>(&a), st);
}

}  // namespace nf

template cudaError_t nf::partials_plan<float>(int64_t, int, bool, nf::Plan*);
template cudaError_t nf::partials_plan<nf::bf16>(int64_t, int, bool, nf::Plan*);
template cudaError_t nf::partials_plan<nf::f16>(int64_t, int, bool, nf::Plan*);
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
