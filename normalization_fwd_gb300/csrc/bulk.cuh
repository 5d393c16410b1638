// Bulk-copy pipeline primitives (sm_90+ PTX, used here on sm_103a): mbarrier
// phase tracking, cp.async.bulk global -> shared copies that complete on an
// mbarrier, and waits that give up after a time limit instead of spinning
// forever.
//
// A pipelined CTA streams tiles of whole rows into a ring of `stages`
// shared-memory slots, every slot in flight at once. Thread 0 fills all
// slots first; after that the warp that releases a slot last (a per-slot
// arrival counter tells it) refills it at once with the CTA's tile
// it + stages, so no thread ever waits for a slot to drain. Each slot has a
// `full` barrier (one arrival plus the transaction bytes of its copies) and
// an `empty` barrier (one arrival per warp). Round r of slot s waits `full`
// with parity r & 1 and `empty` with parity (r & 1) ^ 1.
#pragma once

#include "common.cuh"

namespace nf {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait

// Error bits a kernel leaves in the device error word of its translation
// unit (read and cleared by ln_device_error()).
constexpr unsigned kErrWaitTimeout = 1u;
static __device__ unsigned g_tu_error;

// Read and clear this translation unit's device error word, after `st`.
static inline cudaError_t take_tu_error(cudaStream_t st, unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tu_error, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tu_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  *out |= v;
  return e;
}


__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make the initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait with a suspend-time hint: the warp is parked (issuing nothing and
// polling no shared memory) until the phase completes or about `hint_ns`
// nanoseconds have passed.
constexpr uint32_t kSuspendHintNs = 1000000u;
__device__ __forceinline__ bool mbar_test_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with the given parity to complete; false when
// it has not completed within kWaitLimitNs. Waiting warps sleep in the
// hinted try_wait instead of spinning, so they take no issue slots and no
// shared-memory bandwidth from the warps that work.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_test_suspend(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory; completes as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy that evicts the lines it touches first (data read once).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 16-byte loads from shared memory, always as ld.shared (a generic load of
// a shared address would take the slower L1TEX path). Volatile, so they stay
// after the barrier waits (volatile asm keeps its order) and are never merged
// with an earlier load of the same address.
__device__ __forceinline__ float4 ld_f4_smem(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}
// The same from a 32-bit shared address (row bases are converted once and
// the per-slot offsets are constants the assembler folds into the load).
__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

// A [hidden] parameter row (gamma with the zero-centered +1 folded in, bias,
// beta) as fp32, read by 16-byte vector slot v. Staged rows live in shared
// memory in a split layout: for 8-element vectors the first four elements of
// every vector come first ([v * 4, v * 4 + 4)), the last four after them
// ([hidden / 2 + v * 4, ...)), so consecutive lanes read consecutive 16-byte
// words (no bank conflicts). Unstaged rows are read from global memory in
// the I/O dtype.
template <typename T>
struct ParamRow {
  const float* s;      // staged row, or null
  const T* g;          // the row in global memory
  int hidden;
  bool plus_one;       // add 1 to values read from global (zero-centered gamma)

  // 32-bit shared address of the staged row (valid when s is not null).
  __device__ __forceinline__ uint32_t saddr() const { return smem_addr(s); }

  static __device__ __forceinline__ int staged_index(int i, int hidden) {
    constexpr int VEC = Vec<T>::N;
    if (VEC == 4) return i;
    const int v = i / VEC, e = i % VEC;
    return (e < 4 ? 0 : hidden / 2) + v * 4 + (e & 3);
  }

  // The same values as fp32 pairs; `sa` is saddr() (hoisted by the caller).
  template <bool kStaged>
  __device__ __forceinline__ void load2(int v, float2* out, uint32_t sa = 0) const {
    constexpr int VEC = Vec<T>::N;
    if (kStaged) {
      const float4 a = lds_f4(sa + v * 16);
      out[0] = make_float2(a.x, a.y);
      out[1] = make_float2(a.z, a.w);
      if (VEC == 8) {
        const float4 b = lds_f4(sa + hidden * 2 + v * 16);
        out[2] = make_float2(b.x, b.y);
        out[3] = make_float2(b.z, b.w);
      }
    } else {
      unpack2<T>(*reinterpret_cast<const uint4*>(g + v * VEC), out);
      if (plus_one) {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) out[i] = add2(out[i], splat2(1.0f));
      }
    }
  }

  template <bool kStaged>
  __device__ __forceinline__ void load(int v, float* out) const {
    constexpr int VEC = Vec<T>::N;
    if (kStaged) {
      const float4 a = ld_f4_smem(s + v * 4);
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
      if (VEC == 8) {
        const float4 b = ld_f4_smem(s + hidden / 2 + v * 4);
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
      }
    } else {
      // A coherent load: the compiler reloads it after the "memory" barrier
      // between the two passes instead of keeping it live in registers.
      unpack<T>(*reinterpret_cast<const uint4*>(g + v * VEC), out);
      if (plus_one) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) out[e] += 1.0f;
      }
    }
  }
};

// Stage a parameter row into shared memory (split layout); all threads call
// it. Values get +1 when `plus_one`.
template <typename T>
__device__ __forceinline__ void stage_param_row(const T* g, int hidden, bool plus_one, float* s) {
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) {
    const float x = to_f(g[i]);
    s[ParamRow<T>::staged_index(i, hidden)] = plus_one ? 1.0f + x : x;
  }
}

// Ring layout in dynamic shared memory: `stages` slots of `slot_bytes`, the
// full and empty barriers, the per-slot release counters, then (16-byte
// aligned) whatever the kernel keeps after the ring.
struct Ring {
  unsigned char* base;
  uint32_t slot_bytes;
  int stages;
  uint64_t* full;
  uint64_t* empty;
  unsigned* released;     // warps that released the slot in its current round
  long long* issued;      // tiles issued so far (for the drain after an abort)
  int* abort_now;         // set by a thread whose wait timed out (CTA-wide loops)
  unsigned char* after;   // first byte after the ring
  __device__ unsigned char* slot(int s) const { return base + (size_t)s * slot_bytes; }
};

// Bytes of the ring's bookkeeping after its slots (host and device agree).
__host__ __device__ constexpr size_t ring_aux_bytes(int stages) {
  return ((size_t)stages * (2 * sizeof(uint64_t) + sizeof(unsigned)) + sizeof(long long) +
          sizeof(int) + 15) &
         ~(size_t)15;
}

__device__ __forceinline__ Ring make_ring(unsigned char* smem, uint32_t slot_bytes, int stages) {
  Ring r;
  r.base = smem;
  r.slot_bytes = slot_bytes;
  r.stages = stages;
  r.full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * slot_bytes);
  r.empty = r.full + stages;
  r.issued = reinterpret_cast<long long*>(r.empty + stages);
  r.released = reinterpret_cast<unsigned*>(r.issued + 1);
  r.abort_now = reinterpret_cast<int*>(r.released + stages);
  r.after = smem + (size_t)stages * slot_bytes + ring_aux_bytes(stages);
  return r;
}

// Called by every thread of the CTA before the pipeline starts.
__device__ __forceinline__ void ring_init(const Ring& r) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < r.stages; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], kConsumerWarps);
      r.released[s] = 0;
    }
    *r.issued = 0;
    *r.abort_now = 0;
    fence_mbar_init();
  }
  __syncthreads();
}

// After an aborted wait: wait (bounded) for every tile the producer issued
// but the consumers did not take, so no copy is still writing into shared
// memory when the CTA exits. Called by thread 0.
__device__ __forceinline__ void ring_drain(const Ring& r, int64_t taken, int64_t issued) {
  for (int64_t it = taken; it < issued; ++it) {
    mbar_wait(&r.full[it % r.stages], (uint32_t)((it / r.stages) & 1));
  }
}

// Issue the copies of the CTA's local tile `it` (global tile blockIdx.x +
// it * gridDim.x): for each input (up to two) the tile's rows are one
// contiguous bulk copy, the inputs back to back in the slot. Waits (bounded)
// for the slot to be free; false on timeout. Thread 0 only.
template <typename T, bool kEvictFirst = false>
__device__ __forceinline__ bool issue_tile(const Ring& ring, const BulkCfg& c, int64_t it,
                                           int64_t rows, int hidden, const T* in0,
                                           const T* in1) {
  const int s = (int)(it % ring.stages);
  const uint32_t round = (uint32_t)(it / ring.stages);
  if (!mbar_wait(&ring.empty[s], (round & 1) ^ 1)) return false;
  const int64_t tile = blockIdx.x + it * gridDim.x;
  const uint32_t row_bytes = (uint32_t)hidden * sizeof(T);
  const int64_t r0 = tile * c.tile_rows;
  const int64_t n = rows - r0 < c.tile_rows ? rows - r0 : c.tile_rows;
  const uint32_t bytes = (uint32_t)n * row_bytes;
  mbar_arrive_expect_tx(&ring.full[s], in1 ? 2 * bytes : bytes);
  unsigned char* dst = ring.slot(s);
  unsigned char* dst1 = dst + (size_t)c.tile_rows * row_bytes;
  if (kEvictFirst) {
    const uint64_t pol = l2_evict_first_policy();
    bulk_load_hint(dst, in0 + r0 * hidden, bytes, &ring.full[s], pol);
    if (in1) bulk_load_hint(dst1, in1 + r0 * hidden, bytes, &ring.full[s], pol);
  } else {
    bulk_load(dst, in0 + r0 * hidden, bytes, &ring.full[s]);
    if (in1) bulk_load(dst1, in1 + r0 * hidden, bytes, &ring.full[s]);
  }
  return true;
}

// The pipeline loop: `body(tile, slot)` for each of the CTA's tiles in order.
// With kUniform (bodies with CTA-wide barriers) a thread whose wait timed out
// raises a shared flag and still runs the body (on stale but in-bounds
// shared data), so every thread reaches the body's barriers; after the body
// all threads see the flag and leave together. Returns the tiles consumed;
// `aborted` is set when a wait timed out.
template <bool kUniform, typename T, bool kEvictFirst = false, typename Body>
__device__ __forceinline__ int64_t run_pipeline(const Ring& ring, const BulkCfg& c, int64_t rows,
                                                int hidden, const T* in0, const T* in1,
                                                bool& aborted, Body body) {
  const int S = ring.stages;
  const int64_t n_local = (c.num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
  if (threadIdx.x == 0) {
    int64_t j = 0;
    for (; j < S && j < n_local; ++j) {
      if (!issue_tile<T, kEvictFirst>(ring, c, j, rows, hidden, in0, in1)) {
        aborted = true;
        break;
      }
    }
    *ring.issued = j;
  }
  __syncthreads();
  int64_t it = 0;
  for (; it < n_local; ++it) {
    const int s = (int)(it % S);
    const bool failed = !mbar_wait(&ring.full[s], (uint32_t)((it / S) & 1));
    if (kUniform) {
      if (failed) *(volatile int*)ring.abort_now = 1;
    } else if (failed) {
      aborted = true;
      break;
    }
    body(blockIdx.x + it * gridDim.x, ring.slot(s));
    if (kUniform && *(volatile int*)ring.abort_now) {   // seen by all after the body's barrier
      aborted = true;   // this tile is not counted as taken: the drain waits for its copy
      break;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      mbar_arrive(&ring.empty[s]);
      if (atomicAdd(&ring.released[s], 1u) == kConsumerWarps - 1) {
        // This warp released the slot last: reset its counter and refill it.
        atomicExch(&ring.released[s], 0u);
        const int64_t j = it + S;
        if (j < n_local) {
          if (issue_tile<T, kEvictFirst>(ring, c, j, rows, hidden, in0, in1)) {
            atomicMax(ring.issued, (long long)(j + 1));
          } else {
            aborted = true;
          }
        }
      }
    }
  }
  return it;
}

// Programmatic dependent launch: let the grid launched after this one on
// the stream (the backward's finalize) be scheduled once every CTA of this
// grid has called this; the dependent still waits (griddepcontrol.wait) for
// this grid to complete and its writes to be visible before it reads them.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// End of a pipelined kernel, all threads: record an abort in the error word,
// and on abort let thread 0 drain the copies still in flight. Returns true
// when the kernel aborted (the caller then skips its epilogue).
__device__ __forceinline__ bool pipeline_finish(const Ring& ring, bool aborted, int64_t taken,
                                                int* s_abort, long long* s_taken) {
  if (aborted) {
    atomicOr(&g_tu_error, kErrWaitTimeout);
    atomicExch(s_abort, 1);
  }
  if ((threadIdx.x & 31) == 0) atomicMin(s_taken, (long long)taken);
  __syncthreads();
  if (*s_abort) {
    if (threadIdx.x == 0) ring_drain(ring, *s_taken, *ring.issued);
    return true;
  }
  return false;
}

}  // namespace nf
