// Test helper (built by tests/test_gpu_wait_timeout.py): a kernel that waits,
// with the library's bounded mbarrier wait, on a barrier nothing arrives at.
// The wait must give up after its time limit and report it, leaving the
// context usable. No copy is issued, so nothing is in flight when it returns.
#include <stdint.h>

#include "bulk.cuh"

namespace {

__global__ void never_arrives(int* timed_out, unsigned long long* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    nf::mbar_init(&bar, 1);   // expects one arrival that never comes
    nf::fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = nf::global_ns();
  const bool ok = nf::mbar_wait(&bar, 0);
  const uint64_t t1 = nf::global_ns();
  if (!ok) atomicAdd(timed_out, 1);
  if (threadIdx.x == 0) *waited_ns = t1 - t0;
}

}  // namespace

extern "C" int wait_timeout_launch(int* timed_out, unsigned long long* waited_ns, int threads) {
  never_arrives<<<1, threads>>>(timed_out, waited_ns);
  return (int)cudaGetLastError();
}
