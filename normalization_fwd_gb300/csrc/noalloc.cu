// ln_bwd_noalloc: the fused backward for callers that cannot allocate device
// memory. Its scratch (the per-CTA dgamma/dbeta partials) lives in a static
// device array of this translation unit instead of a caller workspace.
#include "../../include/normfuse.h"
#include "launch.h"

namespace {

// The scratch array. It belongs to this library's module: a context holds
// its bytes from the moment the module is loaded in it (on the first call
// under lazy module loading) until the context is destroyed. In host code
// the name is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress.
__device__ __align__(256) float g_noalloc_scratch[LN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of the scratch array in the current context. It is looked
// up on every call, with the caller's device current, rather than cached: a
// cached address would outlive a cudaDeviceReset (which rebuilds the primary
// context and reloads the module at another address) or be handed to a
// different context made current on the same device. Once the module is
// loaded the lookup is a host-side table query; it enqueues nothing.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" ln_status ln_bwd_noalloc(const void* dy, const void* x_sum, const void* gamma,
                                    const float* mean, const float* rstd, void* dx,
                                    float* dgamma, float* dbeta, cudaStream_t stream,
                                    int64_t rows, int64_t hidden, ln_dtype dtype, ln_mode mode,
                                    int zero_centered_gamma) {
  void* scratch = nullptr;
  if (rows > 0) {
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      nf_set_last_cuda_error((int)e);
      return LN_ERR_CUDA;
    }
  }
  // Every CTA overwrites its whole partial row before the finalize reads it,
  // so nothing in the array has to start at zero.
  const ln_status s = ln_bwd(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, stream, rows,
                             hidden, dtype, mode, zero_centered_gamma, scratch,
                             scratch ? (size_t)LN_NOALLOC_SCRATCH_BYTES : 0);
  // With a non-null, aligned scratch the only workspace failure left is size.
  return s == LN_ERR_WORKSPACE ? LN_ERR_SCRATCH_LIMIT : s;
}
