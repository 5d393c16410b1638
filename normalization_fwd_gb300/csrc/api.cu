// C entry points of the fused normalization library: argument validation,
// per-device caches, dispatch to the per-dtype launchers.
#include <math.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/normfuse.h"
#include "../../include/normfuse_testing.h"
#include "launch.h"

namespace nf {
namespace {

thread_local int g_last_cuda_error = 0;

ln_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return LN_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
std::mutex g_mu;

struct OccEntry {
  const void* fn;
  int block;
  size_t smem;
  int device;
  int blocks;
};
std::vector<OccEntry>& occ_cache() {
  static std::vector<OccEntry> v;
  return v;
}

size_t elem_size(ln_dtype dt) { return dt == LN_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Byte ranges for the overlap check.
struct Range {
  const void* p;
  size_t bytes;
};
bool overlap(const Range& a, const Range& b) {
  if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + a.bytes;
  const uintptr_t b0 = (uintptr_t)b.p, b1 = b0 + b.bytes;
  return a0 < b1 && b0 < a1;
}
bool any_overlap(const Range* outs, int n_out, const Range* ins, int n_in) {
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (overlap(outs[i], ins[j])) return true;
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(outs[i], outs[j])) return true;
  }
  return false;
}

int max_hidden(ln_dtype dt, bool vec) {
  return vec ? kMaxVecSlots * (int)(16 / elem_size(dt)) : kMaxHiddenScalar;
}

template <typename F>
cudaError_t by_dtype(ln_dtype dt, F&& f) {
  switch (dt) {
    case LN_F32: return f(float{});
    case LN_BF16: return f(bf16{});
    default: return f(f16{});
  }
}

}  // namespace

namespace {
// Kernel family per direction; changed only by ln_testing_select_kernels().
std::atomic<int> g_family[3] = {{kFamilyDefault}, {kFamilyDefault}, {kFamilyDefault}};
}  // namespace

int kernel_family(int direction) {
  return g_family[direction].load(std::memory_order_relaxed);
}

int device_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return (int)e;
      g_sm_count[dev] = n;
    }
    *sms = g_sm_count[dev];
    return (int)cudaSuccess;
  }
  return (int)cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

struct SmemEntry {
  const void* fn;
  int device;
  size_t static_bytes;
  size_t optin;       // the device's opt-in shared memory per block
};
std::vector<SmemEntry>& smem_cache() {
  static std::vector<SmemEntry> v;
  return v;
}

// Opt a kernel in to more than 48 KiB of dynamic shared memory. The opt-in
// is a property of the kernel in the current context, which a
// cudaDeviceReset or a caller's own context does not carry over, so it is
// set on every call that needs it, always to the same value (everything
// the device allows beyond the kernel's static shared memory): the call is
// idempotent, and two threads planning different sizes never lower it
// under each other's launch. Only the static size and the device limit,
// which no context changes, are cached.
int allow_dyn_smem(const void* fn, size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  size_t static_bytes = 0, optin = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const SmemEntry* ent = nullptr;
    for (const SmemEntry& s : smem_cache())
      if (s.fn == fn && s.device == dev) ent = &s;
    if (ent == nullptr) {
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, fn);
      if (e != cudaSuccess) return (int)e;
      int opt = 0;
      e = cudaDeviceGetAttribute(&opt, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return (int)e;
      smem_cache().push_back({fn, dev, attr.sharedSizeBytes, (size_t)opt});
      ent = &smem_cache().back();
    }
    static_bytes = ent->static_bytes;
    optin = ent->optin;
  }
  if (smem + static_bytes <= 48 * 1024) return (int)cudaSuccess;
  if (smem + static_bytes > optin) return (int)cudaErrorInvalidValue;
  return (int)cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)(optin - static_bytes));
}

int resident_blocks(const void* fn, int block, size_t smem, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  std::lock_guard<std::mutex> lk(g_mu);
  for (const OccEntry& o : occ_cache()) {
    if (o.fn == fn && o.block == block && o.smem == smem && o.device == dev) {
      *out = o.blocks;
      return (int)cudaSuccess;
    }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem);
  if (e != cudaSuccess) return (int)e;
  occ_cache().push_back({fn, block, smem, dev, n});
  *out = n;
  return (int)cudaSuccess;
}

}  // namespace nf

using namespace nf;

extern "C" {

const char* ln_status_string(ln_status s) {
  switch (s) {
    case LN_OK: return "LN_OK";
    case LN_ERR_NULL: return "LN_ERR_NULL: a required pointer is NULL";
    case LN_ERR_ALIGN: return "LN_ERR_ALIGN: a pointer is not aligned to its element size";
    case LN_ERR_SHAPE: return "LN_ERR_SHAPE: rows < 0 or hidden out of range";
    case LN_ERR_UNSUPPORTED: return "LN_ERR_UNSUPPORTED: unknown dtype or mode";
    case LN_ERR_CUDA: return "LN_ERR_CUDA: a CUDA call failed (see ln_last_cuda_error)";
    case LN_ERR_WORKSPACE: return "LN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case LN_ERR_INVALID: return "LN_ERR_INVALID: bad eps, or outputs overlap inputs";
    case LN_ERR_SCRATCH_LIMIT:
      return "LN_ERR_SCRATCH_LIMIT: the shape needs more scratch than the library's static "
             "array (LN_NOALLOC_SCRATCH_BYTES) holds; use ln_bwd with a workspace";
  }
  return "unknown ln_status";
}

int ln_last_cuda_error(void) { return g_last_cuda_error; }

void nf_set_last_cuda_error(int e) { g_last_cuda_error = e; }

ln_status ln_testing_select_kernels(int forward, int backward, int softmax) {
  const int f[3] = {forward, backward, softmax};
  for (int v : f)
    if (v != LN_TESTING_DEFAULT_KERNELS && v != LN_TESTING_RING_KERNELS) return LN_ERR_INVALID;
  for (int i = 0; i < 3; ++i)
    g_family[i].store(f[i] == LN_TESTING_RING_KERNELS ? kFamilyRing : kFamilyDefault,
                      std::memory_order_relaxed);
  return LN_OK;
}

ln_status ln_testing_plan(int direction, int64_t rows, int64_t hidden, ln_dtype dtype,
                          ln_mode mode, int option, int* out) {
  if (out == nullptr) return LN_ERR_NULL;
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (direction < LN_TESTING_PLAN_FORWARD || direction > LN_TESTING_PLAN_PARTIALS)
    return LN_ERR_UNSUPPORTED;
  if (direction != LN_TESTING_PLAN_SOFTMAX && mode != LN_LAYERNORM && mode != LN_RMSNORM)
    return LN_ERR_UNSUPPORTED;
  if (rows < 1 || hidden < 1) return LN_ERR_SHAPE;
  const size_t es = elem_size(dtype);
  bool vec = (hidden * (int64_t)es) % 16 == 0;
  if (hidden > max_hidden(dtype, vec)) {
    if (!vec || hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
    vec = false;
  }
  const bool rms = mode == LN_RMSNORM;
  Plan p;
  cudaError_t e = by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    switch (direction) {
      case LN_TESTING_PLAN_FORWARD:
        return fwd_plan<T>(rows, (int)hidden, vec, option != 0, rms ? 1 : 2, &p);
      case LN_TESTING_PLAN_BACKWARD:
        return bwd_plan<T>(rows, (int)hidden, rms, option != 0, vec, &p);
      case LN_TESTING_PLAN_SOFTMAX:
        return softmax_plan<T>(rows, (int)hidden, vec, &p);
      default:
        return partials_plan<T>(rows, (int)hidden, vec, &p);
    }
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const int v[6] = {p.kind, p.group, p.n, p.block, p.grid, (int)p.smem};
  for (int i = 0; i < 6; ++i) out[i] = v[i];
  return LN_OK;
}

ln_status ln_device_error(cudaStream_t stream, unsigned* flags) {
  if (flags == nullptr) return LN_ERR_NULL;
  *flags = 0;
  cudaError_t (*readers[])(cudaStream_t, unsigned*) = {
      take_error_fwd_bulk_f32,          take_error_fwd_bulk_bf16,
      take_error_fwd_bulk_f16,          take_error_bwd_bulk_ln_f32,
      take_error_bwd_bulk_ln_bf16,      take_error_bwd_bulk_ln_f16,
      take_error_bwd_bulk_rms_f32,      take_error_bwd_bulk_rms_bf16,
      take_error_bwd_bulk_rms_f16,      take_error_bwd_bulk_ln_dbias_f32,
      take_error_bwd_bulk_ln_dbias_bf16, take_error_bwd_bulk_ln_dbias_f16,
      take_error_bwd_bulk_rms_dbias_f32, take_error_bwd_bulk_rms_dbias_bf16,
      take_error_bwd_bulk_rms_dbias_f16, take_error_softmax_f32,
      take_error_softmax_bf16,          take_error_softmax_f16};
  for (auto r : readers) {
    cudaError_t e = r(stream, flags);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return LN_OK;
}

ln_status ln_fwd(const void* x, const void* bias, const void* residual, const void* gamma,
                 const void* beta, float eps, ln_mode mode, int zero_centered_gamma,
                 void* out_sum, void* y, float* mean, float* rstd, float* amax,
                 cudaStream_t stream, int64_t rows, int64_t hidden, ln_dtype dtype) {
  if (rows > 0 && y == nullptr) return LN_ERR_NULL;
  return ln_fwd_ex(x, bias, residual, gamma, beta, eps, mode, zero_centered_gamma, out_sum, y,
                   mean, rstd, amax, nullptr, nullptr, stream, rows, hidden, dtype);
}

ln_status ln_fwd_ex(const void* x, const void* bias, const void* residual, const void* gamma,
                    const void* beta, float eps, ln_mode mode, int zero_centered_gamma,
                    void* out_sum, void* y, float* mean, float* rstd, float* amax,
                    void* y_fp8, const float* fp8_scale, cudaStream_t stream, int64_t rows,
                    int64_t hidden, ln_dtype dtype) {
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (mode != LN_LAYERNORM && mode != LN_RMSNORM) return LN_ERR_UNSUPPORTED;
  if (rows < 0 || hidden < 1) return LN_ERR_SHAPE;
  if (!(eps >= 0.0f) || !isfinite(eps)) return LN_ERR_INVALID;
  const bool rms = mode == LN_RMSNORM;
  if (rms) {
    beta = nullptr;
    mean = nullptr;
  }
  if (gamma == nullptr) return LN_ERR_NULL;
  if (y_fp8 != nullptr && fp8_scale == nullptr) return LN_ERR_NULL;
  if (rows > 0 && (x == nullptr || (y == nullptr && y_fp8 == nullptr))) return LN_ERR_NULL;
  const size_t es = elem_size(dtype);
  const void* tensors[] = {x, bias, residual, gamma, beta, out_sum, y};
  for (const void* p : tensors)
    if (!aligned(p, es)) return LN_ERR_ALIGN;
  if (!aligned(mean, 4) || !aligned(rstd, 4) || !aligned(amax, 4) || !aligned(fp8_scale, 4))
    return LN_ERR_ALIGN;
  bool vec = (hidden * (int64_t)es) % 16 == 0;
  for (const void* p : tensors)
    if (!aligned(p, 16)) vec = false;
  if (!aligned(y_fp8, 16)) vec = false;
  if (hidden > max_hidden(dtype, vec)) {
    if (!vec || hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
    vec = false;
  }
  const size_t mat = (size_t)rows * (size_t)hidden * es, vecb = (size_t)hidden * es;
  const size_t mat8 = (size_t)rows * (size_t)hidden;
  const Range outs[] = {{out_sum, mat}, {y, mat}, {mean, (size_t)rows * 4},
                        {rstd, (size_t)rows * 4}, {amax, amax ? 4u : 0u}, {y_fp8, mat8}};
  const Range ins[] = {{x, mat}, {residual, mat}, {bias, vecb}, {gamma, vecb}, {beta, vecb},
                       {fp8_scale, fp8_scale ? 4u : 0u}};
  if (any_overlap(outs, 6, ins, 6)) return LN_ERR_INVALID;

  if (amax) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (rows == 0) return LN_OK;

  FwdArgs a;
  a.x = x;
  a.bias = bias;
  a.residual = residual;
  a.gamma = gamma;
  a.beta = beta;
  a.out_sum = out_sum;
  a.y = y;
  a.mean = mean;
  a.rstd = rstd;
  a.amax = reinterpret_cast<unsigned*>(amax);
  a.y_fp8 = static_cast<unsigned char*>(y_fp8);
  a.fp8_scale = y_fp8 ? fp8_scale : nullptr;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.eps = eps;
  a.inv_hidden = 1.0f / (float)hidden;
  a.rms = rms ? 1 : 0;
  a.zero_centered = zero_centered_gamma ? 1 : 0;
  cudaError_t e = by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    Plan p;
    const int n_params = 1 + (bias != nullptr) + (beta != nullptr);
    cudaError_t r = fwd_plan<T>(rows, (int)hidden, vec, residual != nullptr, n_params, &p);
    if (r != cudaSuccess) return r;
    return fwd_launch<T>(a, p, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return LN_OK;
}

ln_status ln_fwd_from_partials(const void* x, const float* psum, const float* psq,
                               int64_t n_tiles, int64_t tile_cols, ln_partials kind,
                               const void* gamma, const void* beta, float eps, ln_mode mode,
                               int zero_centered_gamma, void* y, float* mean, float* rstd,
                               float* amax, cudaStream_t stream, int64_t rows, int64_t hidden,
                               ln_dtype dtype) {
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (mode != LN_LAYERNORM && mode != LN_RMSNORM) return LN_ERR_UNSUPPORTED;
  if (kind != LN_PARTIALS_SUM_SQ && kind != LN_PARTIALS_SUM_M2) return LN_ERR_UNSUPPORTED;
  if (rows < 0 || hidden < 1 || tile_cols < 1) return LN_ERR_SHAPE;
  if (n_tiles != (hidden + tile_cols - 1) / tile_cols) return LN_ERR_SHAPE;
  if (!(eps >= 0.0f) || !isfinite(eps)) return LN_ERR_INVALID;
  const bool rms = mode == LN_RMSNORM;
  if (rms) {
    beta = nullptr;
    mean = nullptr;
  }
  if (gamma == nullptr) return LN_ERR_NULL;
  if (rows > 0 && (x == nullptr || y == nullptr || psum == nullptr || psq == nullptr))
    return LN_ERR_NULL;
  const size_t es = elem_size(dtype);
  const void* tensors[] = {x, gamma, beta, y};
  for (const void* p : tensors)
    if (!aligned(p, es)) return LN_ERR_ALIGN;
  if (!aligned(psum, 4) || !aligned(psq, 4) || !aligned(mean, 4) || !aligned(rstd, 4) ||
      !aligned(amax, 4))
    return LN_ERR_ALIGN;
  bool vec = (hidden * (int64_t)es) % 16 == 0;
  for (const void* p : tensors)
    if (!aligned(p, 16)) vec = false;
  if (hidden > max_hidden(dtype, vec)) {
    if (!vec || hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
    vec = false;
  }
  const size_t mat = (size_t)rows * (size_t)hidden * es, vecb = (size_t)hidden * es;
  const size_t pb = (size_t)rows * (size_t)n_tiles * 4;
  const Range outs[] = {{y, mat}, {mean, (size_t)rows * 4}, {rstd, (size_t)rows * 4},
                        {amax, amax ? 4u : 0u}};
  const Range ins[] = {{x, mat}, {psum, pb}, {psq, pb}, {gamma, vecb}, {beta, vecb}};
  if (any_overlap(outs, 4, ins, 5)) return LN_ERR_INVALID;

  if (amax) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (rows == 0) return LN_OK;
  PartialsArgs a;
  a.x = x;
  a.psum = psum;
  a.psq = psq;
  a.gamma = gamma;
  a.beta = beta;
  a.y = y;
  a.mean = mean;
  a.rstd = rstd;
  a.amax = reinterpret_cast<unsigned*>(amax);
  a.rows = rows;
  a.hidden = (int)hidden;
  a.n_tiles = (int)n_tiles;
  a.tile_cols = (int)(tile_cols < hidden ? tile_cols : hidden);
  a.inv_tile = 1.0f / (float)a.tile_cols;
  a.inv_last = 1.0f / (float)(hidden - (n_tiles - 1) * a.tile_cols);
  a.eps = eps;
  a.inv_hidden = 1.0f / (float)hidden;
  a.kind = kind == LN_PARTIALS_SUM_M2 ? 1 : 0;
  a.rms = rms ? 1 : 0;
  a.zero_centered = zero_centered_gamma ? 1 : 0;
  cudaError_t e = by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    Plan p;
    cudaError_t r = partials_plan<T>(rows, (int)hidden, vec, &p);
    if (r != cudaSuccess) return r;
    return partials_launch(a, p, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return LN_OK;
}

static cudaError_t bwd_plan_any(ln_dtype dtype, int64_t rows, int hidden, bool rms, bool dbias,
                                bool vec, Plan* p) {
  return by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    return bwd_plan<T>(rows, hidden, rms, dbias, vec, p);
  });
}

ln_status ln_softmax_fwd(const void* x, void* y, cudaStream_t stream, int64_t rows,
                         int64_t hidden, ln_dtype dtype) {
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (rows < 0 || hidden < 1) return LN_ERR_SHAPE;
  if (rows > 0 && (x == nullptr || y == nullptr)) return LN_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(y, es)) return LN_ERR_ALIGN;
  bool vec = (hidden * (int64_t)es) % 16 == 0 && aligned(x, 16) && aligned(y, 16);
  if (hidden > max_hidden(dtype, vec)) {
    if (!vec || hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
    vec = false;
  }
  // In place (y == x) is allowed; any other overlap is not.
  const size_t mat = (size_t)rows * (size_t)hidden * es;
  if (x != y && overlap({x, mat}, {y, mat})) return LN_ERR_INVALID;
  if (rows == 0) return LN_OK;

  SmxArgs a;
  a.x = x;
  a.y = y;
  a.rows = rows;
  a.hidden = (int)hidden;
  cudaError_t e = by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    Plan p;
    cudaError_t r = softmax_plan<T>(rows, (int)hidden, vec, &p);
    if (r != cudaSuccess) return r;
    return softmax_launch(a, p, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return LN_OK;
}

ln_status ln_bwd_workspace_bytes(int64_t rows, int64_t hidden, ln_dtype dtype, ln_mode mode,
                                 size_t* bytes) {
  if (bytes == nullptr) return LN_ERR_NULL;
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (mode != LN_LAYERNORM && mode != LN_RMSNORM) return LN_ERR_UNSUPPORTED;
  if (rows < 0 || hidden < 1) return LN_ERR_SHAPE;
  *bytes = 0;
  if (rows == 0) return LN_OK;
  const bool rms = mode == LN_RMSNORM;
  const bool vec_possible = (hidden * (int64_t)elem_size(dtype)) % 16 == 0 &&
                            hidden <= max_hidden(dtype, true);
  if (!vec_possible && hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
  size_t need = 0;
  for (int v = 0; v < 4; ++v) {
    const bool vec = (v & 1) != 0;
    const bool dbias = (v & 2) != 0;   // ln_bwd_ex's layout, so one query serves both calls
    if (vec && !vec_possible) continue;
    if (!vec && hidden > max_hidden(dtype, false)) continue;
    Plan p;
    cudaError_t e = bwd_plan_any(dtype, rows, (int)hidden, rms, dbias, vec, &p);
    if (e != cudaSuccess) return cuda_fail(e);
    const size_t b = (size_t)p.grid * (size_t)p.ws_cols * sizeof(float);
    if (b > need) need = b;
  }
  *bytes = need;
  return LN_OK;
}

ln_status ln_bwd(const void* dy, const void* x_sum, const void* gamma, const float* mean,
                 const float* rstd, void* dx, float* dgamma, float* dbeta, cudaStream_t stream,
                 int64_t rows, int64_t hidden, ln_dtype dtype, ln_mode mode,
                 int zero_centered_gamma, void* workspace, size_t workspace_bytes) {
  return ln_bwd_ex(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, nullptr, stream, rows,
                   hidden, dtype, mode, zero_centered_gamma, workspace, workspace_bytes, LN_F32);
}

ln_status ln_bwd_ex(const void* dy, const void* x_sum, const void* gamma, const float* mean,
                    const float* rstd, void* dx, void* dgamma, void* dbeta, void* dbias,
                    cudaStream_t stream, int64_t rows, int64_t hidden, ln_dtype dtype,
                    ln_mode mode, int zero_centered_gamma, void* workspace,
                    size_t workspace_bytes, ln_dtype grad_dtype) {
  if (dtype != LN_F32 && dtype != LN_BF16 && dtype != LN_F16) return LN_ERR_UNSUPPORTED;
  if (grad_dtype != LN_F32 && grad_dtype != LN_BF16 && grad_dtype != LN_F16)
    return LN_ERR_UNSUPPORTED;
  if (mode != LN_LAYERNORM && mode != LN_RMSNORM) return LN_ERR_UNSUPPORTED;
  if (rows < 0 || hidden < 1) return LN_ERR_SHAPE;
  const bool rms = mode == LN_RMSNORM;
  if (rms) {
    mean = nullptr;
    dbeta = nullptr;
  }
  if (gamma == nullptr || dgamma == nullptr) return LN_ERR_NULL;
  if (rows > 0 && (dy == nullptr || x_sum == nullptr || rstd == nullptr || dx == nullptr ||
                   (!rms && mean == nullptr)))
    return LN_ERR_NULL;
  const size_t es = elem_size(dtype);
  const void* tensors[] = {dy, x_sum, gamma, dx};
  for (const void* p : tensors)
    if (!aligned(p, es)) return LN_ERR_ALIGN;
  const size_t gs = elem_size(grad_dtype);
  if (!aligned(mean, 4) || !aligned(rstd, 4) || !aligned(dgamma, gs) || !aligned(dbeta, gs) ||
      !aligned(dbias, gs))
    return LN_ERR_ALIGN;
  bool vec = (hidden * (int64_t)es) % 16 == 0;
  for (const void* p : tensors)
    if (!aligned(p, 16)) vec = false;
  if (hidden > max_hidden(dtype, vec)) {
    if (!vec || hidden > max_hidden(dtype, false)) return LN_ERR_SHAPE;
    vec = false;
  }
  const size_t mat = (size_t)rows * (size_t)hidden * es;
  const size_t hb = (size_t)hidden * es, h4 = (size_t)hidden * gs, r4 = (size_t)rows * 4;
  const Range outs[] = {{dx, mat}, {dgamma, h4}, {dbeta, h4}, {dbias, h4},
                        {workspace, workspace_bytes}};
  const Range ins[] = {{dy, mat}, {x_sum, mat}, {gamma, hb}, {mean, r4}, {rstd, r4}};
  if (any_overlap(outs, 5, ins, 5)) return LN_ERR_INVALID;

  if (rows == 0) {
    cudaError_t e = cudaMemsetAsync(dgamma, 0, h4, stream);
    if (e == cudaSuccess && dbeta) e = cudaMemsetAsync(dbeta, 0, h4, stream);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, h4, stream);
    return e == cudaSuccess ? LN_OK : cuda_fail(e);
  }
  Plan p;
  cudaError_t e = bwd_plan_any(dtype, rows, (int)hidden, rms, dbias != nullptr, vec, &p);
  if (e != cudaSuccess) return cuda_fail(e);
  const size_t need = (size_t)p.grid * (size_t)p.ws_cols * sizeof(float);
  if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need)
    return LN_ERR_WORKSPACE;

  BwdArgs a;
  a.dy = dy;
  a.x_sum = x_sum;
  a.gamma = gamma;
  a.mean = mean;
  a.rstd = rstd;
  a.dx = dx;
  a.ws = static_cast<float*>(workspace);
  a.rows = rows;
  a.hidden = (int)hidden;
  a.inv_hidden = 1.0f / (float)hidden;
  a.rms = rms ? 1 : 0;
  a.zero_centered = zero_centered_gamma ? 1 : 0;
  a.has_dbias = dbias != nullptr ? 1 : 0;
  a.ws_cols = p.ws_cols;
  e = by_dtype(dtype, [&](auto t) {
    using T = decltype(t);
    return bwd_launch<T>(a, p, dgamma, dbeta, dbias, (int)grad_dtype, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return LN_OK;
}

}  // extern "C"
