// Internal interface between the C entry points (api.cu) and the per-dtype
// translation units that instantiate and launch the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"
#include "partials_kernels.cuh"

namespace nf {

// Largest hidden size each path accepts.
constexpr int kMaxVecSlots = 2048;        // 16-byte vectors per row, vector kernels
constexpr int kMaxHiddenScalar = 8192;    // scalar kernels (shared-memory staged)

// Which kernel a call runs and how it is launched.
struct Plan {
  const void* fn = nullptr;
  bool bulk = false;   // pipelined kernel taking (args, BulkCfg)
  int kind = -1;       // 0 lane group per row, 1 CTA per row, 2 scalar, 3 row group (backward),
                       // 4 lane group from registers, one CTA per row tile,
                       // 5 CTA per row from registers (forward and softmax: one
                       // CTA per row; backward: a persistent grid over the rows),
                       // 6 backward CTA per row with the next row prefetched,
                       // 7 the same with dbeta / dbias summed in shared memory,
                       // 8 with every column sum in shared memory
  int group = 0;       // threads sharing a row
  int n = 0;           // 16-byte vectors per thread per row
  int block = 0;
  size_t smem = 0;     // dynamic shared memory
  int grid = 0;        // CTAs; for the backward also the number of partials
  int ws_cols = 0;     // backward: floats per partial row
  BulkCfg cfg = {0, 0, 0};
};

// Per-device facts, cached (api.cu).
int device_sm_count(int* sms);                                  // returns cudaError_t
int resident_blocks(const void* fn, int block, size_t smem, int* out);  // returns cudaError_t
// Opt `fn` in to `smem` bytes of dynamic shared memory when that plus its
// static shared memory passes the default 48 KiB (cached per kernel).
int allow_dyn_smem(const void* fn, size_t smem);  // returns cudaError_t

// Kernel family per direction (api.cu): 0 = the default for each shape,
// 1 = the bulk-copy ring kernels wherever they apply. Only the testing hook
// ln_testing_select_kernels() changes it; nothing reads the environment.
constexpr int kFamilyForward = 0;
constexpr int kFamilyBackward = 1;
constexpr int kFamilySoftmax = 2;
constexpr int kFamilyDefault = 0;
constexpr int kFamilyRing = 1;
int kernel_family(int direction);

// Kernel tables, one per family and dtype, each defined in its own
// translation unit: (kind, lanes or threads, vectors per thread) -> kernel;
// the backward's also take whether a lane group's row has exactly
// lanes * vectors per thread vectors.
#define NF_DECLARE_TABLES(NAME)                                           \
  const void* fwd_bulk_table_##NAME(int kind, int group, int n);          \
  const void* fwd_reg_table_##NAME(int kind, int group, int n);           \
  const void* bwd_bulk_ln_table_##NAME(int kind, int group, int n, bool exact);       \
  const void* bwd_bulk_rms_table_##NAME(int kind, int group, int n, bool exact);      \
  const void* bwd_bulk_ln_dbias_table_##NAME(int kind, int group, int n, bool exact); \
  const void* bwd_bulk_rms_dbias_table_##NAME(int kind, int group, int n, bool exact); \
  const void* bwd_reg_table_##NAME(int kind, int group, int n);           \
  const void* softmax_table_##NAME(int kind, int group, int n);           \
  const void* partials_table_##NAME(int kind, int group, int n);          \
  cudaError_t take_error_softmax_##NAME(cudaStream_t st, unsigned* out);  \
  cudaError_t take_error_fwd_bulk_##NAME(cudaStream_t st, unsigned* out); \
  cudaError_t take_error_bwd_bulk_ln_##NAME(cudaStream_t st, unsigned* out); \
  cudaError_t take_error_bwd_bulk_rms_##NAME(cudaStream_t st, unsigned* out); \
  cudaError_t take_error_bwd_bulk_ln_dbias_##NAME(cudaStream_t st, unsigned* out); \
  cudaError_t take_error_bwd_bulk_rms_dbias_##NAME(cudaStream_t st, unsigned* out);
NF_DECLARE_TABLES(f32)
NF_DECLARE_TABLES(bf16)
NF_DECLARE_TABLES(f16)
#undef NF_DECLARE_TABLES

// n_params: parameter rows (w, and bias / beta when given).
template <typename T>
cudaError_t fwd_plan(int64_t rows, int hidden, bool vec, bool has_residual, int n_params,
                     Plan* p);
template <typename T> cudaError_t fwd_launch(const FwdArgs& a, const Plan& p, cudaStream_t st);
template <typename T>
cudaError_t bwd_plan(int64_t rows, int hidden, bool rms, bool dbias, bool vec, Plan* p);
template <typename T>
cudaError_t bwd_launch(const BwdArgs& a, const Plan& p, void* dgamma, void* dbeta, void* dbias,
                       int grad_dtype, cudaStream_t st);

// Normalize from partial statistics: plan and launch (plan.cu).
template <typename T> cudaError_t partials_plan(int64_t rows, int hidden, bool vec, Plan* p);
cudaError_t partials_launch(const PartialsArgs& a, const Plan& p, cudaStream_t st);

// Row softmax: plan and launch (plan.cu).
template <typename T> cudaError_t softmax_plan(int64_t rows, int hidden, bool vec, Plan* p);
cudaError_t softmax_launch(const SmxArgs& a, const Plan& p, cudaStream_t st);

// Fixed-order sum of the backward's per-CTA partials (finalize.cu).
// Columns of a partial row: [0, H) dgamma, then [H, 2H) dbeta when `beta_cols`,
// then H columns of dbias when dbias is non-null. out_dtype: 0 fp32,
// 1 bf16, 2 fp16 (the ln_dtype codes) for all three outputs.
cudaError_t launch_bwd_finalize(const float* ws, int P, int C, int H, bool beta_cols,
                                void* dgamma, void* dbeta, void* dbias, int out_dtype,
                                cudaStream_t st);

}  // namespace nf

// Record the cudaError_t that ln_last_cuda_error() reports (api.cu).
extern "C" void nf_set_last_cuda_error(int e);
