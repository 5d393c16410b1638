/*
 * A plain C99 caller of libnormfuse: the boundary used with no Python, no
 * torch and no C++ in the calling program.
 *
 *   abi_from_c check
 *       Host-side validation only (no device needed): the status codes of
 *       rejected calls, the status strings, and that a rejected call writes
 *       nothing.
 *
 *   abi_from_c run DIR DTYPE MODE ROWS HIDDEN EPS
 *       Reads DIR/{x,bias,residual,gamma,beta,dy}.bin (raw elements of
 *       DTYPE: 0 = fp32, 1 = bf16, 2 = fp16; MODE: 0 = LayerNorm,
 *       1 = RMSNorm), runs ln_fwd then ln_bwd on the
 *       device (memory from cudaMalloc, workspace sized by
 *       ln_bwd_workspace_bytes), checks ln_device_error, and writes
 *       DIR/{y,sum,dx}.bin (DTYPE) and DIR/{mean,rstd,dgamma,dbeta,amax}.bin
 *       (fp32).
 *
 * Exit status 0 on success; any failure prints one line and exits 1.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "normfuse.h"
#include "normfuse_testing.h"

static int fail(const char* what, const char* detail) {
  fprintf(stderr, "abi_from_c: %s: %s\n", what, detail);
  return 1;
}

static int expect_status(const char* what, ln_status got, ln_status want) {
  if (got != want) {
    fprintf(stderr, "abi_from_c: %s: status %d (%s), expected %d (%s)\n", what, (int)got,
            ln_status_string(got), (int)want, ln_status_string(want));
    return 1;
  }
  return 0;
}

/* Host-only checks: every call below is rejected before anything is enqueued. */
static int check(void) {
  float host_marker[4] = {-1.0f, -1.0f, -1.0f, -1.0f};
  int bad = 0;
  size_t ws = 0;
  const char* s = ln_status_string(LN_OK);
  if (s == NULL || s[0] == '\0') return fail("ln_status_string", "empty string for LN_OK");
  if (strcmp(ln_status_string(LN_ERR_NULL), ln_status_string(LN_ERR_SHAPE)) == 0)
    return fail("ln_status_string", "two codes share one string");

  /* Missing gamma, missing y, negative rows, hidden 0, unknown dtype/mode, bad eps. */
  bad |= expect_status("ln_fwd gamma NULL",
                       ln_fwd((const void*)16, NULL, NULL, NULL, NULL, 1e-5f, LN_LAYERNORM, 0,
                              NULL, (void*)32, host_marker, NULL, NULL, 0, 4, 64, LN_BF16),
                       LN_ERR_NULL);
  bad |= expect_status("ln_fwd y NULL",
                       ln_fwd((const void*)16, NULL, NULL, (const void*)48, NULL, 1e-5f,
                              LN_LAYERNORM, 0, NULL, NULL, NULL, NULL, NULL, 0, 4, 64, LN_BF16),
                       LN_ERR_NULL);
  bad |= expect_status("ln_fwd rows < 0",
                       ln_fwd((const void*)16, NULL, NULL, (const void*)48, NULL, 1e-5f,
                              LN_LAYERNORM, 0, NULL, (void*)32, NULL, NULL, NULL, 0, -1, 64,
                              LN_BF16),
                       LN_ERR_SHAPE);
  bad |= expect_status("ln_fwd hidden 0",
                       ln_fwd((const void*)16, NULL, NULL, (const void*)48, NULL, 1e-5f,
                              LN_LAYERNORM, 0, NULL, (void*)32, NULL, NULL, NULL, 0, 4, 0,
                              LN_BF16),
                       LN_ERR_SHAPE);
  bad |= expect_status("ln_fwd unknown dtype",
                       ln_fwd((const void*)16, NULL, NULL, (const void*)48, NULL, 1e-5f,
                              LN_LAYERNORM, 0, NULL, (void*)32, NULL, NULL, NULL, 0, 4, 64,
                              (ln_dtype)9),
                       LN_ERR_UNSUPPORTED);
  bad |= expect_status("ln_fwd negative eps",
                       ln_fwd((const void*)16, NULL, NULL, (const void*)48, NULL, -1.0f,
                              LN_LAYERNORM, 0, NULL, (void*)32, NULL, NULL, NULL, 0, 4, 64,
                              LN_BF16),
                       LN_ERR_INVALID);
  bad |= expect_status("ln_fwd odd pointer",
                       ln_fwd((const void*)17, NULL, NULL, (const void*)48, NULL, 1e-5f,
                              LN_LAYERNORM, 0, NULL, (void*)32, NULL, NULL, NULL, 0, 4, 64,
                              LN_BF16),
                       LN_ERR_ALIGN);
  bad |= expect_status("ln_bwd dx overlaps dy",
                       ln_bwd((const void*)16, (const void*)4096, (const void*)8192,
                              (const float*)12288, (const float*)16384, (void*)16, (float*)20480,
                              NULL, 0, 4, 64, LN_BF16, LN_LAYERNORM, 0, (void*)24576, 1 << 20),
                       LN_ERR_INVALID);
  bad |= expect_status("ln_bwd dgamma NULL",
                       ln_bwd((const void*)16, (const void*)32, (const void*)48,
                              (const float*)64, (const float*)80, (void*)96, NULL, NULL, 0, 4,
                              64, LN_BF16, LN_LAYERNORM, 0, (void*)256, 1 << 20),
                       LN_ERR_NULL);
  bad |= expect_status("ln_bwd_workspace_bytes NULL out",
                       ln_bwd_workspace_bytes(4, 64, LN_BF16, LN_LAYERNORM, NULL), LN_ERR_NULL);
  bad |= expect_status("ln_bwd_workspace_bytes bad shape",
                       ln_bwd_workspace_bytes(4, 0, LN_BF16, LN_LAYERNORM, &ws), LN_ERR_SHAPE);
  bad |= expect_status("ln_softmax_fwd x NULL",
                       ln_softmax_fwd(NULL, (void*)32, 0, 4, 64, LN_F32), LN_ERR_NULL);
  bad |= expect_status("ln_device_error NULL flags", ln_device_error(0, NULL), LN_ERR_NULL);
  bad |= expect_status("ln_testing_select_kernels bad family",
                       ln_testing_select_kernels(2, 0, 0), LN_ERR_INVALID);
  bad |= expect_status("ln_testing_plan NULL out",
                       ln_testing_plan(LN_TESTING_PLAN_FORWARD, 16, 384, LN_BF16, LN_LAYERNORM,
                                       1, NULL),
                       LN_ERR_NULL);

  /* A rejected call leaves its outputs untouched (mean is a host array here;
     a call that got past validation would have enqueued device work on it). */
  if (host_marker[0] != -1.0f) return fail("ln_fwd", "a rejected call wrote an output");
  if (bad) return 1;
  printf("check ok\n");
  return 0;
}

static size_t elem_size(int dtype) { return dtype == LN_F32 ? 4u : 2u; }

static int read_file(const char* dir, const char* name, void* dst, size_t bytes) {
  char path[4096];
  FILE* f;
  size_t got;
  snprintf(path, sizeof path, "%s/%s.bin", dir, name);
  f = fopen(path, "rb");
  if (f == NULL) return fail("open", path);
  got = fread(dst, 1, bytes, f);
  fclose(f);
  if (got != bytes) return fail("short read", path);
  return 0;
}

static int write_file(const char* dir, const char* name, const void* src, size_t bytes) {
  char path[4096];
  FILE* f;
  size_t put;
  snprintf(path, sizeof path, "%s/%s.bin", dir, name);
  f = fopen(path, "wb");
  if (f == NULL) return fail("create", path);
  put = fwrite(src, 1, bytes, f);
  fclose(f);
  if (put != bytes) return fail("short write", path);
  return 0;
}

#define CUDA_OK(call)                                                         \
  do {                                                                        \
    cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess) return fail(#call, cudaGetErrorString(e_));        \
  } while (0)

#define LN_OK_OR_FAIL(call)                                                   \
  do {                                                                        \
    ln_status s_ = (call);                                                    \
    if (s_ != LN_OK) return fail(#call, ln_status_string(s_));                \
  } while (0)

enum { IN_X, IN_BIAS, IN_RES, IN_GAMMA, IN_BETA, IN_DY, N_IN };
enum { OUT_Y, OUT_SUM, OUT_DX, N_MAT_OUT };
enum { F_MEAN, F_RSTD, F_DGAMMA, F_DBETA, F_AMAX, N_F32_OUT };

static int run(const char* dir, int dtype, int mode, long long rows, long long hidden,
               float eps) {
  static const char* in_names[N_IN] = {"x", "bias", "residual", "gamma", "beta", "dy"};
  static const char* mat_names[N_MAT_OUT] = {"y", "sum", "dx"};
  static const char* f32_names[N_F32_OUT] = {"mean", "rstd", "dgamma", "dbeta", "amax"};
  const size_t es = elem_size(dtype);
  const size_t mat = (size_t)rows * (size_t)hidden * es, vec = (size_t)hidden * es;
  size_t in_bytes[N_IN], f32_bytes[N_F32_OUT], ws_bytes = 0;
  void *h_in[N_IN], *d_in[N_IN], *h_mat[N_MAT_OUT], *d_mat[N_MAT_OUT];
  float *h_f[N_F32_OUT], *d_f[N_F32_OUT];
  void* ws = NULL;
  unsigned flags = 0;
  int i;

  in_bytes[IN_X] = mat; in_bytes[IN_BIAS] = vec; in_bytes[IN_RES] = mat;
  in_bytes[IN_GAMMA] = vec; in_bytes[IN_BETA] = vec; in_bytes[IN_DY] = mat;
  f32_bytes[F_MEAN] = (size_t)rows * 4; f32_bytes[F_RSTD] = (size_t)rows * 4;
  f32_bytes[F_DGAMMA] = (size_t)hidden * 4; f32_bytes[F_DBETA] = (size_t)hidden * 4;
  f32_bytes[F_AMAX] = 4;

  for (i = 0; i < N_IN; ++i) {
    h_in[i] = malloc(in_bytes[i] ? in_bytes[i] : 1);
    if (h_in[i] == NULL) return fail("malloc", in_names[i]);
    if (read_file(dir, in_names[i], h_in[i], in_bytes[i])) return 1;
    CUDA_OK(cudaMalloc(&d_in[i], in_bytes[i] ? in_bytes[i] : 16));
    CUDA_OK(cudaMemcpy(d_in[i], h_in[i], in_bytes[i], cudaMemcpyHostToDevice));
  }
  for (i = 0; i < N_MAT_OUT; ++i) {
    h_mat[i] = malloc(mat ? mat : 1);
    if (h_mat[i] == NULL) return fail("malloc", mat_names[i]);
    CUDA_OK(cudaMalloc(&d_mat[i], mat ? mat : 16));
  }
  for (i = 0; i < N_F32_OUT; ++i) {
    h_f[i] = (float*)malloc(f32_bytes[i] ? f32_bytes[i] : 1);
    if (h_f[i] == NULL) return fail("malloc", f32_names[i]);
    CUDA_OK(cudaMalloc((void**)&d_f[i], f32_bytes[i] ? f32_bytes[i] : 16));
  }
  LN_OK_OR_FAIL(ln_bwd_workspace_bytes(rows, hidden, (ln_dtype)dtype, (ln_mode)mode, &ws_bytes));
  if (ws_bytes) CUDA_OK(cudaMalloc(&ws, ws_bytes));

  LN_OK_OR_FAIL(ln_fwd(d_in[IN_X], d_in[IN_BIAS], d_in[IN_RES], d_in[IN_GAMMA], d_in[IN_BETA],
                       eps, (ln_mode)mode, 0, d_mat[OUT_SUM], d_mat[OUT_Y], d_f[F_MEAN],
                       d_f[F_RSTD], d_f[F_AMAX], 0, rows, hidden, (ln_dtype)dtype));
  LN_OK_OR_FAIL(ln_bwd(d_in[IN_DY], d_mat[OUT_SUM], d_in[IN_GAMMA], d_f[F_MEAN], d_f[F_RSTD],
                       d_mat[OUT_DX], d_f[F_DGAMMA], d_f[F_DBETA], 0, rows, hidden,
                       (ln_dtype)dtype, (ln_mode)mode, 0, ws, ws_bytes));
  LN_OK_OR_FAIL(ln_device_error(0, &flags));
  if (flags != 0) return fail("ln_device_error", "a kernel reported a failure");
  CUDA_OK(cudaDeviceSynchronize());

  for (i = 0; i < N_MAT_OUT; ++i) {
    CUDA_OK(cudaMemcpy(h_mat[i], d_mat[i], mat, cudaMemcpyDeviceToHost));
    if (write_file(dir, mat_names[i], h_mat[i], mat)) return 1;
  }
  for (i = 0; i < N_F32_OUT; ++i) {
    CUDA_OK(cudaMemcpy(h_f[i], d_f[i], f32_bytes[i], cudaMemcpyDeviceToHost));
    if (write_file(dir, f32_names[i], h_f[i], f32_bytes[i])) return 1;
  }
  for (i = 0; i < N_IN; ++i) { cudaFree(d_in[i]); free(h_in[i]); }
  for (i = 0; i < N_MAT_OUT; ++i) { cudaFree(d_mat[i]); free(h_mat[i]); }
  for (i = 0; i < N_F32_OUT; ++i) { cudaFree(d_f[i]); free(h_f[i]); }
  if (ws) cudaFree(ws);
  printf("run ok: workspace %lu bytes\n", (unsigned long)ws_bytes);
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 2 && strcmp(argv[1], "check") == 0) return check();
  if (argc == 8 && strcmp(argv[1], "run") == 0)
    return run(argv[2], atoi(argv[3]), atoi(argv[4]), atoll(argv[5]), atoll(argv[6]),
               (float)atof(argv[7]));
  fprintf(stderr, "usage: abi_from_c check | abi_from_c run DIR DTYPE MODE ROWS HIDDEN EPS\n");
  return 2;
}
