/* A plain C consumer of the library: one fused DDIM step and one rel-MAE
 * reduction on the GPU through the C ABI alone, with no Python on the path.
 * Built and run by test_gpu_c_consumer.py (needs a GPU).
 *
 *   c_abi_consumer IN OUT
 *   IN:  int64 n, double w, double abar_t, double abar_prev, then x, pred_c,
 *        pred_u as n float32 each;
 *   OUT: x_out as n float32, then the step's M and the reduction's M (double).
 * Exit status 0 on success; 2 for a CUDA error, 3 for a library error (its
 * status and cfg_last_error() go to stderr).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "cfgstep.h"

#define CK(call)                                                            \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));          \
      return 2;                                                             \
    }                                                                       \
  } while (0)
#define CF(call)                                                            \
  do {                                                                      \
    int rc_ = (call);                                                       \
    if (rc_ != CFG_OK) {                                                    \
      fprintf(stderr, "%s: status %d: %s\n", #call, rc_, cfg_last_error()); \
      return 3;                                                             \
    }                                                                       \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int64_t n = 0;
  double w = 0, abar_t = 0, abar_prev = 0;
  if (fread(&n, sizeof n, 1, in) != 1 || fread(&w, sizeof w, 1, in) != 1 ||
      fread(&abar_t, sizeof abar_t, 1, in) != 1 || fread(&abar_prev, sizeof abar_prev, 1, in) != 1 ||
      n <= 0)
    return 1;
  float* host = (float*)malloc(3 * (size_t)n * sizeof(float));
  if (!host || fread(host, sizeof(float), 3 * (size_t)n, in) != 3 * (size_t)n) return 1;
  fclose(in);

  const size_t bytes = (size_t)n * sizeof(float);
  const size_t ws_bytes = cfg_workspace_bytes(n, CFG_F32);
  if (ws_bytes == 0) return 1;
  float *x, *c, *u, *out;
  double* M;
  void* ws;
  cudaStream_t s;
  CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  CK(cudaMalloc((void**)&x, bytes));
  CK(cudaMalloc((void**)&c, bytes));
  CK(cudaMalloc((void**)&u, bytes));
  CK(cudaMalloc((void**)&out, bytes));
  CK(cudaMalloc((void**)&M, 2 * sizeof(double)));
  CK(cudaMalloc(&ws, ws_bytes));
  CK(cudaMemcpyAsync(x, host, bytes, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(c, host + n, bytes, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(u, host + 2 * n, bytes, cudaMemcpyHostToDevice, s));

  CF(cfg_workspace_init(ws, ws_bytes, s));
  CF(cfg_ddim_step(out, x, c, u, n, CFG_F32, (float)w, abar_t, abar_prev, 0.0f, 0, 0, M, NULL,
                   NULL, ws, ws_bytes, s));
  CF(cfg_relmae_reduce(c, u, n, CFG_F32, M + 1, NULL, NULL, 0, ws, ws_bytes, s));
  CK(cudaMemcpyAsync(host, out, bytes, cudaMemcpyDeviceToHost, s));
  double m_host[2];
  CK(cudaMemcpyAsync(m_host, M, sizeof m_host, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));

  FILE* o = fopen(argv[2], "wb");
  if (!o || fwrite(host, sizeof(float), (size_t)n, o) != (size_t)n ||
      fwrite(m_host, sizeof(double), 2, o) != 2)
    return 1;
  fclose(o);
  printf("%s\n", cfg_version());
  CK(cudaFree(x));
  CK(cudaFree(c));
  CK(cudaFree(u));
  CK(cudaFree(out));
  CK(cudaFree(M));
  CK(cudaFree(ws));
  CK(cudaStreamDestroy(s));
  free(host);
  return 0;
}
