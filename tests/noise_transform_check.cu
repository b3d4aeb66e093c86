// Exhaustive accuracy check of the step's Box-Muller factors (built and run by
// test_gpu_noise_transform.py; needs a GPU).
//
// Every uniform the noise uses is u = j / 2^24 with j odd in (0, 2^24), so each
// factor of the pair (rho cos theta, rho sin theta) -- rho = sqrt(-2 ln u_a)
// and sin, cos of theta = 2 pi u_b -- takes 2^23 values.  This evaluates both
// transforms of cfg_noise.cuh on all of them and compares with fp64 values
// from CUDA's double-precision log, sinpi and cospi (errors near 1e-16, far
// below the fp32 errors measured).  Printed, one JSON object:
//   rho_abs, sin_abs, cos_abs      max absolute error of each factor;
//   rho_ulp, sin_ulp, cos_ulp      max error in units of the fp32 ulp of the
//                                  exact value (for the full-accuracy transform).
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <cmath>

#include "cfg_noise.cuh"

using namespace cfg_noise;

__device__ unsigned long long g_err[2][6];

__device__ __forceinline__ void record(int t, int k, double e) {
  atomicMax(&g_err[t][k], static_cast<unsigned long long>(__double_as_longlong(e)));
}

__device__ __forceinline__ double ulp_f32(double v) {
  const double a = fabs(v);
  if (a < 0x1p-126) return 0x1p-149;
  int e;
  frexp(a, &e);                     // a = m 2^e, m in [1/2, 1)
  return ldexp(1.0, e - 24);
}

__global__ void check() {
  for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < (1u << 23);
       t += gridDim.x * blockDim.x) {
    const uint32_t j = 2u * t + 1u;
    const double u = static_cast<double>(j) * 0x1p-24;
    const double rho = sqrt(-2.0 * log(u));
    const double sn = sinpi(2.0 * u), cs = cospi(2.0 * u);
    float s0, c0, s1, c1;
    bm_sincos(j, s0, c0);
    bm_sincos_bf16(j, s1, c1);
    const double r0 = bm_rho(j), r1 = bm_rho_bf16(j);
    record(0, 0, fabs(r0 - rho));
    record(0, 1, fabs(s0 - sn));
    record(0, 2, fabs(c0 - cs));
    record(0, 3, fabs(r0 - rho) / ulp_f32(rho));
    record(0, 4, fabs(s0 - sn) / ulp_f32(sn));
    record(0, 5, fabs(c0 - cs) / ulp_f32(cs));
    record(1, 0, fabs(r1 - rho));
    record(1, 1, fabs(s1 - sn));
    record(1, 2, fabs(c1 - cs));
    record(1, 3, fabs(r1 - rho) / ulp_f32(rho));
    record(1, 4, fabs(s1 - sn) / ulp_f32(sn));
    record(1, 5, fabs(c1 - cs) / ulp_f32(cs));
  }
}

int main() {
  unsigned long long zero[2][6] = {};
  if (cudaMemcpyToSymbol(g_err, zero, sizeof(zero)) != cudaSuccess) return 2;
  check<<<1184, 256>>>();
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    fprintf(stderr, "%s\n", cudaGetErrorString(e));
    return 1;
  }
  unsigned long long bits[2][6];
  if (cudaMemcpyFromSymbol(bits, g_err, sizeof(bits)) != cudaSuccess) return 2;
  const char* names[6] = {"rho_abs", "sin_abs", "cos_abs", "rho_ulp", "sin_ulp", "cos_ulp"};
  const char* which[2] = {"full", "bf16"};
  printf("{");
  for (int t = 0; t < 2; ++t) {
    printf("%s\"%s\": {", t ? ", " : "", which[t]);
    for (int k = 0; k < 6; ++k) {
      double d;
      memcpy(&d, &bits[t][k], sizeof d);
      printf("%s\"%s\": %.6e", k ? ", " : "", names[k], d);
    }
    printf("}");
  }
  printf("}\n");
  return 0;
}
