/* A plain C11 consumer of libfa: device buffers through the CUDA runtime's C API, one fa_fwd call,
 * and a comparison with the float64 oracle's C library on the same bf16 bytes.  Exit status 0 when
 * max |dO| <= 1.5e-2 beyond bf16 output rounding and max |dLSE| <= 1e-3 (test support only). */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"

int fao_attention(const double* q, const double* k, const double* v, double* o, double* lse, long B, long H,
                  long nq, long nk, long d, double scale);

static uint16_t to_bf16(float x) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int main(void) {
  enum { B = 1, H = 2, NQ = 200, NK = 300, D = 64 };
  const size_t nq = (size_t)B * H * NQ * D, nk = (size_t)B * H * NK * D;
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nk * 2), *hv = malloc(nk * 2), *ho = malloc(nq * 2);
  float* hl = malloc((size_t)B * H * NQ * 4);
  double *dq = malloc(nq * 8), *dk = malloc(nk * 8), *dv = malloc(nk * 8), *ro = malloc(nq * 8);
  double* rl = malloc((size_t)B * H * NQ * 8);
  uint64_t st = 0x9E3779B97F4A7C15ull;
  for (size_t i = 0; i < nq + 2 * nk; ++i) { /* xorshift values in [-2, 2) */
    st ^= st << 13; st ^= st >> 7; st ^= st << 17;
    const float x = (float)((double)(st >> 11) / 9007199254740992.0 * 4.0 - 2.0);
    const uint16_t b = to_bf16(x);
    if (i < nq) { hq[i] = b; dq[i] = from_bf16(b); }
    else if (i < nq + nk) { hk[i - nq] = b; dk[i - nq] = from_bf16(b); }
    else { hv[i - nq - nk] = b; dv[i - nq - nk] = from_bf16(b); }
  }
  void *gq, *gk, *gv, *go;
  float* gl;
  if (cudaMalloc(&gq, nq * 2) || cudaMalloc(&gk, nk * 2) || cudaMalloc(&gv, nk * 2) || cudaMalloc(&go, nq * 2) ||
      cudaMalloc((void**)&gl, (size_t)B * H * NQ * 4)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 2;
  }
  cudaMemcpy(gq, hq, nq * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(gk, hk, nk * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(gv, hv, nk * 2, cudaMemcpyHostToDevice);
  const float scale = 0.125f;
  int rc = fa_fwd(gq, gk, gv, go, gl, B, H, NQ, NK, D, scale, FA_BF16, NULL);
  if (rc != FA_OK) {
    fprintf(stderr, "fa_fwd: %s\n", fa_status_string(rc));
    return 3;
  }
  if (cudaDeviceSynchronize() != cudaSuccess || fa_check_device_error() != FA_OK) return 4;
  cudaMemcpy(ho, go, nq * 2, cudaMemcpyDeviceToHost);
  cudaMemcpy(hl, gl, (size_t)B * H * NQ * 4, cudaMemcpyDeviceToHost);
  if (fao_attention(dq, dk, dv, ro, rl, B, H, NQ, NK, D, scale) != 0) return 5;
  double max_o = 0, max_l = 0;
  for (size_t i = 0; i < nq; ++i) {
    const double ref = ro[i], got = from_bf16(ho[i]);
    const double half_step = ldexp(1.0, (int)floor(log2(fmax(fabs(ref), 1e-30))) - 8);
    const double e = fabs(got - ref) - half_step;
    if (!(e <= max_o)) max_o = isnan(e) ? INFINITY : e;
  }
  for (size_t i = 0; i < (size_t)B * H * NQ; ++i) {
    const double e = fabs((double)hl[i] - rl[i]);
    if (!(e <= max_l)) max_l = isnan(e) ? INFINITY : e;
  }
  printf("c consumer: max|dO| beyond bf16 rounding %.3e, max|dLSE| %.3e\n", max_o, max_l);
  return (max_o <= 1.5e-2 && max_l <= 1e-3) ? 0 : 1;
}
