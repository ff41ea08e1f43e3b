/* A plain C11 consumer of libfa: device buffers through the CUDA runtime's C API, one fa_fwd call and
 * one fa_decode_splitkv call, each compared with the float64 oracle's C library on the same bf16 bytes.
 * Exit status 0 when max |dO| <= 1.5e-2 beyond bf16 output rounding for both and the forward's
 * max |dLSE| <= 1e-3 (test support only). */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"

int fao_attention(const double* q, const double* k, const double* v, double* o, double* lse, long B, long H,
                  long nq, long nk, long d, double scale);
int fao_decode_splitkv(const double* q, const double* k, const double* v, double* o, double* lse, long BH, long nk,
                       long d, long splits, double scale, const int* order);

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

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint16_t next_bf16(double* exact) { /* xorshift values in [-2, 2), rounded to bf16 */
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 7;
  rng_state ^= rng_state << 17;
  const float x = (float)((double)(rng_state >> 11) / 9007199254740992.0 * 4.0 - 2.0);
  const uint16_t b = to_bf16(x);
  *exact = from_bf16(b);
  return b;
}

/* largest |got - ref| beyond half a bf16 step of ref */
static double err_beyond_bf16(const uint16_t* got, const double* ref, size_t n) {
  double worst = 0;
  for (size_t i = 0; i < n; ++i) {
    const double half_step = ldexp(1.0, (int)floor(log2(fmax(fabs(ref[i]), 1e-30))) - 8);
    const double e = fabs(from_bf16(got[i]) - ref[i]) - half_step;
    if (!(e <= worst)) worst = isnan(e) ? INFINITY : e;
  }
  return worst;
}

/* One-query-per-head decode, Nk keys in `splits` chunks: fa_decode_splitkv against the oracle's
 * split-and-merge in index order (scale 1/sqrt(d)).  Returns max |dO| beyond bf16 rounding, or a
 * negative value when a call fails. */
static double decode_check(void) {
  enum { B = 2, H = 3, NK = 1000, D = 64, SPLITS = 7 };
  const size_t nq = (size_t)B * H * D, nk = (size_t)B * H * NK * D;
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nk * 2), *hv = malloc(nk * 2), *ho = malloc(nq * 2);
  double *dq = malloc(nq * 8), *dk = malloc(nk * 8), *dv = malloc(nk * 8), *ro = malloc(nq * 8);
  double* rl = malloc((size_t)B * H * 8);
  for (size_t i = 0; i < nq; ++i) hq[i] = next_bf16(&dq[i]);
  for (size_t i = 0; i < nk; ++i) hk[i] = next_bf16(&dk[i]);
  for (size_t i = 0; i < nk; ++i) hv[i] = next_bf16(&dv[i]);
  void *gq, *gk, *gv, *go;
  if (cudaMalloc(&gq, nq * 2) || cudaMalloc(&gk, nk * 2) || cudaMalloc(&gv, nk * 2) || cudaMalloc(&go, nq * 2))
    return -2;
  cudaMemcpy(gq, hq, nq * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(gk, hk, nk * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(gv, hv, nk * 2, cudaMemcpyHostToDevice);
  const int rc = fa_decode_splitkv(gq, gk, gv, go, B, H, NK, D, SPLITS, NULL);
  if (rc != FA_OK) {
    fprintf(stderr, "fa_decode_splitkv: %s\n", fa_status_string(rc));
    return -3;
  }
  if (cudaDeviceSynchronize() != cudaSuccess || fa_check_device_error() != FA_OK) return -4;
  cudaMemcpy(ho, go, nq * 2, cudaMemcpyDeviceToHost);
  if (fao_decode_splitkv(dq, dk, dv, ro, rl, (long)B * H, NK, D, SPLITS, 1.0 / sqrt((double)D), NULL) != 0)
    return -5;
  const double e = err_beyond_bf16(ho, ro, nq);
  cudaFree(gq);
  cudaFree(gk);
  cudaFree(gv);
  cudaFree(go);
  free(hq); free(hk); free(hv); free(ho); free(dq); free(dk); free(dv); free(ro); free(rl);
  return e;
}

int main(void) {
  enum { B = 1, H = 2, NQ = 200, NK = 300, D = 64 };
  const size_t nq = (size_t)B * H * NQ * D, nk = (size_t)B * H * NK * D;
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nk * 2), *hv = malloc(nk * 2), *ho = malloc(nq * 2);
  float* hl = malloc((size_t)B * H * NQ * 4);
  double *dq = malloc(nq * 8), *dk = malloc(nk * 8), *dv = malloc(nk * 8), *ro = malloc(nq * 8);
  double* rl = malloc((size_t)B * H * NQ * 8);
  for (size_t i = 0; i < nq; ++i) hq[i] = next_bf16(&dq[i]);
  for (size_t i = 0; i < nk; ++i) hk[i] = next_bf16(&dk[i]);
  for (size_t i = 0; i < nk; ++i) hv[i] = next_bf16(&dv[i]);
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
  const double max_o = err_beyond_bf16(ho, ro, nq);
  double max_l = 0;
  for (size_t i = 0; i < (size_t)B * H * NQ; ++i) {
    const double e = fabs((double)hl[i] - rl[i]);
    if (!(e <= max_l)) max_l = isnan(e) ? INFINITY : e;
  }
  const double max_dec = decode_check();
  if (max_dec < 0) return (int)(-max_dec) + 4;
  printf("c consumer: fa_fwd max|dO| beyond bf16 rounding %.3e, max|dLSE| %.3e; "
         "fa_decode_splitkv max|dO| beyond bf16 rounding %.3e\n", max_o, max_l, max_dec);
  return (max_o <= 1.5e-2 && max_l <= 1e-3 && max_dec <= 1.5e-2) ? 0 : 1;
}
