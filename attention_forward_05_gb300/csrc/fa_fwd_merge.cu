// fa_fwd_merge.cu -- merge of split-KV partial states of the forward pass.
//
// Source: "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com), demo 2: partial states
// (m, l, o) of key segments merge by rescaling to the largest maximum; the merge is
// associative and commutative, and the closing remarks describe splitting one query's keys
// over several SMs (flash-decoding) - here applied to every query row of a prefill.
//
// One warp per query row: M = max m_s, then l and o accumulate over the splits in index order
// with weights 2^(m_s - M) (maxima are in log2 units), and O = o / l is written in the output
// dtype with LSE = (M + log2 l) ln 2.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int MERGE_ROWS_PER_CTA = 8;

template <int D, bool BF16>
__global__ void __launch_bounds__(32 * MERGE_ROWS_PER_CTA)
    fa_fwd_merge_kernel(const float* __restrict__ ws_o, const float2* __restrict__ ws_ml, void* __restrict__ o,
                        float* __restrict__ lse, long long rows, int n_split) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * MERGE_ROWS_PER_CTA + (threadIdx.x >> 5);
  if (row >= rows) return;
  float M = -INFINITY;
  for (int sp = lane; sp < n_split; sp += 32) M = fmaxf(M, ws_ml[sp * rows + row].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int sp = 0; sp < n_split; ++sp) {
    const float2 ml = ws_ml[sp * rows + row];
    const float w = ex2_approx(ml.x - M);
    L = fmaf(ml.y, w, L);
    const float* src = ws_o + (sp * rows + row) * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(src[lane + 32 * e], w, acc[e]);
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    if constexpr (BF16)
      static_cast<__nv_bfloat16*>(o)[row * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
    else
      static_cast<float*>(o)[row * D + lane + 32 * e] = acc[e] * inv;
  }
  if (lse != nullptr && lane == 0) lse[row] = (M + log2f(L)) * 0.6931471805599453f;
}

cudaError_t launch_fwd_merge(const float* ws_o, const float* ws_ml, void* o, float* lse, long long rows, int d,
                             int n_split, int out_bf16, cudaStream_t stream) {
  const long long grid = (rows + MERGE_ROWS_PER_CTA - 1) / MERGE_ROWS_PER_CTA;
  if (grid <= 0 || grid > 0x7FFFFFFFLL || n_split < 1) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid)), b(32 * MERGE_ROWS_PER_CTA);
  const float2* ml = reinterpret_cast<const float2*>(ws_ml);
  if (d == 64 && out_bf16) fa_fwd_merge_kernel<64, true><<<g, b, 0, stream>>>(ws_o, ml, o, lse, rows, n_split);
  else if (d == 64) fa_fwd_merge_kernel<64, false><<<g, b, 0, stream>>>(ws_o, ml, o, lse, rows, n_split);
  else if (out_bf16) fa_fwd_merge_kernel<128, true><<<g, b, 0, stream>>>(ws_o, ml, o, lse, rows, n_split);
  else fa_fwd_merge_kernel<128, false><<<g, b, 0, stream>>>(ws_o, ml, o, lse, rows, n_split);
  return cudaGetLastError();
}

}  // namespace fa
