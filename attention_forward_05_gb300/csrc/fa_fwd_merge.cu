// fa_fwd_merge.cu -- merge of split-KV partial states of the forward pass.
//
// Source: "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com), demo 2: partial states
// (m, l, o) of key segments merge by rescaling to the largest maximum; the merge is
// associative and commutative, and the closing remarks describe splitting one query's keys
// over several SMs (flash-decoding) - here applied to every query row of a prefill.
//
// One warp per query row: M = max m_s, then l and o accumulate over the splits in index order (or
// in a given order: a permutation of the split indices, validated on the device; any other array
// makes the merge write NaN) with weights 2^(m_s - M) (maxima are in log2 units), and O = o / l is
// written in the output dtype with LSE = (M + log2 l) ln 2.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int MERGE_ROWS_PER_CTA = 8;
constexpr int MERGE_MAX_SPLITS = 4096;

template <int D, bool BF16>
__global__ void __launch_bounds__(32 * MERGE_ROWS_PER_CTA)
    fa_fwd_merge_kernel(const float* __restrict__ ws_o, const float2* __restrict__ ws_ml, void* __restrict__ o,
                        float* __restrict__ lse, long long rows, int n_split, const int* __restrict__ order) {
  constexpr int PER = D / 32;
  __shared__ unsigned seen[MERGE_MAX_SPLITS / 32];
  __shared__ int bad;
  griddep_wait();  // launched as a programmatic dependent of the kernel that writes the partial states
  if (order != nullptr) {  // the order must be a permutation of 0 .. n_split - 1
    for (int i = threadIdx.x; i < (n_split + 31) / 32; i += blockDim.x) seen[i] = 0u;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n_split; i += blockDim.x) {
      const int c = order[i];
      if (c < 0 || c >= n_split) {
        bad = 1;
      } else {
        const unsigned bit = 1u << (c & 31);
        if (atomicOr(&seen[c >> 5], bit) & bit) bad = 1;
      }
    }
    __syncthreads();
  }
  const bool invalid = order != nullptr && bad;
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
  // Splits in groups of 32: lane i fetches the (m, l) of the group's i-th split in merge order and
  // forms its weight 2^(m - M); then the states accumulate in merge order, 8 splits' rows loaded at a
  // time, so that the loads of a group are in flight together rather than one after another.
  for (int i0 = 0; i0 < n_split; i0 += 32) {
    const int cnt = min(32, n_split - i0);
    const int i = i0 + lane;
    const int sp_l = i < n_split ? (order == nullptr ? i : (invalid ? 0 : order[i])) : 0;
    const float2 ml_l = i < n_split ? ws_ml[sp_l * rows + row] : make_float2(-INFINITY, 0.f);
    const float w_l = i < n_split ? ex2_approx(ml_l.x - M) : 0.f;
    for (int u0 = 0; u0 < cnt; u0 += 8) {
      float v[8][PER];
      float w[8], lsp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int src_lane = (u0 + u) & 31;
        const int sp = __shfl_sync(0xffffffffu, sp_l, src_lane);
        w[u] = __shfl_sync(0xffffffffu, w_l, src_lane);
        lsp[u] = __shfl_sync(0xffffffffu, ml_l.y, src_lane);
        const float* src = ws_o + (sp * rows + row) * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[u][e] = (u0 + u < cnt) ? src[lane + 32 * e] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u0 + u < cnt) {
          L = fmaf(lsp[u], w[u], L);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(v[u][e], w[u], acc[e]);
        }
      }
    }
  }
  const float inv = invalid ? __int_as_float(0x7fc00000) : 1.f / L;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    if constexpr (BF16)
      static_cast<__nv_bfloat16*>(o)[row * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
    else
      static_cast<float*>(o)[row * D + lane + 32 * e] = acc[e] * inv;
  }
  if (lse != nullptr && lane == 0) lse[row] = invalid ? __int_as_float(0x7fc00000) : (M + log2f(L)) * 0.6931471805599453f;
}

cudaError_t launch_fwd_merge(const float* ws_o, const float* ws_ml, void* o, float* lse, long long rows, int d,
                             int n_split, int out_bf16, cudaStream_t stream, const int* order) {
  const long long grid = (rows + MERGE_ROWS_PER_CTA - 1) / MERGE_ROWS_PER_CTA;
  if (grid <= 0 || grid > 0x7FFFFFFFLL || n_split < 1 || n_split > MERGE_MAX_SPLITS) return cudaErrorInvalidValue;
  const unsigned g = static_cast<unsigned>(grid);
  const int b = 32 * MERGE_ROWS_PER_CTA;
  const float2* ml = reinterpret_cast<const float2*>(ws_ml);
  // a programmatic dependent of the forward that wrote the states: its launch overlaps that grid's tail
  if (d == 64 && out_bf16) return launch_dependent(fa_fwd_merge_kernel<64, true>, g, b, 0, stream, ws_o, ml, o, lse, rows, n_split, order);
  if (d == 64) return launch_dependent(fa_fwd_merge_kernel<64, false>, g, b, 0, stream, ws_o, ml, o, lse, rows, n_split, order);
  if (out_bf16) return launch_dependent(fa_fwd_merge_kernel<128, true>, g, b, 0, stream, ws_o, ml, o, lse, rows, n_split, order);
  return launch_dependent(fa_fwd_merge_kernel<128, false>, g, b, 0, stream, ws_o, ml, o, lse, rows, n_split, order);
}

}  // namespace fa
