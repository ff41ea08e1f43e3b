// fa_decode.cu -- split-KV decode for one query per head (flash-decoding).
//
// Sources (web pages, cited by title and section):
//   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
//
// Kernel 1 (split): one CTA per (batch*head, chunk).  The chunk's keys and
// values are streamed once from HBM with 16-byte non-allocating loads; each
// group of D/8 lanes holds one key row (8 bf16 per lane), dots it with the
// query by a shuffle reduction, and folds it into a running (m, l, o) with the
// one-pass update of [T3] attn_row_1pass (alpha = 2^(m - m_new)).  The
// per-group states of the CTA are merged and written as one fp32 partial
// state (m, l, o[D]) with o unnormalised ([T3] demo 2).
// Kernel 2 (merge): one warp per (batch*head) merges the chunk states in the
// given order and writes O = o / l as bf16 ([T3] demo 2: the merge is
// associative and commutative, so any order gives the same result up to
// rounding).
//
// All maxima are kept in log2 units (scores pre-multiplied by scale*log2 e).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int DEC_UNROLL = 8;        // 16-byte loads in flight per lane, per operand
constexpr int MERGE_THREADS = 128;   // 4 warps = 4 heads per CTA
constexpr int MAX_SPLITS = 4096;

template <int D>
__global__ void __launch_bounds__(DEC_THREADS) fa_decode_split_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    float* __restrict__ ws_m, float* __restrict__ ws_l, float* __restrict__ ws_o, int Nk, int splits, int L,
    float c) {
  constexpr int LPK = D / 8;     // lanes per key row
  constexpr int KPW = 32 / LPK;  // key rows per warp-wide load
  constexpr int U = DEC_UNROLL;
  __shared__ float sm_m[DEC_WARPS], sm_l[DEC_WARPS];
  griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to complete
  __shared__ float sm_o[DEC_WARPS][D];

  const int split = blockIdx.x % splits;
  const int bh = blockIdx.x / splits;
  const int k0 = split * L;
  const int k1 = min(Nk, k0 + L);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane / LPK;
  const int sub = lane % LPK;

  float qf[8];
  {
    const uint4 w = *reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * D + sub * 8);
    qf[0] = bf16lo(w.x) * c; qf[1] = bf16hi(w.x) * c;
    qf[2] = bf16lo(w.y) * c; qf[3] = bf16hi(w.y) * c;
    qf[4] = bf16lo(w.z) * c; qf[5] = bf16hi(w.z) * c;
    qf[6] = bf16lo(w.w) * c; qf[7] = bf16hi(w.w) * c;
  }
  float m = -INFINITY, l = 0.f;
  float o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;

  const __nv_bfloat16* kb = k + static_cast<size_t>(bh) * Nk * D + sub * 8;
  const __nv_bfloat16* vb = v + static_cast<size_t>(bh) * Nk * D + sub * 8;
  for (int base = k0 + warp * U * KPW; base < k1; base += DEC_WARPS * U * KPW) {
    uint4 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = base + u * KPW + g;
      kr[u] = key < k1 ? ldg_stream(kb + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = base + u * KPW + g;
      vr[u] = key < k1 ? ldg_stream(vb + static_cast<size_t>(key) * D) : make_uint4(0, 0, 0, 0);
    }
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 w = kr[u];
      float a = qf[0] * bf16lo(w.x);
      a = fmaf(qf[1], bf16hi(w.x), a);
      a = fmaf(qf[2], bf16lo(w.y), a);
      a = fmaf(qf[3], bf16hi(w.y), a);
      a = fmaf(qf[4], bf16lo(w.z), a);
      a = fmaf(qf[5], bf16hi(w.z), a);
      a = fmaf(qf[6], bf16lo(w.w), a);
      a = fmaf(qf[7], bf16hi(w.w), a);
      s[u] = a;
    }
#pragma unroll
    for (int off = 1; off < LPK; off <<= 1)
#pragma unroll
      for (int u = 0; u < U; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + u * KPW + g >= k1) s[u] = -INFINITY;
      mx = fmaxf(mx, s[u]);
    }
    const float m_new = fmaxf(m, mx);
    const bool any = m_new != -INFINITY;  // false only while this group has seen no valid key
    const float alpha = any ? ex2_approx(m - m_new) : 1.f;
    float psum = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float pu = any ? ex2_approx(s[u] - m_new) : 0.f;
      psum += pu;
      const uint4 w = vr[u];
      o[0] = fmaf(pu, bf16lo(w.x), o[0]);
      o[1] = fmaf(pu, bf16hi(w.x), o[1]);
      o[2] = fmaf(pu, bf16lo(w.y), o[2]);
      o[3] = fmaf(pu, bf16hi(w.y), o[3]);
      o[4] = fmaf(pu, bf16lo(w.z), o[4]);
      o[5] = fmaf(pu, bf16hi(w.z), o[5]);
      o[6] = fmaf(pu, bf16lo(w.w), o[6]);
      o[7] = fmaf(pu, bf16hi(w.w), o[7]);
    }
    l = l * alpha + psum;
    m = m_new;
  }

  // merge the KPW lane groups of this warp (lanes with equal `sub`)
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float M = fmaxf(m, m2);
    const float wa = (m == -INFINITY) ? 0.f : ex2_approx(m - M);
    const float wb = (m2 == -INFINITY) ? 0.f : ex2_approx(m2 - M);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float o2 = __shfl_xor_sync(0xffffffffu, o[e], off);
      o[e] = o[e] * wa + o2 * wb;
    }
    l = l * wa + l2 * wb;
    m = M;
  }
  if (lane < LPK) {
    if (lane == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_o[warp][sub * 8 + e] = o[e];
  }
  __syncthreads();
  // merge the warps; thread i < D finishes dimension i
  if (threadIdx.x < D) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, sm_m[w]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float wt = (sm_m[w] == -INFINITY) ? 0.f : ex2_approx(sm_m[w] - M);
      Ls = fmaf(sm_l[w], wt, Ls);
      Os = fmaf(sm_o[w][threadIdx.x], wt, Os);
    }
    const size_t st = static_cast<size_t>(bh) * splits + split;
    ws_o[st * D + threadIdx.x] = Os;
    if (threadIdx.x == 0) {
      ws_m[st] = M;
      ws_l[st] = Ls;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(MERGE_THREADS) fa_decode_merge_kernel(
    const float* __restrict__ ws_m, const float* __restrict__ ws_l, const float* __restrict__ ws_o,
    const int* __restrict__ order, __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int BH, int splits) {
  constexpr int PER = D / 32;  // output dimensions per lane (lane-strided)
  __shared__ unsigned seen[MAX_SPLITS / 32];
  __shared__ int bad;
  griddep_wait();  // launched as a programmatic dependent of the split kernel that writes the states
  if (order != nullptr) {  // the order must be a permutation of 0..splits-1
    for (int i = threadIdx.x; i < (splits + 31) / 32; i += blockDim.x) seen[i] = 0u;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < splits; i += blockDim.x) {
      const int cidx = order[i];
      if (cidx < 0 || cidx >= splits) {
        bad = 1;
      } else {
        const unsigned bit = 1u << (cidx & 31);
        if (atomicOr(&seen[cidx >> 5], bit) & bit) bad = 1;
      }
    }
    __syncthreads();
  }
  const bool invalid = (order != nullptr) && bad;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x * (MERGE_THREADS / 32) + warp;
  if (bh >= BH) return;
  const float* mh = ws_m + static_cast<size_t>(bh) * splits;
  const float* lh = ws_l + static_cast<size_t>(bh) * splits;
  const float* oh = ws_o + static_cast<size_t>(bh) * splits * D;

  float M = -INFINITY;
  for (int i = lane; i < splits; i += 32) M = fmaxf(M, mh[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float Ls = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  // Chunks in groups of 32: lane i fetches the (m, l) of the group's i-th chunk in merge order and
  // forms its weight; the states then accumulate in merge order, eight chunks' o rows loaded at a time
  // so that a head's loads are in flight together rather than one after another.
  for (int i0 = 0; i0 < splits; i0 += 32) {
    const int cnt = min(32, splits - i0);
    const int i = i0 + lane;
    const int c_l = i < splits ? ((order == nullptr) ? i : (invalid ? 0 : order[i])) : 0;
    const float m_l = i < splits ? mh[c_l] : -INFINITY;
    const float l_l = i < splits ? lh[c_l] : 0.f;
    const float w_l = (m_l == -INFINITY) ? 0.f : ex2_approx(m_l - M);
    for (int u0 = 0; u0 < cnt; u0 += 8) {
      float v[8][PER];
      float w[8], lw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int src_lane = (u0 + u) & 31;
        const int cidx = __shfl_sync(0xffffffffu, c_l, src_lane);
        w[u] = __shfl_sync(0xffffffffu, w_l, src_lane);
        lw[u] = __shfl_sync(0xffffffffu, l_l, src_lane);
#pragma unroll
        for (int e = 0; e < PER; ++e)
          v[u][e] = (u0 + u < cnt) ? oh[static_cast<size_t>(cidx) * D + lane + 32 * e] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u0 + u < cnt) {
          Ls = fmaf(lw[u], w[u], Ls);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(v[u][e], w[u], acc[e]);
        }
      }
    }
  }
  const float inv = invalid ? __int_as_float(0x7fc00000) : 1.f / Ls;
#pragma unroll
  for (int e = 0; e < PER; ++e) o[static_cast<size_t>(bh) * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
  if (lse != nullptr && lane == 0)
    lse[bh] = invalid ? __int_as_float(0x7fc00000) : (M + log2f(Ls)) * 0.6931471805599453f;
}

template <int D>
static cudaError_t launch_decode_d(const DecodeLaunch& a) {
  const int L = (a.Nk + a.splits - 1) / a.splits;
  const size_t n_states = static_cast<size_t>(a.BH) * a.splits;
  float* ws_m = a.ws;
  float* ws_l = a.ws + n_states;
  float* ws_o = a.ws + 2 * n_states;
  const long long grid1 = static_cast<long long>(a.BH) * a.splits;
  if (grid1 <= 0 || grid1 > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  fa_decode_split_kernel<D><<<static_cast<unsigned>(grid1), DEC_THREADS, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), ws_m, ws_l, ws_o, a.Nk, a.splits, L, a.c);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int heads_per_cta = MERGE_THREADS / 32;
  const unsigned grid2 = static_cast<unsigned>((a.BH + heads_per_cta - 1) / heads_per_cta);
  return launch_dependent(fa_decode_merge_kernel<D>, grid2, MERGE_THREADS, 0, a.stream, ws_m, ws_l, ws_o, a.order,
                          static_cast<__nv_bfloat16*>(a.o), a.lse, a.BH, a.splits);
}

cudaError_t launch_decode_merge(const float* ws_m, const float* ws_l, const float* ws_o, const int* order, void* o,
                                float* lse, int BH, int splits, int d, cudaStream_t stream) {
  if (splits < 1 || splits > MAX_SPLITS || BH < 1) return cudaErrorInvalidValue;
  const int heads_per_cta = MERGE_THREADS / 32;
  const unsigned grid = static_cast<unsigned>((BH + heads_per_cta - 1) / heads_per_cta);
  // a programmatic dependent of the split kernel that wrote the states
  if (d == 64)
    return launch_dependent(fa_decode_merge_kernel<64>, grid, MERGE_THREADS, 0, stream, ws_m, ws_l, ws_o, order,
                            static_cast<__nv_bfloat16*>(o), lse, BH, splits);
  if (d == 128)
    return launch_dependent(fa_decode_merge_kernel<128>, grid, MERGE_THREADS, 0, stream, ws_m, ws_l, ws_o, order,
                            static_cast<__nv_bfloat16*>(o), lse, BH, splits);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeLaunch& a) {
  if (a.splits < 1 || a.splits > MAX_SPLITS) return cudaErrorInvalidValue;
  if (a.d == 64) return launch_decode_d<64>(a);
  if (a.d == 128) return launch_decode_d<128>(a);
  return cudaErrorInvalidValue;
}

}  // namespace fa
