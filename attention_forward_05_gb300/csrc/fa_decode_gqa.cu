// fa_decode_gqa.cu -- split-KV decode for grouped-query heads: G query heads share one key/value head.
//
// Sources (web pages, cited by title and section):
//   [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io), §7: MQA/GQA as an
//        extension (several query heads read one key/value head).
//   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com), demo 2: split-KV (flash-decoding)
//        partial states (m, l, o) and their order-independent merge.
//
// One CTA per (batch, key/value head, chunk).  A producer warp streams the chunk's K and V rows from
// HBM into a shared-memory ring with 1-D bulk copies (each head's rows are contiguous), so every key
// row leaves HBM once however many query heads read it.  Consumer warps read the rows from
// shared memory; a group of D/8 lanes holds 8 dims of one row and keeps, in registers, the running
// (m, l, o) of up to four query heads with the one-pass update of [T3] attn_row_1pass in base 2
// (packed f32x2 arithmetic; o is rescaled only when a maximum grows past a threshold, as in the
// forward).  With eight or more query heads per CTA, sets of four warps take four heads each and
// all read the same staged rows.  The groups' states are merged in the CTA and written as one fp32 partial state per
// (query head, chunk), in the layout the decode merge kernel reads.
//
// The work is HBM-bound for G <= 8 (at most 8 FLOP per byte of K/V), so it runs on the FMA pipes;
// the tensor cores would need M >= 64 rows where a group has G <= 8 queries.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

enum : int { WG_FULL = 0x41, WG_EMPTY, WG_DRAIN };

}  // namespace

template <int D_, int G_>
struct DecGqaCfg {
  static constexpr int D = D_;
  static constexpr int G = G_;                // query heads per key/value head handled by one CTA
  static constexpr int GW = G < 4 ? G : 4;    // query heads per consumer warp
  static constexpr int NQG = G / GW;          // warp sets; each reads every staged row
  static constexpr int T = 64;                // keys per ring stage
  static constexpr int STAGES = D == 64 ? 4 : 2;
  static constexpr int WPS = 4;               // consumer warps per set
  static constexpr int CWARPS = WPS * NQG;    // consumer warps
  static constexpr int NTHREADS = (CWARPS + 1) * 32;
  static constexpr int MINB = NQG > 1 ? 2 : 3;  // CTAs per SM the register budget is sized for
  static constexpr int LPK = D / 8;           // lanes per key row
  static constexpr int KPW = 32 / LPK;        // rows per warp per pass
  static constexpr int ROWS_PER_PASS = WPS * KPW;
  static constexpr int U = NQG > 1 ? 1 : 2;   // rows per lane group per iteration (two fit the registers up to 4 heads)
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = T * ROW_BYTES;   // one of K, V
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 2 * STAGES * 8 + 16;
  static_assert(T % (U * ROWS_PER_PASS) == 0, "whole iterations per tile");
  static_assert(G % GW == 0, "whole warp sets");
};

// lazy rescale threshold (log2 units): a query's reference maximum moves only when a score exceeds
// it by more than this, so p = 2^(s - m_ref) <= 2^8 and o, l keep sharing m_ref
constexpr float kGqaTau = 8.f;

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, C::MINB) fa_decode_gqa_split_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    float* __restrict__ ws_m, float* __restrict__ ws_l, float* __restrict__ ws_o, int* err, int Nk, int splits,
    int L, int H, int Hkv, int qgroups, float c) {
  constexpr int D = C::D, G = C::G, GW = C::GW;
  griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to complete
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float sm_m[C::WPS][G], sm_l[C::WPS][G];
  __shared__ float sm_o[C::WPS][G][D];
  __shared__ int abort_word;

  // blockIdx.x = ((b * Hkv + kvh) * qgroups + qg) * splits + split
  const int split = blockIdx.x % splits;
  const int rest = blockIdx.x / splits;
  const int qg = rest % qgroups;
  const int kvbh = rest / qgroups;
  const int b = kvbh / Hkv;
  const int kvh = kvbh % Hkv;
  const int group = H / Hkv;
  const int h0 = kvh * group + qg * G;  // first query head of this CTA
  const int k0 = split * L;
  const int k1 = min(Nk, k0 + L);
  const int n_tiles = k1 > k0 ? (k1 - k0 + C::T - 1) / C::T : 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  auto bar_full = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
  auto bar_empty = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
  volatile int* abort_flag = &abort_word;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), C::CWARPS);
    }
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const size_t head_off = static_cast<size_t>(kvbh) * Nk * D;
  if (warp == C::CWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int n_done = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % C::STAGES;
        if (!mbar_wait(bar_empty(s), ((t / C::STAGES) & 1) ^ 1, abort_flag, err, WG_EMPTY)) break;
        const int r0 = k0 + t * C::T;
        const uint32_t bytes = static_cast<uint32_t>(min(C::T, k1 - r0)) * C::ROW_BYTES;
        mbar_expect_tx(bar_full(s), 2 * bytes);
        bulk_copy_g2s(sbase + s * C::STAGE_BYTES, k + head_off + static_cast<size_t>(r0) * D, bytes, bar_full(s));
        bulk_copy_g2s(sbase + s * C::STAGE_BYTES + C::TILE_BYTES, v + head_off + static_cast<size_t>(r0) * D, bytes,
                      bar_full(s));
        n_done = t + 1;
      }
      for (int s = 0; s < C::STAGES; ++s) {  // drain the copies issued above
        const int cnt = n_done > s ? (n_done - 1 - s) / C::STAGES + 1 : 0;
        if (cnt > 0) mbar_wait_drain(bar_full(s), (cnt - 1) & 1, err, WG_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int wset = warp / C::WPS;  // warp set: query heads [wset * GW, wset * GW + GW)
    const int wi = warp % C::WPS;    // warp within the set
    const int gidx = lane / C::LPK;  // row within the warp's pass
    const int sub = lane % C::LPK;   // 8-dim slice
    uint64_t q2[GW][4], o2[GW][4];   // packed fp32 pairs: dims (2i, 2i + 1) of the lane's slice
    float m[GW], l[GW];
    const uint64_t c2 = f2_pack(c, c);
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(
          q + (static_cast<size_t>(b) * H + h0 + wset * GW + g) * D + sub * 8);
      q2[g][0] = f2_mul(f2_pack(bf16lo(w.x), bf16hi(w.x)), c2);
      q2[g][1] = f2_mul(f2_pack(bf16lo(w.y), bf16hi(w.y)), c2);
      q2[g][2] = f2_mul(f2_pack(bf16lo(w.z), bf16hi(w.z)), c2);
      q2[g][3] = f2_mul(f2_pack(bf16lo(w.w), bf16hi(w.w)), c2);
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[g][e] = 0ull;
    }
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % C::STAGES;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_full(s), (t / C::STAGES) & 1, abort_flag, err, WG_FULL));
      if (!ok) break;
      const uint8_t* kt = smem + s * C::STAGE_BYTES;
      const uint8_t* vt = kt + C::TILE_BYTES;
      const int r_lim = k1 - (k0 + t * C::T);  // valid rows in this tile
#pragma unroll 1
      for (int it = 0; it < C::T / (C::U * C::ROWS_PER_PASS); ++it) {
        // rows r[u] = (it * U + u) * ROWS_PER_PASS + wi * KPW + gidx of the tile
        bool valid[C::U];
        uint64_t k2[C::U][4], v2[C::U][4];
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
          const int r = (it * C::U + u) * C::ROWS_PER_PASS + wi * C::KPW + gidx;
          // rows past the chunk end hold stale bytes (possibly not even numbers): read zeros instead
          valid[u] = r < r_lim;
          const uint4 zero = make_uint4(0, 0, 0, 0);
          const uint4 kw = valid[u] ? *reinterpret_cast<const uint4*>(kt + r * C::ROW_BYTES + sub * 16) : zero;
          const uint4 vw = valid[u] ? *reinterpret_cast<const uint4*>(vt + r * C::ROW_BYTES + sub * 16) : zero;
          k2[u][0] = f2_pack(bf16lo(kw.x), bf16hi(kw.x));
          k2[u][1] = f2_pack(bf16lo(kw.y), bf16hi(kw.y));
          k2[u][2] = f2_pack(bf16lo(kw.z), bf16hi(kw.z));
          k2[u][3] = f2_pack(bf16lo(kw.w), bf16hi(kw.w));
          v2[u][0] = f2_pack(bf16lo(vw.x), bf16hi(vw.x));
          v2[u][1] = f2_pack(bf16lo(vw.y), bf16hi(vw.y));
          v2[u][2] = f2_pack(bf16lo(vw.z), bf16hi(vw.z));
          v2[u][3] = f2_pack(bf16lo(vw.w), bf16hi(vw.w));
        }
        float sc[C::U][GW];
#pragma unroll
        for (int u = 0; u < C::U; ++u)
#pragma unroll
          for (int g = 0; g < GW; ++g) {
            uint64_t a2 = f2_mul(q2[g][0], k2[u][0]);
            a2 = f2_fma(q2[g][1], k2[u][1], a2);
            a2 = f2_fma(q2[g][2], k2[u][2], a2);
            a2 = f2_fma(q2[g][3], k2[u][3], a2);
            float lo, hi;
            f2_unpack_f(a2, lo, hi);
            sc[u][g] = lo + hi;
          }
#pragma unroll
        for (int off = 1; off < C::LPK; off <<= 1)
#pragma unroll
          for (int u = 0; u < C::U; ++u)
#pragma unroll
            for (int g = 0; g < GW; ++g) sc[u][g] += __shfl_xor_sync(0xffffffffu, sc[u][g], off);
        // the iteration's maximum per query head; rows past the end count as -inf
        float mx[GW];
        bool need_any = false;
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          mx[g] = -INFINITY;
#pragma unroll
          for (int u = 0; u < C::U; ++u) mx[g] = fmaxf(mx[g], valid[u] ? sc[u][g] : -INFINITY);
          need_any |= mx[g] > m[g] + kGqaTau;  // always true on a group's first valid row
        }
        // every lane of a row group holds the same scores, so the decision is uniform per group;
        // one vote per iteration covers all query heads, and the rescale itself is rare
        if (__any_sync(0xffffffffu, need_any)) {
#pragma unroll
          for (int g = 0; g < GW; ++g) {
            if (mx[g] > m[g] + kGqaTau) {
              const float alpha = ex2_approx(m[g] - mx[g]);  // 0 when m was -inf
              const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
              for (int e = 0; e < 4; ++e) o2[g][e] = f2_mul(o2[g][e], a2);
              l[g] *= alpha;
              m[g] = mx[g];
            }
          }
        }
#pragma unroll
        for (int g = 0; g < GW; ++g)
#pragma unroll
          for (int u = 0; u < C::U; ++u) {
            const float p = valid[u] ? ex2_approx(sc[u][g] - m[g]) : 0.f;  // rows past the end take no part
            l[g] += p;
            const uint64_t p2 = f2_pack(p, p);
#pragma unroll
            for (int e = 0; e < 4; ++e) o2[g][e] = f2_fma(p2, v2[u][e], o2[g][e]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
    }
    // merge the KPW row groups of the warp (lanes with equal `sub`), then hand the warp's state over
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) f2_unpack_f(o2[g][e], o[2 * e], o[2 * e + 1]);
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
        const float M = fmaxf(m[g], m2);
        const float wa = (m[g] == -INFINITY) ? 0.f : ex2_approx(m[g] - M);
        const float wb = (m2 == -INFINITY) ? 0.f : ex2_approx(m2 - M);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float o_other = __shfl_xor_sync(0xffffffffu, o[e], off);
          o[e] = o[e] * wa + o_other * wb;
        }
        l[g] = l[g] * wa + l2 * wb;
        m[g] = M;
      }
      const int gq = wset * GW + g;
      if (lane < C::LPK) {
        if (lane == 0) {
          sm_m[wi][gq] = m[g];
          sm_l[wi][gq] = l[g];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) sm_o[wi][gq][sub * 8 + e] = o[e];
      }
    }
  }
  __syncthreads();
  // merge the warps of each set and write one partial state per (query head, chunk)
  for (int i = threadIdx.x; i < G * D; i += C::NTHREADS) {
    const int g = i / D, dim = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::WPS; ++w) M = fmaxf(M, sm_m[w][g]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < C::WPS; ++w) {
      const float wt = (sm_m[w][g] == -INFINITY) ? 0.f : ex2_approx(sm_m[w][g] - M);
      Ls = fmaf(sm_l[w][g], wt, Ls);
      Os = fmaf(sm_o[w][g][dim], wt, Os);
    }
    const size_t st = (static_cast<size_t>(b) * H + h0 + g) * splits + split;
    ws_o[st * D + dim] = Os;
    if (dim == 0) {
      ws_m[st] = M;
      ws_l[st] = Ls;
    }
  }
}

template <class C>
static cudaError_t launch_gqa(const DecodeGqaLaunch& a, float* ws_m, float* ws_l, float* ws_o, int L) {
  cudaError_t e = cudaFuncSetAttribute(fa_decode_gqa_split_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int group = a.H / a.Hkv;
  const int qgroups = group / C::G;
  const long long grid = static_cast<long long>(a.B) * a.Hkv * qgroups * a.splits;
  if (grid <= 0 || grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  fa_decode_gqa_split_kernel<C><<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), ws_m, ws_l, ws_o, a.err, a.Nk, a.splits, L, a.H, a.Hkv, qgroups, a.c);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_gqa_d(const DecodeGqaLaunch& a, float* ws_m, float* ws_l, float* ws_o, int L) {
  const int group = a.H / a.Hkv;
  if (group % 8 == 0) return launch_gqa<DecGqaCfg<D, 8>>(a, ws_m, ws_l, ws_o, L);
  if (group == 4) return launch_gqa<DecGqaCfg<D, 4>>(a, ws_m, ws_l, ws_o, L);
  if (group == 2) return launch_gqa<DecGqaCfg<D, 2>>(a, ws_m, ws_l, ws_o, L);
  if (group == 1) return launch_gqa<DecGqaCfg<D, 1>>(a, ws_m, ws_l, ws_o, L);
  return cudaErrorInvalidValue;
}

int decode_gqa_supported_group(int group) { return group == 1 || group == 2 || group == 4 || group % 8 == 0; }

cudaError_t launch_decode_gqa(const DecodeGqaLaunch& a) {
  if (a.splits < 1 || a.Hkv < 1 || a.H % a.Hkv != 0 || !decode_gqa_supported_group(a.H / a.Hkv))
    return cudaErrorInvalidValue;
  const int L = (a.Nk + a.splits - 1) / a.splits;
  const size_t n_states = static_cast<size_t>(a.B) * a.H * a.splits;
  float* ws_m = a.ws;
  float* ws_l = a.ws + n_states;
  float* ws_o = a.ws + 2 * n_states;
  cudaError_t e;
  if (a.d == 64)
    e = launch_gqa_d<64>(a, ws_m, ws_l, ws_o, L);
  else if (a.d == 128)
    e = launch_gqa_d<128>(a, ws_m, ws_l, ws_o, L);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_decode_merge(ws_m, ws_l, ws_o, a.order, a.o, a.lse, a.B * a.H, a.splits, a.d, a.stream);
}

}  // namespace fa
