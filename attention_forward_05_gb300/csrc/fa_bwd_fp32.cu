// fa_bwd_fp32.cu -- attention backward for fp32 tensors, in fp32 arithmetic on the CUDA cores.
//
// Sources (web pages, cited by title and section):
//   [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io), Exercise 5: the backward
//        rebuilds P_ij = exp(S_ij - m_i) / l_i block by block from the forward's row statistics and
//        accumulates dV_j += P_ij^T dO_i.  The exercise is written for fp32 tensors.
//   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com), demo 3 remarks: one statistic per
//        row, the logsumexp L = m + ln l, is enough: P_ij = exp(S_ij - L_i).
// The other gradients follow from the chain rule through the row softmax:
//   dP = dO V^T,  dS = P * (dP - D) with D_i = sum_c dO_ic O_ic,  dQ = scale dS K,  dK = scale dS^T Q.
//
// The tensor cores multiply fp32 data only as tf32 (10-bit mantissa), and their tf32 form takes
// K-major operands only, which three of the backward's five products do not have.  These kernels
// keep every product in fp32 FMAs instead: the gradients carry fp32 rounding, not tf32 rounding.
// Three launches, no atomics (every gradient element is written by one thread of one CTA):
//   fa_bwd_prep_fp32_kernel  nl_i = -L_i log2(e) and D_i for every query row (padded rows: -inf, 0)
//   fa_bwd_dkdv_fp32_kernel  one CTA per (key/value head, 64 keys): walks the query rows of every
//                            query head sharing the key/value head, 64 (d = 64) or 32 (d = 128) at a
//                            time, and accumulates dV and dK of its keys in registers
//   fa_bwd_dq_fp32_kernel    one CTA per (query head, 64 query rows): walks the keys 64 or 32 at a time
//                            and accumulates dQ of its rows in registers
// Both main kernels are shared-memory tiled products: each of the 256 threads owns a 4 x 4 (d = 64)
// or 4 x 2 (d = 128) block of the step's score tile and a 4 x (d/16) block of the accumulated
// gradient tile.  Operands read along the reduction index are kept transposed in shared memory, with
// rows padded to whole 16-byte groups, so that each thread reads its operands as vectors.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int BW_THREADS = 256;
constexpr int BW_M = 64;  // rows owned by a CTA: keys (dK/dV kernel) or query rows (dQ kernel)

// Row values for the fp32 backward: nl[r] = -L_r log2(e), negd[r] = -D_r over [BH][Nq_pad].
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_fp32_kernel(const float* __restrict__ o,
                                                               const float* __restrict__ dout,
                                                               const float* __restrict__ lse, float* __restrict__ nl,
                                                               float* __restrict__ negd, long long rows_pad, int Nq,
                                                               int Nq_pad) {
  griddep_launch_dependents();  // the dK/dV kernel may start its set-up; it waits for this grid's rows
  constexpr int LPR = D / 4;  // lanes per row, one float4 each (a row is D / 4 lanes of one warp)
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = gt / LPR;
  const int part = static_cast<int>(gt % LPR);
  const bool live = r < rows_pad;
  const long long bh = live ? r / Nq_pad : 0;
  const int i = live ? static_cast<int>(r % Nq_pad) : 0;
  const bool in_range = live && i < Nq;
  float acc = 0.f;
  if (in_range) {
    const size_t off = (static_cast<size_t>(bh) * Nq + i) * D + part * 4;
    const float4 a = *reinterpret_cast<const float4*>(o + off);
    const float4 g = *reinterpret_cast<const float4*>(dout + off);
    acc = a.x * g.x + a.y * g.y + a.z * g.z + a.w * g.w;
  }
  // a row's LPR lanes are consecutive lanes of one warp (LPR = 16 or 32 divides 32)
#pragma unroll
  for (int m = LPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (live && part == 0) {
    nl[r] = in_range ? -lse[static_cast<size_t>(bh) * Nq + i] * 1.4426950408889634f : -INFINITY;
    negd[r] = in_range ? -acc : 0.f;
  }
}

// dst[c][r] = src[r][c] for the NROWS rows of a [*, D] fp32 block (rows >= valid read as zero); dst
// has `ld` words per c.  Each thread loads all its elements before storing any, so the block's global
// loads are in flight together.
template <int D, int NROWS>
__device__ __forceinline__ void load_transposed(float* dst, int ld, const float* src, int valid) {
  constexpr int PER = NROWS * D / BW_THREADS;
  static_assert(PER * BW_THREADS == NROWS * D, "whole rounds");
  float x[PER];
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int idx = it * BW_THREADS + static_cast<int>(threadIdx.x);
    const int r = idx / D, c = idx % D;
    x[it] = r < valid ? src[static_cast<size_t>(r) * D + c] : 0.f;
  }
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int idx = it * BW_THREADS + static_cast<int>(threadIdx.x);
    dst[(idx % D) * ld + idx / D] = x[it];
  }
}

// dst[r][c] = src[r][c] (row-major, D words per row) for the NROWS rows (rows >= valid read as zero).
template <int D, int NROWS>
__device__ __forceinline__ void load_rows(float* dst, const float* src, int valid) {
  constexpr int PER = NROWS * D / 4 / BW_THREADS;
  static_assert(PER * BW_THREADS * 4 == NROWS * D, "whole rounds");
  float4 x[PER];
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int idx = it * BW_THREADS + static_cast<int>(threadIdx.x);
    const int r = idx / (D / 4), c4 = idx % (D / 4);
    x[it] = r < valid ? reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * D)[c4]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int idx = it * BW_THREADS + static_cast<int>(threadIdx.x);
    reinterpret_cast<float4*>(dst + (idx / (D / 4)) * D)[idx % (D / 4)] = x[it];
  }
}

struct BwdF32Params {
  const float *q, *k, *v, *dout, *nl, *negd;
  float *dq, *dk, *dv;
  int Nq, Nk, Nq_pad, H, Hkv, causal, causal_off;
  float c, scale;
};

// Tile shapes.  A CTA owns BM = 64 rows (keys in the dK/dV kernel, query rows in the dQ kernel) and
// streams BN rows of the other side per step: 64 at d = 64, 32 at d = 128 (shared memory).  Thread
// (ty, tx) of 16 x 16 owns rows 4 ty .. 4 ty + 3 of the CTA's side, and in the step's score tile the
// TQ = BN / 16 columns TQ tx ..; in the accumulated gradient tile the CW = d / 16 columns CW tx ...
// Arrays read along the reduction index are transposed, with rows padded to a multiple of 4 floats
// so that every read is one 16-byte (or 8-byte) load.
template <int D>
struct F32Tile {
  static constexpr int BM = BW_M;
  static constexpr int BN = D == 64 ? 64 : 32;
  static constexpr int TQ = BN / 16;
  static constexpr int CW = D / 16;
  static constexpr int MP = BM + 4;  // padded row of a transposed BM-row block
  static constexpr int NP = BN + 4;  // padded row of a transposed BN-row block
};

template <int N>
__device__ __forceinline__ void lds_vec(float (&r)[N], const float* p) {
  static_assert(N == 2 || N == 4, "vector width");
  if constexpr (N == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    r[0] = x.x;
    r[1] = x.y;
    r[2] = x.z;
    r[3] = x.w;
  } else {
    const float2 x = *reinterpret_cast<const float2*>(p);
    r[0] = x.x;
    r[1] = x.y;
  }
}

// Shared memory of the dK/dV kernel (floats): K^T, V^T [D][MP]; per step Q^T, dO^T [D][NP], Q, dO
// [BN][D]; P^T and dS^T as [BN query rows][MP]; the step's nl and -D.
template <int D>
constexpr int dkdv_smem_floats() {
  using T = F32Tile<D>;
  return 2 * D * T::MP + 2 * D * T::NP + 2 * T::BN * D + 2 * T::BN * T::MP + 2 * T::BN;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dkdv_fp32_kernel(const BwdF32Params p) {
  using T = F32Tile<D>;
  constexpr int BM = T::BM, BN = T::BN, TQ = T::TQ, CW = T::CW, MP = T::MP, NP = T::NP;
  extern __shared__ __align__(16) float sm[];
  float* kt = sm;                       // [D][MP]
  float* vt = kt + D * MP;              // [D][MP]
  float* qt = vt + D * MP;              // [D][NP]
  float* dot = qt + D * NP;             // [D][NP]
  float* qr = dot + D * NP;             // [BN][D]
  float* dor = qr + BN * D;             // [BN][D]
  float* ps = dor + BN * D;             // [BN][MP]: P^T of the step, by query row
  float* dss = ps + BN * MP;            // [BN][MP]: dS^T of the step
  float* nl_s = dss + BN * MP;          // [BN]
  float* nd_s = nl_s + BN;              // [BN]

  const int n_kblk = (p.Nk + BM - 1) / BM;
  const int kb = static_cast<int>(blockIdx.x % n_kblk);
  const int bhkv = static_cast<int>(blockIdx.x / n_kblk);
  const int b = bhkv / p.Hkv, hkv = bhkv % p.Hkv;
  const int G = p.H / p.Hkv;
  const int k0 = kb * BM;
  const int kvalid = min(BM, p.Nk - k0);
  const float* kg = p.k + (static_cast<size_t>(bhkv) * p.Nk + k0) * D;
  const float* vg = p.v + (static_cast<size_t>(bhkv) * p.Nk + k0) * D;
  load_transposed<D, BM>(kt, MP, kg, kvalid);
  load_transposed<D, BM>(vt, MP, vg, kvalid);
  // The prep grid's row values are read below, after its completion.  Once every CTA of this grid has
  // passed that point the dQ grid, which reads the same values and nothing this grid writes, may start
  // on the SMs this grid leaves idle.
  griddep_wait();
  griddep_launch_dependents();

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float dv_acc[4][CW], dk_acc[4][CW];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < CW; ++c) dv_acc[r][c] = dk_acc[r][c] = 0.f;

  // query rows that see any key of this block: i >= k0 - causal_off under the mask
  const int i_first = p.causal ? max(0, k0 - p.causal_off) : 0;
  const int i_start = i_first / BN * BN;
  for (int g = 0; g < G; ++g) {
    const size_t bh = static_cast<size_t>(b) * p.H + hkv * G + g;
    for (int i0 = i_start; i0 < p.Nq; i0 += BN) {
      const int qvalid = min(BN, p.Nq - i0);
      __syncthreads();  // the previous step's tiles are no longer read
      const float* qg = p.q + (bh * p.Nq + i0) * D;
      const float* dg = p.dout + (bh * p.Nq + i0) * D;
      load_transposed<D, BN>(qt, NP, qg, qvalid);
      load_transposed<D, BN>(dot, NP, dg, qvalid);
      load_rows<D, BN>(qr, qg, qvalid);
      load_rows<D, BN>(dor, dg, qvalid);
      if (threadIdx.x < BN) {
        const size_t rr = bh * p.Nq_pad + i0 + threadIdx.x;  // Nq_pad >= every i0 + BN read here
        nl_s[threadIdx.x] = p.nl[rr];
        nd_s[threadIdx.x] = p.negd[rr];
      }
      __syncthreads();
      // S^T = K Q^T and dP^T = V dO^T for this thread's 4 x TQ block
      float s[4][TQ], dp[4][TQ];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int qq = 0; qq < TQ; ++qq) s[r][qq] = dp[r][qq] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float a[4], av[4], bq[TQ], bg[TQ];
        lds_vec(a, kt + c * MP + 4 * ty);
        lds_vec(av, vt + c * MP + 4 * ty);
        lds_vec(bq, qt + c * NP + TQ * tx);
        lds_vec(bg, dot + c * NP + TQ * tx);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int qq = 0; qq < TQ; ++qq) {
            s[r][qq] = fmaf(a[r], bq[qq], s[r][qq]);
            dp[r][qq] = fmaf(av[r], bg[qq], dp[r][qq]);
          }
      }
      // P^T and dS^T; masked pairs (key past Nk or past the row's causal limit, row past Nq) give 0
#pragma unroll
      for (int qq = 0; qq < TQ; ++qq) {
        const int il = TQ * tx + qq, i = i0 + il;
        const float nli = nl_s[il], ndi = nd_s[il];
        float pr[4], dsr[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int kj = k0 + 4 * ty + r;
          const bool vis = kj < p.Nk && i < p.Nq && (!p.causal || kj <= i + p.causal_off);
          pr[r] = vis ? ex2_approx(fmaf(s[r][qq], p.c, nli)) : 0.f;
          dsr[r] = pr[r] * (dp[r][qq] + ndi);
        }
        *reinterpret_cast<float4*>(ps + il * MP + 4 * ty) = make_float4(pr[0], pr[1], pr[2], pr[3]);
        *reinterpret_cast<float4*>(dss + il * MP + 4 * ty) = make_float4(dsr[0], dsr[1], dsr[2], dsr[3]);
      }
      __syncthreads();
      // dV += P^T dO, dK += dS^T Q over the step's query rows
#pragma unroll 4
      for (int il = 0; il < BN; ++il) {
        float pr[4], dr[4], go[CW], qv[CW];
        lds_vec(pr, ps + il * MP + 4 * ty);
        lds_vec(dr, dss + il * MP + 4 * ty);
#pragma unroll
        for (int c4 = 0; c4 < CW; c4 += 4) {
          float t0[4], t1[4];
          lds_vec(t0, dor + il * D + tx * CW + c4);
          lds_vec(t1, qr + il * D + tx * CW + c4);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            go[c4 + e] = t0[e];
            qv[c4 + e] = t1[e];
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < CW; ++c) {
            dv_acc[r][c] = fmaf(pr[r], go[c], dv_acc[r][c]);
            dk_acc[r][c] = fmaf(dr[r], qv[c], dk_acc[r][c]);
          }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int kl = 4 * ty + r;
    if (kl >= kvalid) continue;
    const size_t off = (static_cast<size_t>(bhkv) * p.Nk + k0 + kl) * D + tx * CW;
#pragma unroll
    for (int c4 = 0; c4 < CW; c4 += 4) {
      *reinterpret_cast<float4*>(p.dv + off + c4) =
          make_float4(dv_acc[r][c4], dv_acc[r][c4 + 1], dv_acc[r][c4 + 2], dv_acc[r][c4 + 3]);
      *reinterpret_cast<float4*>(p.dk + off + c4) =
          make_float4(dk_acc[r][c4] * p.scale, dk_acc[r][c4 + 1] * p.scale, dk_acc[r][c4 + 2] * p.scale,
                      dk_acc[r][c4 + 3] * p.scale);
    }
  }
}

// Shared memory of the dQ kernel (floats): Q^T, dO^T [D][MP]; per step K^T, V^T [D][NP], K [BN][D];
// dS as [BN keys][MP]; the CTA's nl and -D.
template <int D>
constexpr int dq_smem_floats() {
  using T = F32Tile<D>;
  return 2 * D * T::MP + 2 * D * T::NP + T::BN * D + T::BN * T::MP + 2 * T::BM;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dq_fp32_kernel(const BwdF32Params p) {
  using T = F32Tile<D>;
  constexpr int BM = T::BM, BN = T::BN, TQ = T::TQ, CW = T::CW, MP = T::MP, NP = T::NP;
  extern __shared__ __align__(16) float sm[];
  float* qt = sm;                       // [D][MP]
  float* dot = qt + D * MP;             // [D][MP]
  float* kt = dot + D * MP;             // [D][NP]
  float* vt = kt + D * NP;              // [D][NP]
  float* kr = vt + D * NP;              // [BN][D]
  float* dss = kr + BN * D;             // [BN keys][MP]
  float* nl_s = dss + BN * MP;          // [BM]
  float* nd_s = nl_s + BM;              // [BM]

  const int n_qblk = (p.Nq + BM - 1) / BM;
  const int qb = static_cast<int>(blockIdx.x % n_qblk);
  const int bh = static_cast<int>(blockIdx.x / n_qblk);
  const int b = bh / p.H, h = bh % p.H;
  const int bhkv = b * p.Hkv + h / (p.H / p.Hkv);
  const int i0 = qb * BM;
  const int qvalid = min(BM, p.Nq - i0);
  const float* qg = p.q + (static_cast<size_t>(bh) * p.Nq + i0) * D;
  const float* dg = p.dout + (static_cast<size_t>(bh) * p.Nq + i0) * D;
  load_transposed<D, BM>(qt, MP, qg, qvalid);
  load_transposed<D, BM>(dot, MP, dg, qvalid);
  if (threadIdx.x < BM) {
    const size_t rr = static_cast<size_t>(bh) * p.Nq_pad + i0 + threadIdx.x;  // Nq_pad >= i0 + BM
    nl_s[threadIdx.x] = p.nl[rr];
    nd_s[threadIdx.x] = p.negd[rr];
  }

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float dq_acc[4][CW];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < CW; ++c) dq_acc[r][c] = 0.f;

  // keys any row of this block sees: j <= i0 + BM - 1 + causal_off under the mask
  const int k_end = p.causal ? min(p.Nk, i0 + BM + p.causal_off) : p.Nk;
  for (int j0 = 0; j0 < k_end; j0 += BN) {
    const int kvalid = min(BN, p.Nk - j0);
    __syncthreads();  // the previous step's tiles are no longer read (and the CTA's tiles are in)
    const float* kg = p.k + (static_cast<size_t>(bhkv) * p.Nk + j0) * D;
    const float* vg = p.v + (static_cast<size_t>(bhkv) * p.Nk + j0) * D;
    load_transposed<D, BN>(kt, NP, kg, kvalid);
    load_transposed<D, BN>(vt, NP, vg, kvalid);
    load_rows<D, BN>(kr, kg, kvalid);
    __syncthreads();
    // S = Q K^T and dP = dO V^T for this thread's 4 x TQ block
    float s[4][TQ], dp[4][TQ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int kk = 0; kk < TQ; ++kk) s[r][kk] = dp[r][kk] = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; ++c) {
      float a[4], ag[4], bk[TQ], bv[TQ];
      lds_vec(a, qt + c * MP + 4 * ty);
      lds_vec(ag, dot + c * MP + 4 * ty);
      lds_vec(bk, kt + c * NP + TQ * tx);
      lds_vec(bv, vt + c * NP + TQ * tx);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int kk = 0; kk < TQ; ++kk) {
          s[r][kk] = fmaf(a[r], bk[kk], s[r][kk]);
          dp[r][kk] = fmaf(ag[r], bv[kk], dp[r][kk]);
        }
    }
#pragma unroll
    for (int kk = 0; kk < TQ; ++kk) {
      const int jl = TQ * tx + kk, j = j0 + jl;
      float dsr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int il = 4 * ty + r, i = i0 + il;
        const bool vis = j < p.Nk && i < p.Nq && (!p.causal || j <= i + p.causal_off);
        const float pr = vis ? ex2_approx(fmaf(s[r][kk], p.c, nl_s[il])) : 0.f;
        dsr[r] = pr * (dp[r][kk] + nd_s[il]);
      }
      *reinterpret_cast<float4*>(dss + jl * MP + 4 * ty) = make_float4(dsr[0], dsr[1], dsr[2], dsr[3]);
    }
    __syncthreads();
    // dQ += dS K over the step's keys
#pragma unroll 4
    for (int jl = 0; jl < BN; ++jl) {
      float dr[4], kv[CW];
      lds_vec(dr, dss + jl * MP + 4 * ty);
#pragma unroll
      for (int c4 = 0; c4 < CW; c4 += 4) {
        float t0[4];
        lds_vec(t0, kr + jl * D + tx * CW + c4);
#pragma unroll
        for (int e = 0; e < 4; ++e) kv[c4 + e] = t0[e];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < CW; ++c) dq_acc[r][c] = fmaf(dr[r], kv[c], dq_acc[r][c]);
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int il = 4 * ty + r;
    if (il >= qvalid) continue;
    const size_t off = (static_cast<size_t>(bh) * p.Nq + i0 + il) * D + tx * CW;
#pragma unroll
    for (int c4 = 0; c4 < CW; c4 += 4)
      *reinterpret_cast<float4*>(p.dq + off + c4) =
          make_float4(dq_acc[r][c4] * p.scale, dq_acc[r][c4 + 1] * p.scale, dq_acc[r][c4 + 2] * p.scale,
                      dq_acc[r][c4 + 3] * p.scale);
  }
  // This grid may have started before the dK/dV grid finished; waiting for it here keeps every gradient
  // complete once this grid is, for the work that follows the backward on the stream.
  griddep_wait();
}

template <int D>
cudaError_t launch_bwd_fp32_d(const BwdLaunch& a, const BwdF32Params& p) {
  const long long rows = static_cast<long long>(a.BH) * a.Nq_pad;
  const long long blocks = (rows * (D / 4) + 255) / 256;
  if (blocks <= 0 || blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  fa_bwd_prep_fp32_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
      static_cast<const float*>(a.o), static_cast<const float*>(a.dout), a.lse, a.rowv, a.rowv2, rows, a.Nq,
      a.Nq_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int smem_kv = dkdv_smem_floats<D>() * 4;
  constexpr int smem_q = dq_smem_floats<D>() * 4;
  static_assert(smem_kv <= 227 * 1024 && smem_q <= 227 * 1024, "shared memory");
  if ((e = cudaFuncSetAttribute(fa_bwd_dkdv_fp32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(fa_bwd_dq_fp32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q)) !=
          cudaSuccess)
    return e;
  const long long grid_kv = static_cast<long long>((a.Nk + BW_M - 1) / BW_M) * a.BHkv;
  const long long grid_q = static_cast<long long>((a.Nq + BW_M - 1) / BW_M) * a.BH;
  if (grid_kv <= 0 || grid_kv > 0x7FFFFFFFLL || grid_q <= 0 || grid_q > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  // prep -> dK/dV -> dQ as programmatic dependents (see the kernels for what each waits for)
  if ((e = launch_dependent(fa_bwd_dkdv_fp32_kernel<D>, static_cast<unsigned>(grid_kv), BW_THREADS, smem_kv,
                            a.stream, p)) != cudaSuccess)
    return e;
  return launch_dependent(fa_bwd_dq_fp32_kernel<D>, static_cast<unsigned>(grid_q), BW_THREADS, smem_q, a.stream, p);
}

}  // namespace

int bwd_fp32_nq_align() { return BW_M; }

cudaError_t launch_bwd_fp32(const BwdLaunch& a) {
  if (a.causal && a.Nq > a.Nk) return cudaErrorInvalidValue;
  if (a.Nq_pad % BW_M != 0 || a.Nq_pad < a.Nq) return cudaErrorInvalidValue;  // whole row blocks are read
  BwdF32Params p;
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.dout = static_cast<const float*>(a.dout);
  p.nl = a.rowv;
  p.negd = a.rowv2;
  p.dq = static_cast<float*>(a.dq);
  p.dk = static_cast<float*>(a.dk);
  p.dv = static_cast<float*>(a.dv);
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.Nq_pad = a.Nq_pad;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.causal = a.causal;
  p.causal_off = a.Nk - a.Nq;
  p.c = a.c;
  p.scale = a.scale;
  return a.d == 64 ? launch_bwd_fp32_d<64>(a, p) : launch_bwd_fp32_d<128>(a, p);
}

}  // namespace fa
