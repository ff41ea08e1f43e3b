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
//                            query head sharing the key/value head, 32 at a time, and accumulates
//                            dV and dK of its keys in registers
//   fa_bwd_dq_fp32_kernel    one CTA per (query head, 64 query rows): walks the keys 32 at a time and
//                            accumulates dQ of its rows in registers
// Both main kernels are shared-memory tiled products: each of the 256 threads owns a 4 x 2 block of
// the step's 64 x 32 score tile and a 4 x (D/16) block of the accumulated gradient tile.  Operands
// read along the reduction index are kept transposed in shared memory (one padded row per element
// of the reduction), so that a warp reads consecutive words.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int BW_THREADS = 256;
constexpr int BW_M = 64;  // rows owned by a CTA: keys (dK/dV kernel) or query rows (dQ kernel)
constexpr int BW_N = 32;  // rows streamed per step: query rows (dK/dV) or keys (dQ)
constexpr int PAD_M = BW_M + 1;
constexpr int PAD_N = BW_N + 1;

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

// Shared memory of the dK/dV kernel (floats): K^T, V^T [D][65]; per step Q^T, dO^T [D][33], Q, dO
// [32][D]; P^T and dS^T as [32 query rows][65]; the step's nl and -D.
template <int D>
constexpr int dkdv_smem_floats() {
  return 2 * D * PAD_M + 2 * D * PAD_N + 2 * BW_N * D + 2 * BW_N * PAD_M + 2 * BW_N;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dkdv_fp32_kernel(const BwdF32Params p) {
  extern __shared__ float sm[];
  float* kt = sm;                       // [D][PAD_M]
  float* vt = kt + D * PAD_M;           // [D][PAD_M]
  float* qt = vt + D * PAD_M;           // [D][PAD_N]
  float* dot = qt + D * PAD_N;          // [D][PAD_N]
  float* qr = dot + D * PAD_N;          // [BW_N][D]
  float* dor = qr + BW_N * D;           // [BW_N][D]
  float* ps = dor + BW_N * D;           // [BW_N][PAD_M]: P^T of the step, by query row
  float* dss = ps + BW_N * PAD_M;       // [BW_N][PAD_M]: dS^T of the step
  float* nl_s = dss + BW_N * PAD_M;     // [BW_N]
  float* nd_s = nl_s + BW_N;            // [BW_N]

  const int n_kblk = (p.Nk + BW_M - 1) / BW_M;
  const int kb = static_cast<int>(blockIdx.x % n_kblk);
  const int bhkv = static_cast<int>(blockIdx.x / n_kblk);
  const int b = bhkv / p.Hkv, hkv = bhkv % p.Hkv;
  const int G = p.H / p.Hkv;
  const int k0 = kb * BW_M;
  const int kvalid = min(BW_M, p.Nk - k0);
  const float* kg = p.k + (static_cast<size_t>(bhkv) * p.Nk + k0) * D;
  const float* vg = p.v + (static_cast<size_t>(bhkv) * p.Nk + k0) * D;
  load_transposed<D, BW_M>(kt, PAD_M, kg, kvalid);
  load_transposed<D, BW_M>(vt, PAD_M, vg, kvalid);
  // The prep grid's row values are read below, after its completion.  Once every CTA of this grid has
  // passed that point the dQ grid, which reads the same values and nothing this grid writes, may start
  // on the SMs this grid leaves idle.
  griddep_wait();
  griddep_launch_dependents();

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  // score tile: keys 4 ty .. 4 ty + 3, query rows 2 tx, 2 tx + 1 of the step
  // gradient tile: keys 4 ty .. 4 ty + 3, columns tx * CW .. tx * CW + CW - 1
  constexpr int CW = D / 16;
  float dv_acc[4][CW], dk_acc[4][CW];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < CW; ++c) dv_acc[r][c] = dk_acc[r][c] = 0.f;

  // query rows that see any key of this block: i >= k0 - causal_off under the mask
  const int i_first = p.causal ? max(0, k0 - p.causal_off) : 0;
  const int i_start = i_first / BW_N * BW_N;
  for (int g = 0; g < G; ++g) {
    const size_t bh = static_cast<size_t>(b) * p.H + hkv * G + g;
    for (int i0 = i_start; i0 < p.Nq; i0 += BW_N) {
      const int qvalid = min(BW_N, p.Nq - i0);
      __syncthreads();  // the previous step's tiles are no longer read
      const float* qg = p.q + (bh * p.Nq + i0) * D;
      const float* dg = p.dout + (bh * p.Nq + i0) * D;
      load_transposed<D, BW_N>(qt, PAD_N, qg, qvalid);
      load_transposed<D, BW_N>(dot, PAD_N, dg, qvalid);
      load_rows<D, BW_N>(qr, qg, qvalid);
      load_rows<D, BW_N>(dor, dg, qvalid);
      if (threadIdx.x < BW_N) {
        const size_t rr = bh * p.Nq_pad + i0 + threadIdx.x;  // Nq_pad >= every i0 + BW_N read here
        nl_s[threadIdx.x] = p.nl[rr];
        nd_s[threadIdx.x] = p.negd[rr];
      }
      __syncthreads();
      // S^T = K Q^T and dP^T = V dO^T for this thread's 4 x 2 block
      float s[4][2], dp[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) s[r][0] = s[r][1] = dp[r][0] = dp[r][1] = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) {
        float a[4], av[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          a[r] = kt[c * PAD_M + 4 * ty + r];
          av[r] = vt[c * PAD_M + 4 * ty + r];
        }
        const float b0 = qt[c * PAD_N + 2 * tx], b1 = qt[c * PAD_N + 2 * tx + 1];
        const float g0 = dot[c * PAD_N + 2 * tx], g1 = dot[c * PAD_N + 2 * tx + 1];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          s[r][0] = fmaf(a[r], b0, s[r][0]);
          s[r][1] = fmaf(a[r], b1, s[r][1]);
          dp[r][0] = fmaf(av[r], g0, dp[r][0]);
          dp[r][1] = fmaf(av[r], g1, dp[r][1]);
        }
      }
      // P^T and dS^T; masked pairs (key past Nk or past the row's causal limit, row past Nq) give 0
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int il = 2 * tx + qq, i = i0 + il;
        const float nli = nl_s[il], ndi = nd_s[il];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int kl = 4 * ty + r, kj = k0 + kl;
          const bool vis = kj < p.Nk && i < p.Nq && (!p.causal || kj <= i + p.causal_off);
          const float pr = vis ? ex2_approx(fmaf(s[r][qq], p.c, nli)) : 0.f;
          ps[il * PAD_M + kl] = pr;
          dss[il * PAD_M + kl] = pr * (dp[r][qq] + ndi);
        }
      }
      __syncthreads();
      // dV += P^T dO, dK += dS^T Q over the step's query rows
#pragma unroll 4
      for (int il = 0; il < BW_N; ++il) {
        float pr[4], dr[4], go[CW], qv[CW];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          pr[r] = ps[il * PAD_M + 4 * ty + r];
          dr[r] = dss[il * PAD_M + 4 * ty + r];
        }
#pragma unroll
        for (int c = 0; c < CW; ++c) {
          go[c] = dor[il * D + tx * CW + c];
          qv[c] = qr[il * D + tx * CW + c];
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
    for (int c = 0; c < CW; ++c) {
      p.dv[off + c] = dv_acc[r][c];
      p.dk[off + c] = dk_acc[r][c] * p.scale;
    }
  }
}

// Shared memory of the dQ kernel (floats): Q^T, dO^T [D][65]; per step K^T, V^T [D][33], K [32][D];
// dS as [32 keys][65]; the CTA's nl and -D.
template <int D>
constexpr int dq_smem_floats() {
  return 2 * D * PAD_M + 2 * D * PAD_N + BW_N * D + BW_N * PAD_M + 2 * BW_M;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dq_fp32_kernel(const BwdF32Params p) {
  extern __shared__ float sm[];
  float* qt = sm;                       // [D][PAD_M]
  float* dot = qt + D * PAD_M;          // [D][PAD_M]
  float* kt = dot + D * PAD_M;          // [D][PAD_N]
  float* vt = kt + D * PAD_N;           // [D][PAD_N]
  float* kr = vt + D * PAD_N;           // [BW_N][D]
  float* dss = kr + BW_N * D;           // [BW_N keys][PAD_M]
  float* nl_s = dss + BW_N * PAD_M;     // [BW_M]
  float* nd_s = nl_s + BW_M;            // [BW_M]

  const int n_qblk = (p.Nq + BW_M - 1) / BW_M;
  const int qb = static_cast<int>(blockIdx.x % n_qblk);
  const int bh = static_cast<int>(blockIdx.x / n_qblk);
  const int b = bh / p.H, h = bh % p.H;
  const int bhkv = b * p.Hkv + h / (p.H / p.Hkv);
  const int i0 = qb * BW_M;
  const int qvalid = min(BW_M, p.Nq - i0);
  const float* qg = p.q + (static_cast<size_t>(bh) * p.Nq + i0) * D;
  const float* dg = p.dout + (static_cast<size_t>(bh) * p.Nq + i0) * D;
  load_transposed<D, BW_M>(qt, PAD_M, qg, qvalid);
  load_transposed<D, BW_M>(dot, PAD_M, dg, qvalid);
  if (threadIdx.x < BW_M) {
    const size_t rr = static_cast<size_t>(bh) * p.Nq_pad + i0 + threadIdx.x;  // Nq_pad >= i0 + BW_M
    nl_s[threadIdx.x] = p.nl[rr];
    nd_s[threadIdx.x] = p.negd[rr];
  }

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  // score tile: query rows 4 ty .. 4 ty + 3, keys 2 tx, 2 tx + 1 of the step
  // gradient tile: query rows 4 ty .. 4 ty + 3, columns tx * CW .. tx * CW + CW - 1
  constexpr int CW = D / 16;
  float dq_acc[4][CW];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < CW; ++c) dq_acc[r][c] = 0.f;

  // keys any row of this block sees: j <= i0 + BW_M - 1 + causal_off under the mask
  const int k_end = p.causal ? min(p.Nk, i0 + BW_M + p.causal_off) : p.Nk;
  for (int j0 = 0; j0 < k_end; j0 += BW_N) {
    const int kvalid = min(BW_N, p.Nk - j0);
    __syncthreads();  // the previous step's tiles are no longer read (and the CTA's tiles are in)
    const float* kg = p.k + (static_cast<size_t>(bhkv) * p.Nk + j0) * D;
    const float* vg = p.v + (static_cast<size_t>(bhkv) * p.Nk + j0) * D;
    load_transposed<D, BW_N>(kt, PAD_N, kg, kvalid);
    load_transposed<D, BW_N>(vt, PAD_N, vg, kvalid);
    load_rows<D, BW_N>(kr, kg, kvalid);
    __syncthreads();
    // S = Q K^T and dP = dO V^T for this thread's 4 x 2 block
    float s[4][2], dp[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) s[r][0] = s[r][1] = dp[r][0] = dp[r][1] = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; ++c) {
      float a[4], ag[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = qt[c * PAD_M + 4 * ty + r];
        ag[r] = dot[c * PAD_M + 4 * ty + r];
      }
      const float b0 = kt[c * PAD_N + 2 * tx], b1 = kt[c * PAD_N + 2 * tx + 1];
      const float v0 = vt[c * PAD_N + 2 * tx], v1 = vt[c * PAD_N + 2 * tx + 1];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        s[r][0] = fmaf(a[r], b0, s[r][0]);
        s[r][1] = fmaf(a[r], b1, s[r][1]);
        dp[r][0] = fmaf(ag[r], v0, dp[r][0]);
        dp[r][1] = fmaf(ag[r], v1, dp[r][1]);
      }
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int jl = 2 * tx + kk, j = j0 + jl;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int il = 4 * ty + r, i = i0 + il;
        const bool vis = j < p.Nk && i < p.Nq && (!p.causal || j <= i + p.causal_off);
        const float pr = vis ? ex2_approx(fmaf(s[r][kk], p.c, nl_s[il])) : 0.f;
        dss[jl * PAD_M + il] = pr * (dp[r][kk] + nd_s[il]);
      }
    }
    __syncthreads();
    // dQ += dS K over the step's keys
#pragma unroll 4
    for (int jl = 0; jl < BW_N; ++jl) {
      float dr[4], kv[CW];
#pragma unroll
      for (int r = 0; r < 4; ++r) dr[r] = dss[jl * PAD_M + 4 * ty + r];
#pragma unroll
      for (int c = 0; c < CW; ++c) kv[c] = kr[jl * D + tx * CW + c];
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
    for (int c = 0; c < CW; ++c) p.dq[off + c] = dq_acc[r][c] * p.scale;
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
      static_cast<const float*>(a.o), static_cast<const float*>(a.dout), a.lse, const_cast<float*>(p.nl),
      const_cast<float*>(p.negd), rows, a.Nq, a.Nq_pad);
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
