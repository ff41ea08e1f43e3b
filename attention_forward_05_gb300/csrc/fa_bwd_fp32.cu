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
// gradient tile.  Every operand stays row-major in shared memory (rows padded by 16 bytes, so the
// 16-byte reads of a quarter-warp hit distinct banks), and the next step's tiles stream in with
// asynchronous copies while the current step computes.
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

struct BwdF32Params {
  const float *q, *k, *v, *dout, *nl, *negd;
  float *dq, *dk, *dv;
  int Nq, Nk, Nq_pad, H, Hkv, causal, causal_off;
  float c, scale;
};

// Tile shapes.  A CTA owns BM = 64 rows (keys in the dK/dV kernel, query rows in the dQ kernel) and
// streams BN rows of the other side per step: 64 at d = 64, 32 at d = 128 (shared memory).  Thread
// (ty, tx) of 16 x 16 owns the CTA-side rows ty + 16 r (r < 4), the step-side rows tx + 16 q (q < TQ)
// of the step's score tile, and the gradient columns 64 h + 4 tx .. + 3 (h < d / 64).  Every operand
// sits row-major in shared memory with rows padded to D + 4 floats, so that the 16-byte reads of a
// quarter-warp (eight consecutive step-side rows, or one row's consecutive columns) hit distinct
// banks, and a CTA-side read is a broadcast.  P^T / dS (written by the score phase, read by the
// gradient phase) are stored by step-side row with the thread's four CTA-side rows adjacent: column
// 4 ty + r holds CTA row ty + 16 r.
template <int D>
struct F32Tile {
  static constexpr int BM = BW_M;
  static constexpr int BN = D == 64 ? 64 : 32;
  static constexpr int TQ = BN / 16;
  static constexpr int NH = D / 64;        // 4-column groups of gradient columns per thread
  static constexpr int LD = D + 4;         // padded row of a [rows][D] tile
  static constexpr int MP = BM + 4;        // padded row of a [step rows][BM] tile
};

template <int N>
__device__ __forceinline__ void lds_vec(float (&r)[N], const float* p) {
  static_assert(N == 4, "vector width");
  const float4 x = *reinterpret_cast<const float4*>(p);
  r[0] = x.x;
  r[1] = x.y;
  r[2] = x.z;
  r[3] = x.w;
}

// 16-byte asynchronous copy global -> shared; `ok` false writes zeros (the source is not read).
__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// dst[r][c] = src[r][c] for the NROWS rows of a [*, D] fp32 block into rows of LD floats (rows >= valid
// are zero), as 16-byte asynchronous copies spread over the CTA's threads.  src is row 0 of the block,
// always a valid row.
template <int D, int NROWS>
__device__ __forceinline__ void copy_rows_async(float* dst, const float* src, int valid) {
  constexpr int G = D / 4;
  constexpr int PER = NROWS * G / BW_THREADS;
  static_assert(PER * BW_THREADS == NROWS * G, "whole rounds");
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int idx = it * BW_THREADS + static_cast<int>(threadIdx.x);
    const int r = idx / G, g = idx % G;
    const bool ok = r < valid;
    cp_async16(dst + r * (D + 4) + 4 * g, src + static_cast<size_t>(ok ? r : 0) * D + 4 * g, ok);
  }
}

// n floats (a multiple of 4, 16-byte aligned on both sides) by threads 0 .. n/4 - 1.
__device__ __forceinline__ void copy_vec_async(float* dst, const float* src, int n) {
  const int g = static_cast<int>(threadIdx.x);
  if (g < n / 4) cp_async16(dst + 4 * g, src + 4 * g, true);
}

// Shared memory of the dK/dV kernel (floats): K, V [BM][LD]; two stages of Q, dO [BN][LD] and the step's
// nl, -D [BN]; P^T and dS^T as [BN][MP].
template <int D>
constexpr int dkdv_smem_floats() {
  using T = F32Tile<D>;
  return 2 * T::BM * T::LD + 2 * (2 * T::BN * T::LD + 2 * T::BN) + 2 * T::BN * T::MP;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dkdv_fp32_kernel(const BwdF32Params p) {
  using T = F32Tile<D>;
  constexpr int BM = T::BM, BN = T::BN, TQ = T::TQ, NH = T::NH, LD = T::LD, MP = T::MP;
  constexpr int STAGE = 2 * BN * LD + 2 * BN;
  extern __shared__ __align__(16) float sm[];
  float* ks = sm;                       // [BM][LD]
  float* vs = ks + BM * LD;             // [BM][LD]
  float* st0 = vs + BM * LD;            // stage s at st0 + s * STAGE: Q [BN][LD], dO [BN][LD], nl [BN], -D [BN]
  float* ps = st0 + 2 * STAGE;          // [BN][MP]: P^T of the step, by query row
  float* dss = ps + BN * MP;            // [BN][MP]: dS^T of the step

  const int n_kblk = (p.Nk + BM - 1) / BM;
  const int kb = static_cast<int>(blockIdx.x % n_kblk);
  const int bhkv = static_cast<int>(blockIdx.x / n_kblk);
  const int b = bhkv / p.Hkv, hkv = bhkv % p.Hkv;
  const int G = p.H / p.Hkv;
  const int k0 = kb * BM;
  const int kvalid = min(BM, p.Nk - k0);
  copy_rows_async<D, BM>(ks, p.k + (static_cast<size_t>(bhkv) * p.Nk + k0) * D, kvalid);
  copy_rows_async<D, BM>(vs, p.v + (static_cast<size_t>(bhkv) * p.Nk + k0) * D, kvalid);
  cp_async_commit();
  // The prep grid's row values are read below, after its completion.  Once every CTA of this grid has
  // passed that point the dQ grid, which reads the same values and nothing this grid writes, may start
  // on the SMs this grid leaves idle.
  griddep_wait();
  griddep_launch_dependents();

  // steps: (query head g of the group, query tile i0), query tiles that see any key of this block
  const int i_first = p.causal ? max(0, k0 - p.causal_off) : 0;
  const int i_start = i_first / BN * BN;
  const int n_i = (p.Nq - i_start + BN - 1) / BN;
  const int n_steps = G * n_i;
  auto step_bh = [&](int t) { return static_cast<size_t>(b) * p.H + hkv * G + t / n_i; };
  auto step_i0 = [&](int t) { return i_start + (t % n_i) * BN; };
  auto issue_step = [&](int t) {
    float* st = st0 + (t & 1) * STAGE;
    const size_t bh = step_bh(t);
    const int i0 = step_i0(t);
    const int qvalid = min(BN, p.Nq - i0);
    copy_rows_async<D, BN>(st, p.q + (bh * p.Nq + i0) * D, qvalid);
    copy_rows_async<D, BN>(st + BN * LD, p.dout + (bh * p.Nq + i0) * D, qvalid);
    copy_vec_async(st + 2 * BN * LD, p.nl + bh * p.Nq_pad + i0, BN);  // Nq_pad >= every i0 + BN read here
    copy_vec_async(st + 2 * BN * LD + BN, p.negd + bh * p.Nq_pad + i0, BN);
    cp_async_commit();
  };
  issue_step(0);

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float dv_acc[4][4 * NH], dk_acc[4][4 * NH];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4 * NH; ++c) dv_acc[r][c] = dk_acc[r][c] = 0.f;

  for (int t = 0; t < n_steps; ++t) {
    if (t + 1 < n_steps) {
      issue_step(t + 1);  // into the other stage, released at the end of step t - 1
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // every thread's copies of step t (and of K, V) are in
    const float* qs = st0 + (t & 1) * STAGE;
    const float* dos = qs + BN * LD;
    const float* nl_s = dos + BN * LD;
    const float* nd_s = nl_s + BN;
    const int i0 = step_i0(t);
    // S^T = K Q^T and dP^T = V dO^T for this thread's 4 x TQ block, summed over c in order
    float s[4][TQ], dp[4][TQ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int qq = 0; qq < TQ; ++qq) s[r][qq] = dp[r][qq] = 0.f;
#pragma unroll 2
    for (int c = 0; c < D; c += 4) {
      float a[4][4], av[4][4], bq[TQ][4], bg[TQ][4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        lds_vec(a[r], ks + (ty + 16 * r) * LD + c);
        lds_vec(av[r], vs + (ty + 16 * r) * LD + c);
      }
#pragma unroll
      for (int qq = 0; qq < TQ; ++qq) {
        lds_vec(bq[qq], qs + (tx + 16 * qq) * LD + c);
        lds_vec(bg[qq], dos + (tx + 16 * qq) * LD + c);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int qq = 0; qq < TQ; ++qq) {
            s[r][qq] = fmaf(a[r][e], bq[qq][e], s[r][qq]);
            dp[r][qq] = fmaf(av[r][e], bg[qq][e], dp[r][qq]);
          }
    }
    // P^T and dS^T; masked pairs (key past Nk or past the row's causal limit, row past Nq) give 0
#pragma unroll
    for (int qq = 0; qq < TQ; ++qq) {
      const int il = tx + 16 * qq, i = i0 + il;
      const float nli = nl_s[il], ndi = nd_s[il];
      float pr[4], dsr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int kj = k0 + ty + 16 * r;
        const bool vis = kj < p.Nk && i < p.Nq && (!p.causal || kj <= i + p.causal_off);
        pr[r] = vis ? ex2_approx(fmaf(s[r][qq], p.c, nli)) : 0.f;
        dsr[r] = pr[r] * (dp[r][qq] + ndi);
      }
      *reinterpret_cast<float4*>(ps + il * MP + 4 * ty) = make_float4(pr[0], pr[1], pr[2], pr[3]);
      *reinterpret_cast<float4*>(dss + il * MP + 4 * ty) = make_float4(dsr[0], dsr[1], dsr[2], dsr[3]);
    }
    __syncthreads();
    // dV += P^T dO, dK += dS^T Q over the step's query rows, in order
#pragma unroll 4
    for (int il = 0; il < BN; ++il) {
      float pr[4], dr[4], go[NH][4], qv[NH][4];
      lds_vec(pr, ps + il * MP + 4 * ty);
      lds_vec(dr, dss + il * MP + 4 * ty);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        lds_vec(go[h], dos + il * LD + 64 * h + 4 * tx);
        lds_vec(qv[h], qs + il * LD + 64 * h + 4 * tx);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dv_acc[r][4 * h + e] = fmaf(pr[r], go[h][e], dv_acc[r][4 * h + e]);
            dk_acc[r][4 * h + e] = fmaf(dr[r], qv[h][e], dk_acc[r][4 * h + e]);
          }
    }
    __syncthreads();  // this stage and P^T, dS^T may be overwritten
  }
  cp_async_wait<0>();  // n_steps >= 1, so every copy was waited for above; kept for a zero-step grid
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int kl = ty + 16 * r;
    if (kl >= kvalid) continue;
    const size_t off = (static_cast<size_t>(bhkv) * p.Nk + k0 + kl) * D + 4 * tx;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      *reinterpret_cast<float4*>(p.dv + off + 64 * h) =
          make_float4(dv_acc[r][4 * h], dv_acc[r][4 * h + 1], dv_acc[r][4 * h + 2], dv_acc[r][4 * h + 3]);
      *reinterpret_cast<float4*>(p.dk + off + 64 * h) =
          make_float4(dk_acc[r][4 * h] * p.scale, dk_acc[r][4 * h + 1] * p.scale, dk_acc[r][4 * h + 2] * p.scale,
                      dk_acc[r][4 * h + 3] * p.scale);
    }
  }
}

// Shared memory of the dQ kernel (floats): Q, dO [BM][LD] and the CTA's nl, -D [BM]; two stages of K, V
// [BN][LD]; dS as [BN keys][MP].
template <int D>
constexpr int dq_smem_floats() {
  using T = F32Tile<D>;
  return 2 * T::BM * T::LD + 2 * T::BM + 2 * (2 * T::BN * T::LD) + T::BN * T::MP;
}

template <int D>
__global__ void __launch_bounds__(BW_THREADS) fa_bwd_dq_fp32_kernel(const BwdF32Params p) {
  using T = F32Tile<D>;
  constexpr int BM = T::BM, BN = T::BN, TQ = T::TQ, NH = T::NH, LD = T::LD, MP = T::MP;
  constexpr int STAGE = 2 * BN * LD;
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                       // [BM][LD]
  float* dos = qs + BM * LD;            // [BM][LD]
  float* nl_s = dos + BM * LD;          // [BM]
  float* nd_s = nl_s + BM;              // [BM]
  float* st0 = nd_s + BM;               // stage s at st0 + s * STAGE: K [BN][LD], V [BN][LD]
  float* dss = st0 + 2 * STAGE;         // [BN keys][MP]

  const int n_qblk = (p.Nq + BM - 1) / BM;
  const int qb = static_cast<int>(blockIdx.x % n_qblk);
  const int bh = static_cast<int>(blockIdx.x / n_qblk);
  const int b = bh / p.H, h = bh % p.H;
  const int bhkv = b * p.Hkv + h / (p.H / p.Hkv);
  const int i0 = qb * BM;
  const int qvalid = min(BM, p.Nq - i0);
  copy_rows_async<D, BM>(qs, p.q + (static_cast<size_t>(bh) * p.Nq + i0) * D, qvalid);
  copy_rows_async<D, BM>(dos, p.dout + (static_cast<size_t>(bh) * p.Nq + i0) * D, qvalid);
  copy_vec_async(nl_s, p.nl + static_cast<size_t>(bh) * p.Nq_pad + i0, BM);  // Nq_pad >= i0 + BM
  copy_vec_async(nd_s, p.negd + static_cast<size_t>(bh) * p.Nq_pad + i0, BM);
  cp_async_commit();

  // keys any row of this block sees: j <= i0 + BM - 1 + causal_off under the mask
  const int k_end = p.causal ? min(p.Nk, i0 + BM + p.causal_off) : p.Nk;
  const int n_steps = (k_end + BN - 1) / BN;
  auto issue_step = [&](int t) {
    float* st = st0 + (t & 1) * STAGE;
    const int j0 = t * BN;
    const int kvalid = min(BN, p.Nk - j0);
    copy_rows_async<D, BN>(st, p.k + (static_cast<size_t>(bhkv) * p.Nk + j0) * D, kvalid);
    copy_rows_async<D, BN>(st + BN * LD, p.v + (static_cast<size_t>(bhkv) * p.Nk + j0) * D, kvalid);
    cp_async_commit();
  };
  issue_step(0);

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float dq_acc[4][4 * NH];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4 * NH; ++c) dq_acc[r][c] = 0.f;

  for (int t = 0; t < n_steps; ++t) {
    if (t + 1 < n_steps) {
      issue_step(t + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* kst = st0 + (t & 1) * STAGE;
    const float* vst = kst + BN * LD;
    const int j0 = t * BN;
    // S = Q K^T and dP = dO V^T for this thread's 4 x TQ block, summed over c in order
    float s[4][TQ], dp[4][TQ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int kk = 0; kk < TQ; ++kk) s[r][kk] = dp[r][kk] = 0.f;
#pragma unroll 2
    for (int c = 0; c < D; c += 4) {
      float a[4][4], ag[4][4], bk[TQ][4], bv[TQ][4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        lds_vec(a[r], qs + (ty + 16 * r) * LD + c);
        lds_vec(ag[r], dos + (ty + 16 * r) * LD + c);
      }
#pragma unroll
      for (int kk = 0; kk < TQ; ++kk) {
        lds_vec(bk[kk], kst + (tx + 16 * kk) * LD + c);
        lds_vec(bv[kk], vst + (tx + 16 * kk) * LD + c);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int kk = 0; kk < TQ; ++kk) {
            s[r][kk] = fmaf(a[r][e], bk[kk][e], s[r][kk]);
            dp[r][kk] = fmaf(ag[r][e], bv[kk][e], dp[r][kk]);
          }
    }
#pragma unroll
    for (int kk = 0; kk < TQ; ++kk) {
      const int jl = tx + 16 * kk, j = j0 + jl;
      float dsr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int il = ty + 16 * r, i = i0 + il;
        const bool vis = j < p.Nk && i < p.Nq && (!p.causal || j <= i + p.causal_off);
        const float pr = vis ? ex2_approx(fmaf(s[r][kk], p.c, nl_s[il])) : 0.f;
        dsr[r] = pr * (dp[r][kk] + nd_s[il]);
      }
      *reinterpret_cast<float4*>(dss + jl * MP + 4 * ty) = make_float4(dsr[0], dsr[1], dsr[2], dsr[3]);
    }
    __syncthreads();
    // dQ += dS K over the step's keys, in order
#pragma unroll 4
    for (int jl = 0; jl < BN; ++jl) {
      float dr[4], kv[NH][4];
      lds_vec(dr, dss + jl * MP + 4 * ty);
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) lds_vec(kv[hh], kst + jl * LD + 64 * hh + 4 * tx);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
          for (int e = 0; e < 4; ++e) dq_acc[r][4 * hh + e] = fmaf(dr[r], kv[hh][e], dq_acc[r][4 * hh + e]);
    }
    __syncthreads();  // this stage and dS may be overwritten
  }
  cp_async_wait<0>();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int il = ty + 16 * r;
    if (il >= qvalid) continue;
    const size_t off = (static_cast<size_t>(bh) * p.Nq + i0 + il) * D + 4 * tx;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
      *reinterpret_cast<float4*>(p.dq + off + 64 * hh) =
          make_float4(dq_acc[r][4 * hh] * p.scale, dq_acc[r][4 * hh + 1] * p.scale, dq_acc[r][4 * hh + 2] * p.scale,
                      dq_acc[r][4 * hh + 3] * p.scale);
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
