// fa_bwd.cu -- backward launches: the per-row prep pass and the bf16 instantiations of the dK/dV
// and dQ kernels (fa_bwd_kernel.cuh).
//
// Source: "Flash Attention 代码填空 (Level 2-3)", Exercise 5 (recompute P from the saved row
// statistics, dV_j += P_ij^T dO_i); the remaining gradients are the chain rule through the softmax.
#include "fa_bwd_kernel.cuh"

namespace fa {

// Tile choices.  dK/dV: 128 keys per CTA, 64 query rows per step; the ring of Q/dO tiles is deep
// enough that copies land before the MMA warp reaches them (it only refills a stage after the
// gradient MMAs of the step it held have completed): 8 stages at d = 64, 4 at d = 128.
// dQ: two 128-row query tiles per CTA, 64 keys per step; K/V rings of 6 stages at d = 64 (+0.8% over 4)
// and 3 at d = 128 (+1.7% over 2).
// d=64 uses three score slots in TMEM (512 columns), d=128 two (its dV and dK take 256).
// ATMEM (d = 64 only: tensor memory has no room at d = 128): the dQ kernel's S and dP MMAs take Q and
// dO from tensor memory.
using BwdKV64 = BwdKVCfg<64, 64, 8, 3>;
using BwdKV128 = BwdKVCfg<128, 64, 4, 2>;
using BwdQ64 = BwdQCfg<64, 64, 6, true>;
using BwdQ128 = BwdQCfg<128, 64, 3, false>;

// D_i = sum_c dO_ic O_ic (fp32 over the bf16 inputs) and nl_i = -L_i log2(e) for the rows of
// [BH][Nq_pad], written interleaved by row pairs: rowv[pair] = (nl_2i, nl_2i+1, -D_2i, -D_2i+1)
// (negated, so the kernels form dP - D with one add).
// Rows i >= Nq get D = 0 and nl = -inf, so their P is exactly 0.
// A group of D/8 lanes covers one row with 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ dout,
                                                          const float* __restrict__ lse, float* __restrict__ rowv,
                                                          long long rows_pad, int Nq, int Nq_pad) {
  griddep_launch_dependents();  // the dK/dV kernel may start its set-up; it waits for this grid's rows
  constexpr int LPR = D / 8;  // lanes per row
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = gt / LPR;
  const int part = static_cast<int>(gt % LPR);
  const bool live = r < rows_pad;
  const long long bh = live ? r / Nq_pad : 0;
  const int i = live ? static_cast<int>(r % Nq_pad) : 0;
  const bool in_range = live && i < Nq;
  float acc = 0.f;
  if (in_range) {
    const size_t off = (static_cast<size_t>(bh) * Nq + i) * D + part * 8;
    const uint4 a = ldg_stream(o + off);
    const uint4 g = ldg_stream(dout + off);
    acc = bf16lo(a.x) * bf16lo(g.x) + bf16hi(a.x) * bf16hi(g.x);
    acc += bf16lo(a.y) * bf16lo(g.y) + bf16hi(a.y) * bf16hi(g.y);
    acc += bf16lo(a.z) * bf16lo(g.z) + bf16hi(a.z) * bf16hi(g.z);
    acc += bf16lo(a.w) * bf16lo(g.w) + bf16hi(a.w) * bf16hi(g.w);
  }
#pragma unroll
  for (int m = LPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (live && part == 0) {
    const size_t base = static_cast<size_t>(r - (r & 1)) * 2 + (r & 1);  // Nq_pad is even: pairs stay in a head
    rowv[base] = in_range ? -lse[static_cast<size_t>(bh) * Nq + i] * 1.4426950408889634f : -INFINITY;
    rowv[base + 2] = in_range ? -acc : 0.f;
  }
}

cudaError_t launch_bwd_prep(const BwdLaunch& a) {
  const long long rows = static_cast<long long>(a.BH) * a.Nq_pad;
  const long long threads = rows * (a.d / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks <= 0 || blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (a.d == 64)
    fa_bwd_prep_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse, a.rowv, rows, a.Nq,
        a.Nq_pad);
  else
    fa_bwd_prep_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse, a.rowv, rows, a.Nq,
        a.Nq_pad);
  return cudaGetLastError();
}

template <class C>
cudaError_t launch_dkdv(const BwdLaunch& a) {
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkdv_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  BwdKVParams p;
  p.dk = a.dk;
  p.dv = a.dv;
  p.rowv = a.rowv;
  p.err = a.err;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.Nq_pad = a.Nq_pad;
  p.n_kblk = (a.Nk + C::BK - 1) / C::BK;
  p.n_qt = (a.Nq + C::BQ - 1) / C::BQ;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.causal = a.causal;
  p.causal_off = a.Nk - a.Nq;
  p.c = a.c;
  p.scale = a.scale;
  p.fault = a.fault;
  if (p.n_qt * C::BQ > a.Nq_pad) return cudaErrorInvalidValue;  // the vectors are read in whole steps
  const long long grid = static_cast<long long>(p.n_kblk) * a.BHkv;
  if (grid <= 0 || grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_dependent(fa_bwd_dkdv_kernel<C>, static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, a.stream,
                          *a.tm_k_kv, *a.tm_v_kv, *a.tm_q_kv, *a.tm_do_kv, p);
}

template <class C>
cudaError_t launch_dq(const BwdLaunch& a) {
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_dq_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  BwdQParams p;
  p.dq = a.dq;
  p.rowv = a.rowv;
  p.err = a.err;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.Nq_pad = a.Nq_pad;
  p.n_qblk = (a.Nq + C::BR * C::NQT - 1) / (C::BR * C::NQT);
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.causal = a.causal;
  p.causal_off = a.Nk - a.Nq;
  p.c = a.c;
  p.scale = a.scale;
  const long long grid = static_cast<long long>(p.n_qblk) * a.BH;
  if (grid <= 0 || grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  // Launched as a programmatic dependent of the dK/dV kernel, which it does not read (the row values
  // of the prep kernel are complete once every dK/dV CTA has passed its wait): its CTAs fill the
  // SMs that the dK/dV grid's last wave leaves idle.
  return launch_dependent(fa_bwd_dq_kernel<C>, static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, a.stream,
                          *a.tm_q_q, *a.tm_do_q, *a.tm_k_q, *a.tm_v_q, p);
}

BwdGeometry bwd_geometry(int d) {
  BwdGeometry g;
  g.kv_keys = BwdKV64::BK;
  g.kv_qrows = BwdKV64::BQ;
  g.q_rows = BwdQ64::BR;
  g.q_keys = BwdQ64::BC;
  g.nq_align = BwdKV64::BQ;
  static_assert(BwdKV64::BQ == BwdKV128::BQ && BwdQ64::BC == BwdQ128::BC, "one geometry for both head sizes");
  (void)d;
  return g;
}

cudaError_t launch_bwd_bf16(const BwdLaunch& a) {
  if (a.causal && a.Nq > a.Nk) return cudaErrorInvalidValue;
  cudaError_t e = launch_bwd_prep(a);
  if (e != cudaSuccess) return e;
  if (a.d == 64) {
    if ((e = launch_dkdv<BwdKV64>(a)) != cudaSuccess) return e;
    return launch_dq<BwdQ64>(a);
  }
  if ((e = launch_dkdv<BwdKV128>(a)) != cudaSuccess) return e;
  return launch_dq<BwdQ128>(a);
}

}  // namespace fa
