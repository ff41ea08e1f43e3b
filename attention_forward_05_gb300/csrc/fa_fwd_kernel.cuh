// fa_fwd_kernel.cuh -- fused FlashAttention forward for sm_103a.
//
// Sources (web pages, cited by title and section):
//   [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
//   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
//
// Algorithm: Q-outer / KV-inner tiling with the online-softmax recurrence
// ([T1] §2.3 and §3.1): for each key tile j the row maximum m, the running sum
// l and the unnormalised output O are updated with alpha = exp(m_old - m_new);
// O is divided by l once after the last tile ([T3] demo 3, deferred
// normalisation).  The score tile lives only in tensor memory.
//
// One CTA owns NQT query tiles of 128 rows of one (batch, head) and walks all
// key tiles of Bc rows.  Warp roles:
//   warps 0 .. 4*NQT-1   softmax warpgroup t = warp/4 owns query tile t; thread
//                        = one query row (TMEM lane).  It reads S_t from TMEM,
//                        updates m and l, rescales O_t in TMEM when needed,
//                        writes P_t (bf16, or fp32 for the TF32 path) back over
//                        S_t, and finally writes O_t / l and the LSE.
//   warp 4*NQT           TMA producer: Q once, then K_j and V_j into a ring of
//                        STAGES shared-memory slots (mbarrier full/empty pairs).
//   warp 4*NQT+1         MMA issuer (one thread): S_t = Q_t K_j^T (both operands
//                        in shared memory, K-major, 128-byte swizzle) and
//                        O_t += P_t V_j (P from tensor memory, V MN-major).
// With NQT = 2 the two query tiles ping-pong: while warpgroup 0 does the
// softmax of step j the tensor core computes tile 1's products, and vice versa
// ([T3] demo 3 remark on FA3-style ping-pong of softmax and MMA).
//
// Lazy rescale: a row's reference maximum m_ref only moves when the new
// maximum exceeds it by more than tau (log2 units).  P = 2^(t - m_ref) then
// stays below 2^tau, and since O and l share m_ref, O / l is unchanged; with
// tau = 0 this is exactly the per-step correction of [T1] §2.3.  Once a row
// has a reference maximum, tiles take fast paths that compute P against it
// straight away: a row sum of P of at most 2^tau proves that no score moved
// past m_ref + tau, so a row maximum is formed only where that test fails.
#pragma once

#include <type_traits>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

template <typename T, int D_, int BC_, int NQT_, int STAGES_, int MINB_ = 1, bool PV2_ = false>
struct FwdCfg {
  using Elem = T;
  static constexpr int D = D_;
  static constexpr int BC = BC_;
  static constexpr int NQT = NQT_;
  static constexpr int STAGES = STAGES_;
  static constexpr int MINB = MINB_;    // CTAs per SM the launch bounds ask for
  // PV2: the softmax hands over P in two halves (key columns [0, BC/2) first), and P V of the first
  // half is issued while the second half is still being exponentiated.
  static constexpr bool PV2 = PV2_;
  static constexpr int BR = 128;
  static constexpr int ESZ = static_cast<int>(sizeof(T));
  static constexpr bool TF32 = (ESZ == 4);
  static constexpr uint32_t FMT = TF32 ? 2u : 1u;
  static constexpr int CHUNK = 128 / ESZ;  // elements per 128-byte swizzled row segment
  static constexpr int NCH = D / CHUNK;    // segments per row
  static constexpr int Q_CH_BYTES = BR * 128;
  static constexpr int KV_CH_BYTES = BC * 128;
  static constexpr int Q_BYTES = NCH * Q_CH_BYTES;
  static constexpr int KV_BYTES = NCH * KV_CH_BYTES;
  // V as the B operand of O += P V.  bf16: V tiles [Bc keys][D] are MN-major.  tf32 MMAs accept only
  // K-major operands, so the fp32 path reads a key-major copy V^T [D][Nk] and its tiles are [D rows][Bc].
  static constexpr bool V_KMAJOR = TF32;
  static constexpr int NCH_V = V_KMAJOR ? BC / CHUNK : NCH;
  static constexpr int V_CH_BYTES = V_KMAJOR ? D * 128 : KV_CH_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // barriers: q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[NQT], p_full[NQT], o_done[NQT], drain
  static constexpr int NBAR = 1 + 4 * STAGES + 4 * NQT + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  // Key-split CTAs (FwdParams::ks_half) exist for the two-tile bf16 configuration without the two-half
  // hand-over; their tile slot 1 leaves its rows' (m, l) here for the merge.
  static constexpr bool KS = NQT == 2 && !TF32 && !PV2;
  static constexpr int OFF_ML = OFF_MISC + 16;
  static constexpr int ML_BYTES = KS ? BR * 8 : 0;
  static constexpr int SMEM_BYTES = OFF_ML + ML_BYTES + 1024;  // + slack to align the base to 1024
  static constexpr int MMA_K = 32 / ESZ;                  // K of one tcgen05.mma (32 bytes)
  static constexpr int O_COL0 = NQT * BC;                 // TMEM: S_t at t*BC, O_t at O_COL0 + t*D
  static constexpr int TMEM_NEED = NQT * (BC + D);
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int P_COLS = BC * ESZ / 4;  // 32-bit TMEM columns of one P row
  static constexpr int P_COLS_PER_K = MMA_K * ESZ / 4;
  static constexpr int COLS = BC;         // key columns of one softmax thread (one query row)
  static constexpr int PCOLS_W = P_COLS;  // P columns written by one softmax warpgroup
  static constexpr int OCOLS = D;         // O columns rescaled and stored by one softmax warpgroup
  static constexpr int NWARPS = 4 * NQT + 2;
  static constexpr int NTHREADS = 32 * NWARPS;
  static constexpr int LOAD_WARP = 4 * NQT;
  static constexpr int MMA_WARP = 4 * NQT + 1;
  // Registers per thread: each of the SM's 4 sub-partitions holds 16384 registers and
  // ceil(warps per SM / 4) warps, in 8-register steps.
  static constexpr int WARPS_PER_SUBPART = (NWARPS * MINB + 3) / 4;
  static constexpr int MAXREG_RAW = (16384 / (WARPS_PER_SUBPART * 32)) / 8 * 8;
  static constexpr int MAXREG = MAXREG_RAW > 248 ? 248 : MAXREG_RAW;
  static_assert(D % CHUNK == 0, "head dim must be a whole number of 128-byte segments");
  static_assert(BC % 32 == 0 && BC >= 32 && BC <= 256, "key tile");
  static_assert(COLS % 32 == 0 && PCOLS_W % 32 == 0 && OCOLS % 32 == 0, "whole 32-column chunks");
  static_assert(!PV2 || (!TF32 && BC >= 128 && (BC / 2) % 64 == 0), "P handed over in two halves of whole packed chunks");
  static_assert(TMEM_NEED <= 512 / MINB, "tensor memory");
  static_assert(SMEM_BYTES * MINB <= 227 * 1024, "shared memory");
};

struct FwdParams {
  void* o;
  float* lse;
  int* err;
  int Nq, Nk, n_qblk;
  int BH, H, Hkv;       // query heads per batch H; key/value heads Hkv (H % Hkv == 0)
  int kv_per_split;     // keys per split (a multiple of Bc); the CTA covers [split*kv_per_split, ...)
  int n_split;          // 1: write O and LSE; > 1: write unnormalised partial states for the merge
  float* ws_o;          // [n_split][BH][Nq][D] fp32 unnormalised O (split mode)
  float* ws_ml;         // [n_split][BH][Nq][2] fp32 (m in log2 units, l) (split mode)
  int causal;           // 1: query row i sees keys j <= i + causal_off only
  int causal_off;       // Nk - Nq (mask aligned to the bottom-right corner)
  float c, tau;
  float p_lim;          // 2^tau: largest row sum of P that proves no maximum moved past m_ref + tau
  int fault;
  // Key-split CTAs (no mask, n_split == 1; ks_half = 0: none).  CTAs below n_whole are the usual ones;
  // CTA n_whole + i takes one 128-row query tile, number ks_tile0 + i of the head-major list of 128-row
  // tiles, and gives its two tile slots the keys [0, ks_half) and [ks_half, Nk); at the end slot 0
  // merges the two partial states (both in this CTA's tensor memory) and writes O and the LSE.
  int n_whole, ks_tile0, ks_half;
};

// wait-site identifiers recorded with a timeout
enum : int { W_Q = 1, W_KF, W_VF, W_KE, W_VE, W_SF, W_PF, W_OD, W_DRAIN_MMA, W_DRAIN_K, W_DRAIN_V };

// Row maximum (MAX) or minimum of the BC scores a thread holds: 4 independent
// chains over groups of 8 elements, two new elements per 3-input max/min.
template <int NCOL, bool MAX>
__device__ __forceinline__ float row_extreme(const uint32_t (&sr)[NCOL / 32][32]) {
  static_assert(NCOL % 8 == 0, "groups of 8");
  float a[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float x = __uint_as_float(sr[0][2 * u]), y = __uint_as_float(sr[0][2 * u + 1]);
    a[u] = MAX ? fmaxf(x, y) : fminf(x, y);
  }
#pragma unroll
  for (int g = 1; g < NCOL / 8; ++g)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = 8 * g + 2 * u;  // e and e + 1 lie in the same 32-column chunk
      const float x = __uint_as_float(sr[e / 32][e % 32]), y = __uint_as_float(sr[e / 32][e % 32 + 1]);
      a[u] = MAX ? max3f(a[u], x, y) : min3f(a[u], x, y);
    }
  return MAX ? max3f(a[0], a[1], fmaxf(a[2], a[3])) : min3f(a[0], a[1], fminf(a[2], a[3]));
}

// bf16 P: for 32-bit column q, elements 2q (low half) and 2q+1 (high half) of the row.
template <int NCOL, bool TAIL>
__device__ __forceinline__ void softmax_p_bf16(const uint32_t (&sr)[NCOL / 32][32], uint32_t (&pk)[NCOL / 64][32],
                                               uint64_t c2, uint64_t negm2, int valid, uint64_t (&rs2)[2]) {
#pragma unroll
  for (int qc = 0; qc < NCOL / 2; ++qc) {
    const int e0 = 2 * qc;
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[e0 / 32][e0 % 32]), __uint_as_float(sr[e0 / 32][e0 % 32 + 1])),
                              c2, negm2);
    float x0, x1;
    f2_unpack_f(x, x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if (TAIL) {
      if (e0 >= valid) p0 = 0.f;
      if (e0 + 1 >= valid) p1 = 0.f;
    }
    rs2[qc & 1] = f2_add(rs2[qc & 1], f2_pack(p0, p1));
    pk[qc / 32][qc % 32] = pack_bf16x2(p0, p1);
  }
}

// tf32 P: one element per 32-bit column, rounded to the nearest tf32 (the MMA would truncate).
template <int NCOL, bool TAIL>
__device__ __forceinline__ void softmax_p_tf32(uint32_t (&sr)[NCOL / 32][32], uint64_t c2, uint64_t negm2, int valid,
                                               uint64_t (&rs2)[2]) {
#pragma unroll
  for (int e0 = 0; e0 < NCOL; e0 += 2) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[e0 / 32][e0 % 32]), __uint_as_float(sr[e0 / 32][e0 % 32 + 1])),
                              c2, negm2);
    float x0, x1;
    f2_unpack_f(x, x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if (TAIL) {
      if (e0 >= valid) p0 = 0.f;
      if (e0 + 1 >= valid) p1 = 0.f;
    }
    rs2[(e0 >> 1) & 1] = f2_add(rs2[(e0 >> 1) & 1], f2_pack(p0, p1));
    sr[e0 / 32][e0 % 32] = round_tf32_bits(p0);
    sr[e0 / 32][e0 % 32 + 1] = round_tf32_bits(p1);
  }
}

// Warp-collective: r[0..15] to 16 consecutive 32-bit TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_st16_lo(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <class C>
__global__ void __maxnreg__(C::MAXREG)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Without a mask, blockIdx.x = (split * BH + bh) * n_qblk + qb: CTAs sharing a head and key range
  // are adjacent.  With a causal mask a CTA's work grows with its query block, so the query block is
  // the slowest index, last block first: blockIdx.x = (n_qblk - 1 - qb) * (n_split * BH) + split * BH
  // + bh.  The longest CTAs start first and the shortest fill the last wave.
  int qb, bh, split, q0;
  // a key-split CTA (FwdParams): both tile slots hold the same 128 query rows, over two key ranges
  const bool ks = C::KS && p.ks_half > 0 && static_cast<int>(blockIdx.x) >= p.n_whole;
  if (p.causal) {
    const int per_qb = p.n_split * p.BH;
    qb = p.n_qblk - 1 - static_cast<int>(blockIdx.x / per_qb);
    bh = static_cast<int>(blockIdx.x % per_qb) % p.BH;
    split = static_cast<int>(blockIdx.x % per_qb) / p.BH;
    q0 = qb * C::BR * C::NQT;
  } else if (ks) {
    const int nq1 = (p.Nq + C::BR - 1) / C::BR;
    const int tile = p.ks_tile0 + static_cast<int>(blockIdx.x) - p.n_whole;
    bh = tile / nq1;
    qb = 0;
    split = 0;
    q0 = (tile % nq1) * C::BR;
  } else {
    qb = static_cast<int>(blockIdx.x % p.n_qblk);
    bh = static_cast<int>(blockIdx.x / p.n_qblk) % p.BH;
    split = static_cast<int>(blockIdx.x / (p.n_qblk * p.BH));
    q0 = qb * C::BR * C::NQT;
  }
  const int kvh = (bh / p.H) * p.Hkv + (bh % p.H) / (p.H / p.Hkv);  // key/value head of this query head
  const int k_begin = split * p.kv_per_split;
  const int k_end = min(p.Nk, k_begin + p.kv_per_split);  // the host makes every split non-empty
  // keys past the causal limit of the CTA's last row are never loaded or multiplied
  const int k_hi = p.causal ? min(k_end, q0 + C::NQT * C::BR + p.causal_off) : k_end;
  // key range of tile slot t (the CTA's range, or one of the two halves in a key-split CTA)
  auto slot_lo = [&](int t) { return ks && t == 1 ? p.ks_half : k_begin; };
  auto slot_hi = [&](int t) { return ks && t == 0 ? min(k_end, p.ks_half) : k_end; };
  const int T = ks ? (slot_hi(0) + C::BC - 1) / C::BC
                   : (k_hi > k_begin ? (k_hi - k_begin + C::BC - 1) / C::BC : 0);  // 0 only in split mode
  // Key tiles query tile t needs: with a causal mask the tiles past its own last row's limit are
  // skipped (no products, no softmax); the last tile needs all T.
  auto tile_steps = [&](int t) {
    if (ks) return (slot_hi(t) - slot_lo(t) + C::BC - 1) / C::BC;
    const int hi = p.causal ? min(k_end, q0 + (t + 1) * C::BR + p.causal_off) : k_end;
    return hi > k_begin ? (hi - k_begin + C::BC - 1) / C::BC : 0;
  };
  const int trow = ks ? 0 : C::BR;  // rows of tile slot t start at q0 + t * trow

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_q = bar0;
  auto bar_kf = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_vf = [&](int s) { return bar0 + 8u * (1 + C::STAGES + s); };
  auto bar_ke = [&](int s) { return bar0 + 8u * (1 + 2 * C::STAGES + s); };
  auto bar_ve = [&](int s) { return bar0 + 8u * (1 + 3 * C::STAGES + s); };
  auto bar_sf = [&](int t) { return bar0 + 8u * (1 + 4 * C::STAGES + t); };
  auto bar_pf = [&](int t) { return bar0 + 8u * (1 + 4 * C::STAGES + C::NQT + t); };
  auto bar_od = [&](int t) { return bar0 + 8u * (1 + 4 * C::STAGES + 2 * C::NQT + t); };
  const uint32_t bar_drain = bar0 + 8u * (1 + 4 * C::STAGES + 3 * C::NQT);
  auto bar_ph = [&](int t) { return bar0 + 8u * (2 + 4 * C::STAGES + 3 * C::NQT + t); };  // first half of P
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_kf(s), 1);
      mbar_init(bar_vf(s), 1);
      mbar_init(bar_ke(s), 1);
      mbar_init(bar_ve(s), 1);
    }
    for (int t = 0; t < C::NQT; ++t) {
      mbar_init(bar_sf(t), 1);
      mbar_init(bar_pf(t), 4);  // one arrive per softmax warp of the tile
      mbar_init(bar_ph(t), 4);
      mbar_init(bar_od(t), 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // After the fp32 prep kernel this grid is its programmatic dependent: the set-up above overlapped
  // that kernel, whose rounded Q, K and V^T are read only after this wait (a no-op otherwise).  A
  // merge kernel launched after this one (split mode) may be scheduled once every CTA has started;
  // it waits for this grid's completion before it reads the partial states.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && T > 0) {
      int nk_done = 0, nv_done = 0;  // key tiles whose K (resp. V) copy was issued: tiles 0 .. n-1
      mbar_expect_tx(bar_q, C::NQT * C::Q_BYTES);
#pragma unroll
      for (int t = 0; t < C::NQT; ++t)
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sbase + C::OFF_Q + t * C::Q_BYTES + c * C::Q_CH_BYTES, &tm_q, bar_q, c * C::CHUNK,
                      q0 + t * trow, bh);
      if constexpr (C::KS) {
        if (ks) {
          // Copy n = 2j + t is key tile j of slot t (slot 1 may have one tile fewer): ring stage n % STAGES.
          const int T1 = tile_steps(1);
          int n = 0;
          for (int j = 0; j < T; ++j) {
            for (int t = 0; t < 2; ++t) {
              if (t == 1 && j >= T1) break;
              const int s = n % C::STAGES;
              const uint32_t ph = ((n / C::STAGES) & 1) ^ 1;
              const int key = slot_lo(t) + j * C::BC;
              if (!mbar_wait(bar_ke(s), ph, abort_flag, p.err, W_KE)) goto ks_loads_done;
              mbar_expect_tx(bar_kf(s), C::KV_BYTES);
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sbase + C::OFF_K + s * C::KV_BYTES + c * C::KV_CH_BYTES, &tm_k, bar_kf(s), c * C::CHUNK,
                            key, kvh);
              nk_done = n + 1;
              if (!mbar_wait(bar_ve(s), ph, abort_flag, p.err, W_VE)) goto ks_loads_done;
              mbar_expect_tx(bar_vf(s), C::KV_BYTES);
#pragma unroll
              for (int c = 0; c < C::NCH_V; ++c)
                tma_load_3d(sbase + C::OFF_V + s * C::KV_BYTES + c * C::V_CH_BYTES, &tm_v, bar_vf(s), c * C::CHUNK,
                            key, kvh);
              nv_done = n + 1;
              ++n;
            }
          }
        ks_loads_done:;
        }
      }
      for (int j = 0; !ks && j < T; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = ((j / C::STAGES) & 1) ^ 1;
        if (!mbar_wait(bar_ke(s), ph, abort_flag, p.err, W_KE)) break;
        if (!(p.fault == 1 && j == 0)) {
          mbar_expect_tx(bar_kf(s), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sbase + C::OFF_K + s * C::KV_BYTES + c * C::KV_CH_BYTES, &tm_k, bar_kf(s),
                        c * C::CHUNK, k_begin + j * C::BC, kvh);
        }
        nk_done = j + 1;
        if (!mbar_wait(bar_ve(s), ph, abort_flag, p.err, W_VE)) break;
        mbar_expect_tx(bar_vf(s), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH_V; ++c) {
          if constexpr (C::V_KMAJOR)
            tma_load_3d(sbase + C::OFF_V + s * C::KV_BYTES + c * C::V_CH_BYTES, &tm_v, bar_vf(s),
                        k_begin + j * C::BC + c * C::CHUNK, 0, kvh);
          else
            tma_load_3d(sbase + C::OFF_V + s * C::KV_BYTES + c * C::V_CH_BYTES, &tm_v, bar_vf(s), c * C::CHUNK,
                        k_begin + j * C::BC, kvh);
        }
        nv_done = j + 1;
      }
      // Drain: every copy this thread issued must land before the CTA exits.  Stage s received
      // the tiles j < n with j % STAGES == s; the last of them completes phase (count - 1).
      mbar_wait_drain(bar_q, 0, p.err, W_DRAIN_K);
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) {
        int nks = (nk_done > s) ? (nk_done - 1 - s) / C::STAGES + 1 : 0;
        if (!ks && p.fault == 1 && s == 0 && nk_done > 0) --nks;  // the skipped copy of tile 0
        const int nvs = (nv_done > s) ? (nv_done - 1 - s) / C::STAGES + 1 : 0;
        if (nks > 0) mbar_wait_drain(bar_kf(s), (nks - 1) & 1, p.err, W_DRAIN_K);
        if (nvs > 0) mbar_wait_drain(bar_vf(s), (nvs - 1) & 1, p.err, W_DRAIN_V);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop, so descriptors and addresses are warp-uniform (uniform
    // registers); one elected lane issues a tile's products and commits of a step in one region
    // (issue_qk and issue_pv are called from that lane; electing per instruction measured 2-5%
    // slower at d=64).  Waits are taken by all lanes and agreed with __all_sync.
    {
      auto wait_all = [&](uint32_t bar, uint32_t parity, int where) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err, where));
      };
      constexpr uint32_t idesc_qk = make_idesc(C::FMT, C::BR, C::BC, 0, 0);
      constexpr uint32_t idesc_pv = make_idesc(C::FMT, C::BR, C::D, 0, C::V_KMAJOR ? 0 : 1);
      // Shared-memory descriptors are built once; each MMA only adds a compile-time offset to the
      // address field (bytes >> 4, bits 0-13: every address here is below 256 KB, so no carry).
      // Rebuilding them per instruction made the issuing thread, not the tensor core, the bottleneck.
      const uint64_t dq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dv0 = C::V_KMAJOR ? sdesc_sw128(sbase + C::OFF_V, 16, 1024)
                                       : sdesc_sw128(sbase + C::OFF_V, C::V_CH_BYTES, 1024);
      auto issue_qk = [&](int t, int s) {
        const uint32_t d_tmem = tmem + t * C::BC;
        const uint64_t qa = dq0 + static_cast<uint64_t>((t * C::Q_BYTES) >> 4);
        const uint64_t kb = dk0 + static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::D / C::MMA_K; ++kk) {
          const int e = kk * C::MMA_K;  // element offset along d: 128-byte segment, then 32-byte step inside it
          const uint32_t oq = ((e / C::CHUNK) * C::Q_CH_BYTES + (e % C::CHUNK) * C::ESZ) >> 4;
          const uint32_t ok_ = ((e / C::CHUNK) * C::KV_CH_BYTES + (e % C::CHUNK) * C::ESZ) >> 4;
          mma_ss<C::TF32>(d_tmem, qa + oq, kb + ok_, idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc, int kk0 = 0, int kk1 = C::BC / C::MMA_K) {
        const uint32_t d_tmem = tmem + C::O_COL0 + t * C::D;
        const uint32_t a_tmem = tmem + t * C::BC;
        const uint64_t vb = dv0 + static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = kk0; kk < kk1; ++kk) {
          uint32_t ov;
          if constexpr (C::V_KMAJOR) {  // [D rows][Bc keys]: step along keys inside 128-byte segments
            const int e = kk * C::MMA_K;
            ov = ((e / C::CHUNK) * C::V_CH_BYTES + (e % C::CHUNK) * C::ESZ) >> 4;
          } else {  // [Bc keys][D]: MN-major, 8-key groups 1024 B apart, 64-column segments LBO apart
            ov = (kk * C::MMA_K * 128) >> 4;
          }
          mma_ts<C::TF32>(d_tmem, a_tmem + kk * C::P_COLS_PER_K, vb + ov, idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
      };
      auto commit = [&](uint32_t bar) {
        if (elect_one()) mma_commit(bar);
        __syncwarp();
      };
      if (C::KS && ks) {
        // Key-split CTA: slot t's key tile j is copy n = 2j + t of the ring (stage n % STAGES); each
        // stage serves one slot, so it is released after that slot's products.
        const int T1 = tile_steps(1);
        bool ok = wait_all(bar_q, 0, W_Q);
        for (int t = 0; ok && t < 2; ++t) {  // the first Q K^T of each slot: copies 0 and 1
          ok = wait_all(bar_kf(t % C::STAGES), (t / C::STAGES) & 1, W_KF);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            issue_qk(t, t % C::STAGES);
            mma_commit(bar_sf(t));
            mma_commit(bar_ke(t % C::STAGES));
          }
          __syncwarp();
        }
        for (int j = 0; ok && j < T; ++j) {
          for (int t = 0; t < 2; ++t) {
            const int Tt = t == 0 ? T : T1;
            if (j >= Tt) break;
            const int n = 2 * j + t, s = n % C::STAGES;
            const int n1 = n + 2, s1 = n1 % C::STAGES;
            const bool next = j + 1 < Tt;
            ok = wait_all(bar_vf(s), (n / C::STAGES) & 1, W_VF);
            if (ok && next) ok = wait_all(bar_kf(s1), (n1 / C::STAGES) & 1, W_KF);
            if (ok) ok = wait_all(bar_pf(t), j & 1, W_PF);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
              issue_pv(t, s, j > 0);
              mma_commit(bar_ve(s));
              if (next) {
                issue_qk(t, s1);
                mma_commit(bar_sf(t));
                mma_commit(bar_ke(s1));
              } else {
                mma_commit(bar_od(t));
              }
            }
            __syncwarp();
          }
        }
      } else {
      bool ok = T > 0 && wait_all(bar_q, 0, W_Q) && wait_all(bar_kf(0), 0, W_KF);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int t = 0; t < C::NQT; ++t) {
            if (tile_steps(t) > 0) {
              issue_qk(t, 0);
              mma_commit(bar_sf(t));
            }
          }
          mma_commit(bar_ke(0));
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % C::STAGES;
        const int j1 = j + 1;
        const int s1 = j1 % C::STAGES;
        // V_j and K_{j+1} are normally resident long before P_t(j) is ready: wait for them first so
        // the chain P ready -> P V -> next Q K^T holds nothing but MMA issue.
        ok = wait_all(bar_vf(s), (j / C::STAGES) & 1, W_VF);
        if (ok && j1 < T) ok = wait_all(bar_kf(s1), (j1 / C::STAGES) & 1, W_KF);
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < C::NQT; ++t) {
          // tile t takes part in steps j < T_t only (T_t = T for the last tile)
          const int Tt = t == C::NQT - 1 ? T : tile_steps(t);
          if (j < Tt) {
            if constexpr (C::PV2) {  // first half of P V as soon as the first half of P is in
              ok = wait_all(bar_ph(t), j & 1, W_PF);
              if (!ok) break;
              tc_fence_after();
              if (elect_one()) issue_pv(t, s, j > 0, 0, C::BC / C::MMA_K / 2);
              __syncwarp();
            }
            ok = wait_all(bar_pf(t), j & 1, W_PF);
            if (!ok) break;
            tc_fence_after();
          }
          // one elected lane issues the step's products and commits for this tile in one go
          if (elect_one()) {
            if (j < Tt) {
              if constexpr (C::PV2)
                issue_pv(t, s, true, C::BC / C::MMA_K / 2, C::BC / C::MMA_K);
              else
                issue_pv(t, s, j > 0);
            }
            if (t == C::NQT - 1) mma_commit(bar_ve(s));
            if (j < Tt) {
              if (j1 < Tt) {
                issue_qk(t, s1);
                mma_commit(bar_sf(t));
              } else {
                mma_commit(bar_od(t));
              }
            }
            if (t == C::NQT - 1 && j1 < T) mma_commit(bar_ke(s1));
          }
          __syncwarp();
        }
      }
      }
      // Drain: all MMAs issued above complete before tensor memory is freed.
      commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, p.err, W_DRAIN_MMA);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    // Warpgroup t = warp / 4 owns query tile t; thread = query row.
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * C::BC;
    const uint32_t tP = tmem + lane_base + t * C::BC;
    const uint32_t tO = tmem + lane_base + C::O_COL0 + t * C::D;
    // keys this row may see in the CTA's range: [k_begin, row_lim)
    const int row_lim = p.causal ? min(k_end, q0 + t * C::BR + row + 1 + p.causal_off) : slot_hi(t);
    const int kb = slot_lo(t);
    const float c = p.c;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const uint64_t c2 = f2_pack(c, c);
    const float& p_lim = p.p_lim;  // read from the kernel parameters where used (no register held)
    const int Tt = tile_steps(t);      // key tiles of this query tile
    for (int j = 0; j < Tt; ++j) {
      bool okw = mbar_wait(bar_sf(t), j & 1, abort_flag, p.err, W_SF);
      okw = __all_sync(0xffffffffu, okw);
      const int valid = row_lim - kb - j * C::BC;  // valid key columns here (may be <= 0)
      if constexpr (!C::TF32 && C::COLS <= 64) {
        // Fast path once every row of the warp has a reference maximum: P is computed against m_ref
        // while the scores are still arriving, 32 columns at a time (the load of the next chunk
        // overlaps the work on this one).  No row maximum is formed: the row sum bounds every P of
        // the row, so a sum of at most 2^tau shows that no score moved past m_ref + tau.  Otherwise
        // (rarely, and always when a maximum did move) the warp falls through to the general path
        // below, which reloads S (not yet overwritten), takes the row maxima and rescales where
        // needed.  A tile with masked columns (causal diagonal, ragged last tile) takes the masked
        // copy of the path, whose P is 0 past each row's `valid` columns.
        // Only for 64-column tiles: with 128 columns the extra live registers spill and the
        // d = 128 kernel measured 25% slower.
        auto fast = [&](auto masked) -> bool {
          constexpr bool TAIL = decltype(masked)::value;
          tc_fence_after();
          const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
          uint32_t sc[2][32];
          uint32_t pk[C::PCOLS_W / 32][32];
          uint64_t rs2[2] = {0ull, 0ull};
          tmem_ld32(tS, sc[0]);
          tmem_wait_ld();
          reg_fence(sc[0]);
#pragma unroll
          for (int cc = 0; cc < C::COLS / 32; ++cc) {
            if (cc + 1 < C::COLS / 32) tmem_ld32(tS + (cc + 1) * 32, sc[(cc + 1) & 1]);
            const uint32_t(&cur)[32] = sc[cc & 1];
#pragma unroll
            for (int qc = 0; qc < 16; ++qc) {
              const uint64_t x = f2_fma(f2_pack(__uint_as_float(cur[2 * qc]), __uint_as_float(cur[2 * qc + 1])), c2,
                                        negm2);
              float x0, x1;
              f2_unpack_f(x, x0, x1);
              float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              if constexpr (TAIL) {
                if (cc * 32 + 2 * qc >= valid) p0 = 0.f;
                if (cc * 32 + 2 * qc + 1 >= valid) p1 = 0.f;
              }
              rs2[qc & 1] = f2_add(rs2[qc & 1], f2_pack(p0, p1));
              const int w = cc * 16 + qc;  // packed column of this pair
              pk[w / 32][w % 32] = pack_bf16x2(p0, p1);
            }
            if (cc + 1 < C::COLS / 32) {
              tmem_wait_ld();
              reg_fence(sc[(cc + 1) & 1]);
            }
          }
          float r0, r1, r2, r3;
          f2_unpack_f(rs2[0], r0, r1);
          f2_unpack_f(rs2[1], r2, r3);
          const float l_tile = (r0 + r1) + (r2 + r3);
          if (!__all_sync(0xffffffffu, l_tile <= p_lim)) return false;
#pragma unroll
          for (int i = 0; i < C::PCOLS_W / 32; ++i) tmem_st32(tP + i * 32, pk[i]);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_pf(t));
          l += l_tile;
          return true;
        };
        if (__all_sync(0xffffffffu, m_ref != -INFINITY)) {
          if (!okw) {
            ok = false;
            break;
          }
          const bool full = __all_sync(0xffffffffu, valid >= C::COLS);
          if (full ? fast(std::false_type{}) : fast(std::true_type{})) continue;
        }
      }
      if constexpr (C::PV2) {
        // Fast path of the two-half hand-over, for a full tile once every row of the warp has a
        // reference maximum: the first half's exponentials start as soon as S is loaded, with no row
        // maximum in front of them.  The first half is handed over when its row sum is at most 2^tau
        // (so none of its scores moved past m_ref + tau) and the second half's maximum is at most
        // m_ref + tau: O then needs no correction.  Otherwise nothing has been stored yet and the
        // warp falls through to the general path, which reloads S.  (Worth it only with a large tau:
        // at tau = 8 the peaked inputs sent a third of the warp-steps down both paths.)
        if (__all_sync(0xffffffffu, valid >= C::COLS && m_ref != -INFINITY)) {
          if (!okw) {
            ok = false;
            break;
          }
          constexpr int HC = C::COLS / 2;
          tc_fence_after();
          uint32_t sv[C::COLS / 32][32];
#pragma unroll
          for (int i = 0; i < C::COLS / 32; ++i) tmem_ld32(tS + i * 32, sv[i]);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < C::COLS / 32; ++i) reg_fence(sv[i]);
          auto& sv_a = reinterpret_cast<uint32_t(&)[HC / 32][32]>(sv[0]);
          auto& sv_b = reinterpret_cast<uint32_t(&)[HC / 32][32]>(sv[HC / 32]);
          const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
          uint32_t pk[C::PCOLS_W / 32][32];
          auto& pk_a = reinterpret_cast<uint32_t(&)[HC / 64][32]>(pk[0]);
          auto& pk_b = reinterpret_cast<uint32_t(&)[HC / 64][32]>(pk[HC / 64]);
          uint64_t rs_a[2] = {0ull, 0ull};
          softmax_p_bf16<HC, false>(sv_a, pk_a, c2, negm2, HC, rs_a);
          const float m_b = (c >= 0.f ? row_extreme<HC, true>(sv_b) : row_extreme<HC, false>(sv_b)) * c;
          float r0, r1, r2, r3;
          f2_unpack_f(rs_a[0], r0, r1);
          f2_unpack_f(rs_a[1], r2, r3);
          const float l_a = (r0 + r1) + (r2 + r3);
          if (__all_sync(0xffffffffu, l_a <= p_lim && m_b <= m_ref + p.tau)) {
#pragma unroll
            for (int i = 0; i < HC / 64; ++i) tmem_st32(tP + i * 32, pk_a[i]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ph(t));
            uint64_t rs_b[2] = {0ull, 0ull};
            softmax_p_bf16<HC, false>(sv_b, pk_b, c2, negm2, HC, rs_b);
#pragma unroll
            for (int i = 0; i < HC / 64; ++i) tmem_st32(tP + (HC / 64 + i) * 32, pk_b[i]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pf(t));
            f2_unpack_f(rs_b[0], r0, r1);
            f2_unpack_f(rs_b[1], r2, r3);
            l += l_a + ((r0 + r1) + (r2 + r3));
            continue;
          }
        }
      }
      // 64-column bf16 tiles: the general path works on one 32-column chunk at a time (the maximum, then
      // P chunk by chunk), which halves the registers it holds; P and the row sum come out the same.
      constexpr bool CHUNKED = !C::TF32 && !C::PV2 && C::COLS == 64;
      uint32_t sr[CHUNKED ? 1 : C::COLS / 32][32];
      float m_part = -INFINITY;
      if constexpr (CHUNKED) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          tmem_ld32(tS + cc * 32, sr[0]);
          tmem_wait_ld();
          reg_fence(sr[0]);
          const int vc = valid - cc * 32;
          if (vc > 0) {
            if (vc < 32) {  // ragged: repeat the chunk's column 0 so max/min ignore the pad
              const uint32_t s0 = sr[0][0];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (e >= vc) sr[0][e] = s0;
            }
            m_part = fmaxf(m_part, (c >= 0.f ? row_extreme<32, true>(sr) : row_extreme<32, false>(sr)) * c);
          }
        }
      } else {  // loaded even when the wait gave up (then the values are stale and unused): a conditional
                // load would keep the row in local memory
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < C::COLS / 32; ++i) tmem_ld32(tS + i * 32, sr[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < C::COLS / 32; ++i) reg_fence(sr[i]);
        if (valid > 0) {
          if (valid < C::COLS) {  // ragged last tile: repeat column 0 so max/min ignore the pad
            const uint32_t s0 = sr[0][0];
#pragma unroll
            for (int i = 0; i < C::COLS / 32; ++i)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (i * 32 + e >= valid) sr[i][e] = s0;
          }
          // extreme of the raw scores (max for scale >= 0, min for scale < 0), times scale*log2(e)
          m_part = (c >= 0.f ? row_extreme<C::COLS, true>(sr) : row_extreme<C::COLS, false>(sr)) * c;
        }
      }
      const float m_tile = m_part;
      ok = okw;
      if (!ok) break;
      const float m_new = fmaxf(m_ref, m_tile);
      const bool need = m_new > m_ref + p.tau;  // always true on the first tile (m_ref = -inf)
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile
        m_ref = m_new;
      }
      // P = 2^(s*c - m_ref) (packed fp32 pairs), row sum in fp32, P written over S in TMEM
      const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
      uint64_t rs2[2] = {0ull, 0ull};
      if constexpr (C::TF32) {
        if (valid >= C::COLS) softmax_p_tf32<C::COLS, false>(sr, c2, negm2, valid, rs2);
        else softmax_p_tf32<C::COLS, true>(sr, c2, negm2, valid, rs2);
#pragma unroll
        for (int i = 0; i < C::COLS / 32; ++i) tmem_st32(tP + i * 32, sr[i]);
      } else if constexpr (C::PV2) {
        // First half of P, then the O correction (P V of this step accumulates into the corrected
        // O), then the signal for the first half of P V; the second half of P follows.
        constexpr int HC = C::COLS / 2;
        uint32_t pk[C::PCOLS_W / 32][32];
        auto& sr_a = reinterpret_cast<uint32_t(&)[HC / 32][32]>(sr[0]);
        auto& sr_b = reinterpret_cast<uint32_t(&)[HC / 32][32]>(sr[HC / 32]);
        auto& pk_a = reinterpret_cast<uint32_t(&)[HC / 64][32]>(pk[0]);
        auto& pk_b = reinterpret_cast<uint32_t(&)[HC / 64][32]>(pk[HC / 64]);
        if (valid >= HC) softmax_p_bf16<HC, false>(sr_a, pk_a, c2, negm2, valid, rs2);
        else softmax_p_bf16<HC, true>(sr_a, pk_a, c2, negm2, valid, rs2);
#pragma unroll
        for (int i = 0; i < HC / 64; ++i) tmem_st32(tP + i * 32, pk_a[i]);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < C::OCOLS / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(tO + cc * 32, orr);
            tmem_wait_ld();
            reg_fence(orr);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2);
              f2_unpack(v, orr[e], orr[e + 1]);
            }
            tmem_st32(tO + cc * 32, orr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ph(t));
        if (valid >= C::COLS) softmax_p_bf16<HC, false>(sr_b, pk_b, c2, negm2, valid - HC, rs2);
        else softmax_p_bf16<HC, true>(sr_b, pk_b, c2, negm2, valid - HC, rs2);
#pragma unroll
        for (int i = 0; i < HC / 64; ++i) tmem_st32(tP + (HC / 64 + i) * 32, pk_b[i]);
      } else if constexpr (CHUNKED) {
        // chunk cc's 16 packed P columns go over S columns 16cc .. 16cc+15, which hold chunk 0 (already read)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          tmem_ld32(tS + cc * 32, sr[0]);
          tmem_wait_ld();
          reg_fence(sr[0]);
          const int vc = valid - cc * 32;
          uint32_t pk[32];
#pragma unroll
          for (int qc = 0; qc < 16; ++qc) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[0][2 * qc]), __uint_as_float(sr[0][2 * qc + 1])), c2,
                                      negm2);
            float x0, x1;
            f2_unpack_f(x, x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (2 * qc >= vc) p0 = 0.f;
            if (2 * qc + 1 >= vc) p1 = 0.f;
            rs2[qc & 1] = f2_add(rs2[qc & 1], f2_pack(p0, p1));  // the same accumulator order as one pass
            pk[qc] = pack_bf16x2(p0, p1);
          }
          tmem_st16_lo(tP + cc * 16, pk);
        }
      } else {
        uint32_t pk[C::PCOLS_W / 32][32];
        if (valid >= C::COLS) softmax_p_bf16<C::COLS, false>(sr, pk, c2, negm2, valid, rs2);
        else softmax_p_bf16<C::COLS, true>(sr, pk, c2, negm2, valid, rs2);
#pragma unroll
        for (int i = 0; i < C::PCOLS_W / 32; ++i) tmem_st32(tP + i * 32, pk[i]);
      }
      // correction of O_t: its last update (P V of step j-1) completed before S_t of step j did,
      // and P V of step j is not issued before every warpgroup of the tile arrives below
      // (with PV2 it was applied above, before the first half of P was handed over)
      if (!C::PV2 && j > 0 && __any_sync(0xffffffffu, need)) {
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int cc = 0; cc < C::OCOLS / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(tO + cc * 32, orr);
          tmem_wait_ld();
          reg_fence(orr);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t v = f2_mul(f2_pack(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2);
            f2_unpack(v, orr[e], orr[e + 1]);
          }
          tmem_st32(tO + cc * 32, orr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pf(t));
      float r0, r1, r2, r3;  // the row sum is not needed by the MMA: update it after the signal
      f2_unpack_f(rs2[0], r0, r1);
      f2_unpack_f(rs2[1], r2, r3);
      l = l * alpha + ((r0 + r1) + (r2 + r3));
    }
    // ---------------------------------------------------------- epilogue: O / l, LSE
    if (ok && Tt > 0) {
      bool okw = mbar_wait(bar_od(t), 0, abort_flag, p.err, W_OD);
      ok = __all_sync(0xffffffffu, okw);
    }
    if (C::KS && ks) {
      // Key-split CTA: slot 1 leaves its rows' (m, l) in shared memory; slot 0 merges the two partial
      // states (both O in this CTA's tensor memory, on the same lanes) in key order and writes O and the
      // LSE ("CS349E 第 11 讲 01_online_softmax.py", demo 2: partial states merge by rescaling to the
      // larger maximum).  Every thread of both warpgroups reaches the barrier.
      float2* ml1 = reinterpret_cast<float2*>(smem + C::OFF_ML);
      if (t == 1 && ok) ml1[row] = make_float2(m_ref, l);
      tc_fence_before();
      named_bar_sync(1, 2 * C::BR);
      const int qrow = q0 + row;
      const bool in_range = qrow < p.Nq;
      if (t == 0 && ok) {  // warp-uniform: the TMEM loads below are warp-collective; only stores are per row
        tc_fence_after();
        const float2 o1 = ml1[row];
        const float M = fmaxf(m_ref, o1.x);
        const float a0 = ex2_approx(m_ref - M), a1 = ex2_approx(o1.x - M);
        const float L = fmaf(o1.y, a1, l * a0);
        const float inv_l = 1.f / L;
        const float w0 = a0 * inv_l, w1 = a1 * inv_l;
        uint8_t* orow = static_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * p.Nq + qrow) * (C::D * C::ESZ);
        const uint32_t tO1 = tO + C::D;  // slot 1's O: the next D columns, same lanes
#pragma unroll
        for (int cc = 0; cc < C::OCOLS / 16; ++cc) {
          uint32_t r0[16], r1[16];
          tmem_ld16x(tO + cc * 16, r0);
          tmem_ld16x(tO1 + cc * 16, r1);
          tmem_wait_ld();
          reg_fence(r0);
          reg_fence(r1);
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_bf16x2(fmaf(__uint_as_float(r1[2 * e]), w1, __uint_as_float(r0[2 * e]) * w0),
                               fmaf(__uint_as_float(r1[2 * e + 1]), w1, __uint_as_float(r0[2 * e + 1]) * w0));
          if (in_range) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 16 * 2);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        if (p.lse != nullptr && in_range)
          p.lse[static_cast<size_t>(bh) * p.Nq + qrow] = (M + log2f(L)) * 0.6931471805599453f;
      }
    } else if (Tt == 0) {  // split mode, key range entirely above the tile's causal diagonal: empty state (-inf, 0, 0)
      const int qrow = q0 + t * trow + row;
      if (qrow < p.Nq) {
        const size_t srow = (static_cast<size_t>(split) * p.BH + bh) * p.Nq + qrow;
        float* wrow = p.ws_o + srow * C::D;
#pragma unroll
        for (int c4 = 0; c4 < C::OCOLS / 4; ++c4) reinterpret_cast<uint4*>(wrow)[c4] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<float2*>(p.ws_ml)[srow] = make_float2(-INFINITY, 0.f);
      }
    } else if (ok && p.n_split > 1) {  // partial state (m, l, unnormalised O) of this key range, for the merge
      tc_fence_after();
      const int qrow = q0 + t * trow + row;
      const bool in_range = qrow < p.Nq;
      const size_t srow = (static_cast<size_t>(split) * p.BH + bh) * p.Nq + qrow;
      float* wrow = p.ws_o + srow * C::D;
#pragma unroll
      for (int cc = 0; cc < C::OCOLS / 32; ++cc) {
        uint32_t orr[32];
        tmem_ld32(tO + cc * 32, orr);
        tmem_wait_ld();
        reg_fence(orr);
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(wrow + cc * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) dst[v4] = make_uint4(orr[4 * v4], orr[4 * v4 + 1], orr[4 * v4 + 2], orr[4 * v4 + 3]);
        }
      }
      if (in_range) reinterpret_cast<float2*>(p.ws_ml)[srow] = make_float2(m_ref, l);
    } else if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const int qrow = q0 + t * trow + row;
      const bool in_range = qrow < p.Nq;
      uint8_t* orow = static_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * p.Nq + qrow) * (C::D * C::ESZ);
#pragma unroll
      for (int cc = 0; cc < C::OCOLS / 32; ++cc) {
        uint32_t orr[32];
        tmem_ld32(tO + cc * 32, orr);
        tmem_wait_ld();
        reg_fence(orr);
        if (in_range) {
          if constexpr (C::TF32) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32 * 4);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              uint4 w;
              w.x = __float_as_uint(__uint_as_float(orr[4 * v4 + 0]) * inv_l);
              w.y = __float_as_uint(__uint_as_float(orr[4 * v4 + 1]) * inv_l);
              w.z = __float_as_uint(__uint_as_float(orr[4 * v4 + 2]) * inv_l);
              w.w = __float_as_uint(__uint_as_float(orr[4 * v4 + 3]) * inv_l);
              dst[v4] = w;
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32 * 2);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(orr[8 * v4 + 0]) * inv_l, __uint_as_float(orr[8 * v4 + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(orr[8 * v4 + 2]) * inv_l, __uint_as_float(orr[8 * v4 + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(orr[8 * v4 + 4]) * inv_l, __uint_as_float(orr[8 * v4 + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(orr[8 * v4 + 6]) * inv_l, __uint_as_float(orr[8 * v4 + 7]) * inv_l);
              dst[v4] = w;
            }
          }
        }
      }
      if (p.lse != nullptr && in_range)
        p.lse[static_cast<size_t>(bh) * p.Nq + qrow] = (m_ref + log2f(l)) * 0.6931471805599453f;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::LOAD_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <class C>
cudaError_t launch_fwd(const FwdLaunch& a) {
  // per device and cheap: set on every launch so any current device is covered
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.err = a.err;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.n_qblk = (a.Nq + C::BR * C::NQT - 1) / (C::BR * C::NQT);
  p.BH = a.BH;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.kv_per_split = a.kv_per_split;
  p.n_split = a.n_split;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.causal = a.causal;
  p.causal_off = a.Nk - a.Nq;
  if (a.causal && (a.Nq > a.Nk || a.n_split < 1)) return cudaErrorInvalidValue;
  p.c = a.c;
  p.tau = a.tau;
  p.p_lim = exp2f(a.tau);
  p.fault = a.fault;
  p.n_whole = 0;
  p.ks_tile0 = 0;
  p.ks_half = 0;
  if (a.ks_half > 0) {
    // key-split CTAs after ks_whole usual ones: the configuration must have them, no mask, one split, and
    // both key halves non-empty (the first a whole number of key tiles)
    const long long nq1 = (static_cast<long long>(a.Nq) + C::BR - 1) / C::BR;
    if (!C::KS || a.causal || a.n_split != 1 || a.ks_half % C::BC != 0 || a.ks_half >= a.Nk || a.ks_whole < 0 ||
        a.ks_tile0 < 0 || a.ks_count < 1 || static_cast<long long>(a.ks_tile0) + a.ks_count > nq1 * a.BH)
      return cudaErrorInvalidValue;
    p.n_whole = a.ks_whole;
    p.ks_tile0 = a.ks_tile0;
    p.ks_half = a.ks_half;
  }
  if (a.n_split < 1 || a.kv_per_split < C::BC || a.kv_per_split % C::BC != 0 ||
      static_cast<long long>(a.n_split - 1) * a.kv_per_split >= a.Nk)
    return cudaErrorInvalidValue;  // every split must own at least one key
  long long grid = static_cast<long long>(p.n_qblk) * a.BH * a.n_split;
  if (a.ks_half > 0) grid = static_cast<long long>(a.ks_whole) + a.ks_count;
  if (grid <= 0 || grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (a.dependent)
    return launch_dependent(fa_fwd_kernel<C>, static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, a.stream,
                            *a.tm_q, *a.tm_k, *a.tm_v, p);
  fa_fwd_kernel<C><<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, a.stream>>>(*a.tm_q, *a.tm_k,
                                                                                        *a.tm_v, p);
  return cudaGetLastError();
}

}  // namespace fa
