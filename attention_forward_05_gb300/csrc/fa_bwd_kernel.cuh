// fa_bwd_kernel.cuh -- FlashAttention backward for sm_103a (bf16 operands, fp32 accumulation).
//
// Sources (web pages, cited by title and section):
//   [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io), Exercise 5: the forward keeps
//        only O and the row statistics; the backward recomputes S_ij = Q_i K_j^T / sqrt(d) and
//        P_ij = exp(S_ij - m_i) / l_i block by block and accumulates dV_j += P_ij^T dO_i.
//   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com), demo 3 remarks: the backward needs a
//        single statistic per row, the logsumexp L = m + ln l, so that P_ij = exp(S_ij - L_i).
// The other gradients follow from the chain rule through the row softmax:
//   dP = dO V^T,  dS_ij = P_ij (dP_ij - D_i) with D_i = sum_c dO_ic O_ic,
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Three launches, no atomics (the result does not depend on scheduling):
//   fa_bwd_prep_kernel  -L_i log2(e) and -D_i for every query row (padded rows get -inf and 0),
//                       interleaved by row pairs: (nl_2i, nl_2i+1, -D_2i, -D_2i+1), so one 16-byte
//                       shared-memory load gives a column pair both values.
//   fa_bwd_dkdv_kernel  one CTA per (key/value head, 128-key tile); it walks every query tile of every
//                       query head that shares the key/value head, with S^T and dP^T computed key-major
//                       (keys on the TMEM lanes), so P^T and dS^T are the tensor-memory A operands of
//                       dV += P^T dO and dK += dS^T Q.  dV and dK stay in tensor memory throughout.
//                       A step's warpgroup writes P^T first (dV starts on it) and forms dS^T once dP^T
//                       has landed, while dV runs.
//   fa_bwd_dq_kernel    one CTA per two 128-row query tiles; it walks the key tiles, recomputes S and
//                       dP, and accumulates dQ += dS K with dS read from tensor memory.  dS goes over
//                       dP, so the next step's S is issued as soon as the warpgroup has read S (its
//                       exponentials then overlap dQ and the next dP).
// Both main kernels keep the forward's warp roles: one TMA warp, MMA-issuing warps, and warpgroups
// of thread-per-row elementwise work that take turns, so the tensor core computes the next products
// while a warpgroup works on the last ones.
#pragma once

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Non-blocking test of an mbarrier phase (no suspend); true when the phase with this parity completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Warp-collective load of 16 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Warp-collective store of 8 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

template <int NWARPS, int MINB>
struct RegBudget {  // registers per thread: 16384 per SM sub-partition, shared by ceil(warps/4) warps
  static constexpr int PER_SUB = (NWARPS * MINB + 3) / 4;
  static constexpr int RAW = (16384 / (PER_SUB * 32)) / 8 * 8;
  static constexpr int VALUE = RAW > 248 ? 248 : RAW;
};

// wait sites recorded with a timeout (distinct from the forward's)
enum : int { WB_KV = 0x21, WB_SF, WB_SE, WB_PF, WB_DONE, WB_Q, WB_KF, WB_VF, WB_KE, WB_VE, WB_OD, WB_DRAIN };

// ------------------------------------------------------------------------------------------ dK, dV

template <int D_, int BQ_, int STAGES_, int NSLOT_>
struct BwdKVCfg {
  static constexpr int D = D_;
  static constexpr int BK = 128;             // keys per CTA (TMEM lanes, M of every MMA)
  static constexpr int BQ = BQ_;             // query rows per step (N of S^T and dP^T, K of dV and dK)
  static constexpr int STAGES = STAGES_;     // ring of (Q_i, dO_i, row values)
  static constexpr int NSLOT = NSLOT_;       // TMEM slots for (S^T, dP^T); one elementwise warpgroup each
  static constexpr int CHUNK = 64;           // bf16 elements per 128-byte swizzled row segment
  static constexpr int NCH = D / CHUNK;
  static constexpr int MMA_K = 16;
  static constexpr int KV_CH_BYTES = BK * 128;
  static constexpr int KV_BYTES = NCH * KV_CH_BYTES;
  static constexpr int QS_CH_BYTES = BQ * 128;
  static constexpr int QS_BYTES = NCH * QS_CH_BYTES;
  static constexpr int VEC_BYTES = BQ * 8;   // (-L log2 e, -D) of the step's rows, interleaved by pairs
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;              // stage s at + s * QS_BYTES
  static constexpr int OFF_DO = OFF_Q + STAGES * QS_BYTES;
  static constexpr int OFF_VEC = OFF_DO + STAGES * QS_BYTES;  // stage s at + s * VEC_BYTES
  static constexpr int OFF_BAR = OFF_VEC + STAGES * VEC_BYTES;
  // barriers: kv_full, st_full[S], st_empty[S], s_full[NSLOT] (S^T complete), ds_full[NSLOT] (dS^T
  // written), g_free[NSLOT], done, drain (score issuer), drain (gradient issuer), dp_full[NSLOT] (dP^T
  // complete), pt_full[NSLOT] (P^T written)
  static constexpr int NBAR = 1 + 2 * STAGES + 5 * NSLOT + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  // TMEM: slot b holds S^T at b*2*BQ and dP^T at b*2*BQ + BQ; P^T and dS^T (bf16 pairs) are written
  // over the first BQ/2 columns of each.  dV and dK accumulate after the slots.
  static constexpr int COL_DV = NSLOT * 2 * BQ;
  static constexpr int COL_DK = COL_DV + D;
  static constexpr int TMEM_NEED = NSLOT * 2 * BQ + 2 * D;
  static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  // Two MMA-issuing warps on different SM sub-partitions: one thread issues each tcgen05.mma in
  // about 44 cycles, longer than an M=128, N=64 product takes, so one issuer cannot keep the tensor
  // core busy with these shapes and two can.
  static constexpr int NWARPS = 4 * NSLOT + 3;
  static constexpr int NTHREADS = NWARPS * 32;
  static constexpr int LOAD_WARP = 4 * NSLOT;
  static constexpr int MMA_WARP = 4 * NSLOT + 1;   // S^T, dP^T
  static constexpr int GRAD_WARP = 4 * NSLOT + 2;  // dV, dK
  static constexpr int MAXREG = RegBudget<NWARPS, 1>::VALUE;
  static_assert(D % CHUNK == 0 && BQ % 32 == 0 && BQ <= 128, "tile");
  static_assert(NSLOT >= 2 && STAGES >= NSLOT, "the ring must hold the steps in flight");
  static_assert(TMEM_NEED <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(QS_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

struct BwdKVParams {
  void* dk;              // [B, Hkv, Nk, D] bf16
  void* dv;
  const float* rowv;     // [B*H][Nq_pad/2][4]: (-L log2 e, -D) of row pairs; padded rows -inf and 0
  int* err;
  int Nq, Nk, Nq_pad, n_kblk, n_qt;
  int H, Hkv;
  int causal, causal_off;  // query row i sees keys j <= i + causal_off
  float c;                 // scale * log2(e)
  float scale;
  int fault;               // test only: 1 = the load warp skips the K/V copy (the waits for it run out)
};

// First part of a dK/dV elementwise step (thread = key row, BQ query columns): P^T = 2^(s c - L log2 e)
// into registers (f32 pairs) and, as bf16 pairs, over the first BQ/2 columns of S^T, the A operand of
// dV += P^T dO.  rv holds the step's (-L log2 e, -D) by column pairs.  MASK: columns q < qmin are above
// the causal diagonal (P = 0).
template <class C, bool MASK>
__device__ __forceinline__ void dkdv_p_first(uint32_t tS, const float4* rv, uint64_t c2, int qmin,
                                             uint64_t (&pp)[C::BQ / 2]) {
  constexpr int NCHK = C::BQ / 16;
  uint32_t sr[NCHK][16];
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) tmem_ld16(tS + cc * 16, sr[cc]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) reg_fence(sr[cc]);
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) {
    uint32_t pk_p[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int q = cc * 16 + e;
      const float4 vv = rv[q / 2];
      const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1])), c2,
                                f2_pack(vv.x, vv.y));
      float x0, x1;
      f2_unpack_f(x, x0, x1);
      float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if (MASK) {
        if (q < qmin) p0 = 0.f;
        if (q + 1 < qmin) p1 = 0.f;
      }
      pp[q / 2] = f2_pack(p0, p1);
      pk_p[e / 2] = pack_bf16x2(p0, p1);
    }
    tmem_st8(tS + cc * 8, pk_p);
  }
}

// Second part: dS^T = P^T (dP^T - D) from the f32 P^T, as bf16 pairs over the first BQ/2 columns of dP^T,
// the A operand of dK += dS^T Q (16-column chunks with the next chunk's TMEM load in flight; chunk cc's
// 8 packed columns go over columns already read).
template <class C>
__device__ __forceinline__ void dkdv_ds_second(uint32_t tdP, const float4* rv, const uint64_t (&pp)[C::BQ / 2]) {
  constexpr int NCHK = C::BQ / 16;
  uint32_t dr[2][16];
  tmem_ld16(tdP, dr[0]);
  tmem_wait_ld();
  reg_fence(dr[0]);
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) {
    if (cc + 1 < NCHK) tmem_ld16(tdP + (cc + 1) * 16, dr[(cc + 1) & 1]);
    const uint32_t(&d16)[16] = dr[cc & 1];
    uint32_t pk_ds[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int q = cc * 16 + e;
      const float4 vv = rv[q / 2];
      const uint64_t t = f2_add(f2_pack(__uint_as_float(d16[e]), __uint_as_float(d16[e + 1])), f2_pack(vv.z, vv.w));
      const uint64_t ds = f2_mul(pp[q / 2], t);
      float ds0, ds1;
      f2_unpack_f(ds, ds0, ds1);
      pk_ds[e / 2] = pack_bf16x2(ds0, ds1);
    }
    tmem_st8(tdP + cc * 8, pk_ds);
    if (cc + 1 < NCHK) {
      tmem_wait_ld();
      reg_fence(dr[(cc + 1) & 1]);
    }
  }
}

template <class C>
__global__ void __maxnreg__(C::MAXREG)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const BwdKVParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // With a causal mask a key tile sees fewer query rows the later it lies, so the key tile is the
  // slowest grid index, low tiles first: the longest CTAs of every head start in the first wave.
  // Without a mask the key tiles of one head are adjacent.
  const int n_kvbh = static_cast<int>(gridDim.x) / p.n_kblk;
  const int kb = p.causal ? static_cast<int>(blockIdx.x) / n_kvbh : static_cast<int>(blockIdx.x % p.n_kblk);
  const int kvbh = p.causal ? static_cast<int>(blockIdx.x) % n_kvbh : static_cast<int>(blockIdx.x / p.n_kblk);
  const int b = kvbh / p.Hkv;
  const int g = kvbh % p.Hkv;
  const int G = p.H / p.Hkv;  // query heads per key/value head
  const int k0 = kb * C::BK;
  // query tiles that see at least one key of the tile: rows i >= k0 - causal_off
  const int i_lo = p.causal ? max(0, k0 - p.causal_off) / C::BQ : 0;
  const int per_head = p.n_qt - i_lo;
  const int T = G * per_head;  // steps: (query head, query tile) pairs, >= 1

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t bar_kv = bar0;
  auto bar_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bar0 + 8u * (1 + C::STAGES + s); };
  auto bar_sf = [&](int w) { return bar0 + 8u * (1 + 2 * C::STAGES + w); };
  auto bar_dsf = [&](int w) { return bar0 + 8u * (1 + 2 * C::STAGES + C::NSLOT + w); };  // dS^T written
  auto bar_gf = [&](int w) { return bar0 + 8u * (1 + 2 * C::STAGES + 2 * C::NSLOT + w); };
  const uint32_t bar_done = bar0 + 8u * (1 + 2 * C::STAGES + 3 * C::NSLOT);
  const uint32_t bar_drain = bar_done + 8u;
  const uint32_t bar_drain_g = bar_done + 16u;
  auto bar_dpf = [&](int w) { return bar_done + 24u + 8u * w; };                // dP^T complete
  auto bar_ptf = [&](int w) { return bar_done + 24u + 8u * (C::NSLOT + w); };  // P^T written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int w = 0; w < C::NSLOT; ++w) {
      mbar_init(bar_sf(w), 1);
      mbar_init(bar_dsf(w), 4);  // one arrive per warp of the warpgroup
      mbar_init(bar_gf(w), 1);
      mbar_init(bar_dpf(w), 1);
      mbar_init(bar_ptf(w), 4);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain_g, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the prep kernel: the set-up above overlaps its tail, and
  // the row values it writes are read only after this wait.  Then the dQ kernel launched after this
  // one (it reads nothing this kernel writes) may take the SMs this grid's last wave leaves idle.
  griddep_wait();
  griddep_launch_dependents();

  auto step_head = [&](int s) { return b * p.H + g * G + s / per_head; };  // query (batch, head) index
  auto step_qt = [&](int s) { return i_lo + s % per_head; };               // query tile

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int n_done = 0;
      if (p.fault != 1) {
        mbar_expect_tx(bar_kv, 2 * C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sbase + C::OFF_K + c * C::KV_CH_BYTES, &tm_k, bar_kv, c * C::CHUNK, k0, kvbh);
          tma_load_3d(sbase + C::OFF_V + c * C::KV_CH_BYTES, &tm_v, bar_kv, c * C::CHUNK, k0, kvbh);
        }
      }
      for (int s = 0; s < T; ++s) {
        const int st = s % C::STAGES;
        if (!mbar_wait(bar_empty(st), ((s / C::STAGES) & 1) ^ 1, abort_flag, p.err, WB_SE)) break;
        const int bh = step_head(s);
        const int q0 = step_qt(s) * C::BQ;
        mbar_expect_tx(bar_full(st), 2 * C::QS_BYTES + C::VEC_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sbase + C::OFF_Q + st * C::QS_BYTES + c * C::QS_CH_BYTES, &tm_q, bar_full(st), c * C::CHUNK,
                      q0, bh);
          tma_load_3d(sbase + C::OFF_DO + st * C::QS_BYTES + c * C::QS_CH_BYTES, &tm_do, bar_full(st),
                      c * C::CHUNK, q0, bh);
        }
        // rows q0 .. q0 + BQ - 1 of the interleaved row values: 2 floats per row
        bulk_load_1d(sbase + C::OFF_VEC + st * C::VEC_BYTES, p.rowv + (static_cast<size_t>(bh) * p.Nq_pad + q0) * 2,
                     C::VEC_BYTES, bar_full(st));
        n_done = s + 1;
      }
      // drain every copy issued above before the CTA exits
      if (p.fault != 1) mbar_wait_drain(bar_kv, 0, p.err, WB_DRAIN);
#pragma unroll
      for (int st = 0; st < C::STAGES; ++st) {
        const int cnt = n_done > st ? (n_done - 1 - st) / C::STAGES + 1 : 0;
        if (cnt > 0) mbar_wait_drain(bar_full(st), (cnt - 1) & 1, p.err, WB_DRAIN);
      }
    }
  } else if (warp == C::MMA_WARP || warp == C::GRAD_WARP) {
    // ------------------------------------------------------------ MMA issuers (whole warp, elected issue)
    // A phase that already completed is seen by one non-blocking test; only otherwise does the warp
    // enter the bounded wait.
    auto wait_all = [&](uint32_t bar, uint32_t parity, int where) {
      if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err, where)) != 0;
    };
    auto commit = [&](uint32_t bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    bool ok = wait_all(bar_kv, 0, WB_KV);
    if (warp == C::MMA_WARP) {
      // S^T = K Q^T and dP^T = V dO^T of step s into slot s % NSLOT, as soon as the step's tiles have
      // landed and the gradient MMAs of step s - NSLOT (the slot's previous user) have completed.
      constexpr uint32_t idesc_s = make_idesc(1, C::BK, C::BQ, 0, 0);
      const uint64_t dk0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      const uint64_t dqk0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);    // Q as K-major B
      const uint64_t ddok0 = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);  // dO as K-major B
      for (int s = 0; ok && s < T; ++s) {
        ok = wait_all(bar_full(s % C::STAGES), (s / C::STAGES) & 1, WB_SF);
        if (ok && s >= C::NSLOT) ok = wait_all(bar_gf(s % C::NSLOT), ((s / C::NSLOT) - 1) & 1, WB_PF);
        if (!ok) break;
        tc_fence_after();
        const int st = s % C::STAGES;
        const uint32_t col = (s % C::NSLOT) * 2 * C::BQ;
        const uint64_t so = static_cast<uint64_t>((st * C::QS_BYTES) >> 4);
        if (elect_one()) {  // one lane issues the whole batch
#pragma unroll
          for (int kk = 0; kk < C::D / C::MMA_K; ++kk) {
            const int e = kk * C::MMA_K;
            const uint32_t oa = ((e / C::CHUNK) * C::KV_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
            const uint32_t ob = ((e / C::CHUNK) * C::QS_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
            mma_ss<0>(tmem + col, dk0 + oa, dqk0 + so + ob, idesc_s, kk > 0);
          }
          mma_commit(bar_sf(s % C::NSLOT));  // S^T alone: the exponentials may start
#pragma unroll
          for (int kk = 0; kk < C::D / C::MMA_K; ++kk) {
            const int e = kk * C::MMA_K;
            const uint32_t oa = ((e / C::CHUNK) * C::KV_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
            const uint32_t ob = ((e / C::CHUNK) * C::QS_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
            mma_ss<0>(tmem + col + C::BQ, dv0 + oa, ddok0 + so + ob, idesc_s, kk > 0);
          }
          mma_commit(bar_dpf(s % C::NSLOT));
        }
        __syncwarp();
      }
      commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, p.err, WB_DRAIN);
    } else {
      // dV += P^T dO of step s as soon as its warpgroup has written P^T, dK += dS^T Q once it has written
      // dS^T (the warpgroup forms dS^T while dV runs).
      constexpr uint32_t idesc_g = make_idesc(1, C::BK, C::D, 0, 1);   // B MN-major
      const uint64_t dqm0 = sdesc_sw128(sbase + C::OFF_Q, C::QS_CH_BYTES, 1024);   // Q as MN-major B
      const uint64_t ddom0 = sdesc_sw128(sbase + C::OFF_DO, C::QS_CH_BYTES, 1024); // dO as MN-major B
      for (int s = 0; ok && s < T; ++s) {
        const int st = s % C::STAGES;
        const uint32_t col = (s % C::NSLOT) * 2 * C::BQ;
        const uint64_t so = static_cast<uint64_t>((st * C::QS_BYTES) >> 4);
        ok = wait_all(bar_full(st), (s / C::STAGES) & 1, WB_SF);  // complete already
        ok = ok && wait_all(bar_ptf(s % C::NSLOT), (s / C::NSLOT) & 1, WB_PF);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::BQ / C::MMA_K; ++kk) {
            const uint32_t ob = (kk * C::MMA_K * 128) >> 4;  // 16 query rows = two 8-row swizzle atoms
            mma_ts<0>(tmem + C::COL_DV, tmem + col + kk * (C::MMA_K / 2), ddom0 + so + ob, idesc_g,
                      (s > 0 || kk > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
        ok = wait_all(bar_dsf(s % C::NSLOT), (s / C::NSLOT) & 1, WB_PF);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::BQ / C::MMA_K; ++kk) {
            const uint32_t ob = (kk * C::MMA_K * 128) >> 4;
            mma_ts<0>(tmem + C::COL_DK, tmem + col + C::BQ + kk * (C::MMA_K / 2), dqm0 + so + ob, idesc_g,
                      (s > 0 || kk > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
        commit(bar_gf(s % C::NSLOT));       // the slot may be overwritten
        commit(bar_empty(s % C::STAGES));   // the stage may be refilled (its score MMAs completed earlier)
      }
      if (ok) commit(bar_done);
      commit(bar_drain_g);
      mbar_wait_drain(bar_drain_g, 0, p.err, WB_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    // Warpgroup w handles the steps s with s % NSLOT == w; thread = key row (TMEM lane).
    const int w = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int key = k0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + w * 2 * C::BQ;
    const uint32_t tdP = tS + C::BQ;
    const uint64_t c2 = f2_pack(p.c, p.c);
    bool ok = true;
    for (int s = w; s < T; s += C::NSLOT) {
      const int st = s % C::STAGES;
      bool okw = mbar_wait(bar_sf(w), (s / C::NSLOT) & 1, abort_flag, p.err, WB_SF);
      // the stage's row values came by TMA: observe its completion (already complete) before reading
      okw = okw && mbar_wait(bar_full(st), (s / C::STAGES) & 1, abort_flag, p.err, WB_SF);
      ok = __all_sync(0xffffffffu, okw);
      if (!ok) break;
      tc_fence_after();
      const float4* rv = reinterpret_cast<const float4*>(smem + C::OFF_VEC + st * C::VEC_BYTES);
      // causal: query column q (row step_qt(s)*BQ + q) is visible to this key when q >= qmin
      const int qmin = p.causal ? key - p.causal_off - step_qt(s) * C::BQ : 0;
      uint64_t pp[C::BQ / 2];
      if (__any_sync(0xffffffffu, qmin > 0))
        dkdv_p_first<C, true>(tS, rv, c2, qmin, pp);
      else
        dkdv_p_first<C, false>(tS, rv, c2, qmin, pp);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ptf(w));  // dV += P^T dO may start
      okw = mbar_wait(bar_dpf(w), (s / C::NSLOT) & 1, abort_flag, p.err, WB_SF);
      ok = __all_sync(0xffffffffu, okw);
      if (!ok) break;
      tc_fence_after();
      dkdv_ds_second<C>(tdP, rv, pp);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dsf(w));
    }
    // ---------------------------------------------------------- epilogue: warpgroup 0 writes dV, 1 writes dK
    bool okd = ok && w < 2 && mbar_wait(bar_done, 0, abort_flag, p.err, WB_DONE);
    okd = __all_sync(0xffffffffu, okd);
    if (okd) {
      tc_fence_after();
      const float mul = w == 0 ? 1.f : p.scale;
      const uint32_t tacc = tmem + lane_base + (w == 0 ? C::COL_DV : C::COL_DK);
      uint8_t* out = static_cast<uint8_t*>(w == 0 ? p.dv : p.dk) +
                     (static_cast<size_t>(kvbh) * p.Nk + key) * (C::D * 2);
      const bool in_range = key < p.Nk;
#pragma unroll
      for (int cc = 0; cc < C::D / 32; ++cc) {
        uint32_t a[32];
        tmem_ld32(tacc + cc * 32, a);
        tmem_wait_ld();
        reg_fence(a);
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(out + cc * 64);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 wv;
            wv.x = pack_bf16x2(__uint_as_float(a[8 * v4 + 0]) * mul, __uint_as_float(a[8 * v4 + 1]) * mul);
            wv.y = pack_bf16x2(__uint_as_float(a[8 * v4 + 2]) * mul, __uint_as_float(a[8 * v4 + 3]) * mul);
            wv.z = pack_bf16x2(__uint_as_float(a[8 * v4 + 4]) * mul, __uint_as_float(a[8 * v4 + 5]) * mul);
            wv.w = pack_bf16x2(__uint_as_float(a[8 * v4 + 6]) * mul, __uint_as_float(a[8 * v4 + 7]) * mul);
            dst[v4] = wv;
          }
        }
      }
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

// ------------------------------------------------------------------------------------------ dQ

template <int D_, int BC_, int STAGES_, bool ATMEM_>
struct BwdQCfg {
  static constexpr int D = D_;
  static constexpr int BR = 128;           // query rows per tile (TMEM lanes)
  static constexpr int NQT = 2;            // query tiles per CTA, alternating between the two warpgroups
  static constexpr int BC = BC_;           // keys per step
  static constexpr int STAGES = STAGES_;   // ring of (K_j, V_j)
  // ATMEM: the elementwise warpgroups copy Q_t and dO_t into tensor memory once, and S and dP take
  // them as the A operand there: each MMA then reads only K or V from shared memory (an N = 64 MMA
  // reading both operands from shared memory is bound by its bandwidth).
  static constexpr bool ATMEM = ATMEM_;
  static constexpr int CHUNK = 64;
  static constexpr int NCH = D / CHUNK;
  static constexpr int MMA_K = 16;
  static constexpr int Q_CH_BYTES = BR * 128;
  static constexpr int Q_BYTES = NCH * Q_CH_BYTES;
  static constexpr int KV_CH_BYTES = BC * 128;
  static constexpr int KV_BYTES = NCH * KV_CH_BYTES;
  static constexpr int OFF_Q = 0;                              // tile t at + t * Q_BYTES
  static constexpr int OFF_DO = OFF_Q + NQT * Q_BYTES;
  static constexpr int OFF_K = OFF_DO + NQT * Q_BYTES;         // stage s at + s * KV_BYTES
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // barriers: q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[NQT], ds_full[NQT],
  // o_done[NQT], drain (S issuer), drain (dP, dQ issuer), a_in_tmem[NQT], s_read[NQT] (the warpgroup has
  // read S), dp_full[NQT]
  static constexpr int NBAR = 1 + 4 * STAGES + 6 * NQT + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  // TMEM: tile t holds S at t*2*BC and dP at t*2*BC + BC (dS, bf16 pairs, over the first BC/2 columns
  // of dP), dQ at 2*NQT*BC + t*D; with ATMEM, Q_t and dO_t as bf16 pairs (D/2 columns each) after them.
  static constexpr int COL_DQ = 2 * NQT * BC;
  static constexpr int COL_QA = COL_DQ + NQT * D;
  static constexpr int COL_DOA = COL_QA + NQT * (D / 2);
  static constexpr int TMEM_NEED = 2 * NQT * BC + NQT * D + (ATMEM ? NQT * D : 0);
  static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int NWARPS = 4 * NQT + 3;
  static constexpr int NTHREADS = NWARPS * 32;
  static constexpr int LOAD_WARP = 4 * NQT;
  static constexpr int MMA_WARP = 4 * NQT + 1;   // S (two issuing warps, as in the dK/dV kernel)
  static constexpr int GRAD_WARP = 4 * NQT + 2;  // dQ, then the next step's dP
  static constexpr int MAXREG = RegBudget<NWARPS, 1>::VALUE;
  static_assert(D % CHUNK == 0 && BC % 64 == 0 && BC <= 128, "tile");
  static_assert(!ATMEM || NCH == 1, "A operands copied into tensor memory from one 128-byte row segment");
  static_assert(TMEM_NEED <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct BwdQParams {
  void* dq;              // [B, H, Nq, D] bf16
  const float* rowv;     // [B*H][Nq_pad/2][4]: (-L log2 e, -D) of row pairs
  int* err;
  int Nq, Nk, Nq_pad, n_qblk;
  int H, Hkv;
  int causal, causal_off;
  float c, scale;
};

// First part of a dQ elementwise step (thread = query row, BC key columns): P = 2^(s c - L log2 e) from S
// into registers as f32 pairs.  TAIL: columns >= valid are masked (P = 0).  Every TMEM load has completed
// on return, so the S issuer may overwrite S with the next step's.
template <class C, bool TAIL>
__device__ __forceinline__ void dq_p_regs(uint32_t tS, uint64_t c2, uint64_t nl_2, int valid,
                                          uint64_t (&pp)[C::BC / 2]) {
  constexpr int NCHK = C::BC / 16;
  uint32_t sr[NCHK][16];
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) tmem_ld16(tS + cc * 16, sr[cc]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) reg_fence(sr[cc]);
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc)
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int col = cc * 16 + e;
      const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1])), c2, nl_2);
      float x0, x1;
      f2_unpack_f(x, x0, x1);
      float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if (TAIL) {
        if (col >= valid) p0 = 0.f;
        if (col + 1 >= valid) p1 = 0.f;
      }
      pp[col / 2] = f2_pack(p0, p1);
    }
}

// Second part: dS = P (dP - D), written as bf16 pairs over the first BC/2 columns of dP, the A operand of
// dQ += dS K (16-column chunks with the next chunk's TMEM load in flight; chunk cc's 8 packed columns go
// over dP columns 8 cc .. 8 cc + 7, all read already).
template <class C>
__device__ __forceinline__ void dq_ds_regs(uint32_t tdP, uint64_t nd_2, const uint64_t (&pp)[C::BC / 2]) {
  constexpr int NCHK = C::BC / 16;
  uint32_t dr[2][16];
  tmem_ld16(tdP, dr[0]);
  tmem_wait_ld();
  reg_fence(dr[0]);
#pragma unroll
  for (int cc = 0; cc < NCHK; ++cc) {
    if (cc + 1 < NCHK) tmem_ld16(tdP + (cc + 1) * 16, dr[(cc + 1) & 1]);
    const uint32_t(&d16)[16] = dr[cc & 1];
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const uint64_t tt = f2_add(f2_pack(__uint_as_float(d16[e]), __uint_as_float(d16[e + 1])), nd_2);
      const uint64_t ds = f2_mul(pp[(cc * 16 + e) / 2], tt);
      float ds0, ds1;
      f2_unpack_f(ds, ds0, ds1);
      pk[e / 2] = pack_bf16x2(ds0, ds1);
    }
    tmem_st8(tdP + cc * 8, pk);
    if (cc + 1 < NCHK) {
      tmem_wait_ld();
      reg_fence(dr[(cc + 1) & 1]);
    }
  }
}

template <class C>
__global__ void __maxnreg__(C::MAXREG)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const BwdQParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // With a causal mask the query block is the slowest grid index, last block first, so the longest
  // CTAs of every head start in the first wave; without a mask the blocks of one head are adjacent.
  const int n_bh = static_cast<int>(gridDim.x) / p.n_qblk;
  const int qb = p.causal ? p.n_qblk - 1 - static_cast<int>(blockIdx.x) / n_bh : static_cast<int>(blockIdx.x % p.n_qblk);
  const int bh = p.causal ? static_cast<int>(blockIdx.x) % n_bh : static_cast<int>(blockIdx.x / p.n_qblk);
  const int kvh = (bh / p.H) * p.Hkv + (bh % p.H) / (p.H / p.Hkv);
  const int q0 = qb * C::BR * C::NQT;
  const int k_hi = p.causal ? min(p.Nk, q0 + C::NQT * C::BR + p.causal_off) : p.Nk;
  const int T = (k_hi + C::BC - 1) / C::BC;  // >= 1: every row sees at least one key

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
  const uint32_t bar_drain_g = bar_drain + 8u;
  auto bar_qa = [&](int t) { return bar_drain + 16u + 8u * t; };                 // Q_t, dO_t in TMEM (ATMEM)
  auto bar_sr = [&](int t) { return bar_drain + 16u + 8u * (C::NQT + t); };      // S_t read
  auto bar_dpf = [&](int t) { return bar_drain + 16u + 8u * (2 * C::NQT + t); };  // dP_t complete
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
      mbar_init(bar_pf(t), 4);
      mbar_init(bar_od(t), 1);
      mbar_init(bar_qa(t), 4);
      mbar_init(bar_sr(t), 4);
      mbar_init(bar_dpf(t), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain_g, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int nk_done = 0, nv_done = 0;
      mbar_expect_tx(bar_q, 2 * C::NQT * C::Q_BYTES);
#pragma unroll
      for (int t = 0; t < C::NQT; ++t)
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sbase + C::OFF_Q + t * C::Q_BYTES + c * C::Q_CH_BYTES, &tm_q, bar_q, c * C::CHUNK,
                      q0 + t * C::BR, bh);
          tma_load_3d(sbase + C::OFF_DO + t * C::Q_BYTES + c * C::Q_CH_BYTES, &tm_do, bar_q, c * C::CHUNK,
                      q0 + t * C::BR, bh);
        }
      for (int j = 0; j < T; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = ((j / C::STAGES) & 1) ^ 1;
        if (!mbar_wait(bar_ke(s), ph, abort_flag, p.err, WB_KE)) break;
        mbar_expect_tx(bar_kf(s), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sbase + C::OFF_K + s * C::KV_BYTES + c * C::KV_CH_BYTES, &tm_k, bar_kf(s), c * C::CHUNK,
                      j * C::BC, kvh);
        nk_done = j + 1;
        if (!mbar_wait(bar_ve(s), ph, abort_flag, p.err, WB_VE)) break;
        mbar_expect_tx(bar_vf(s), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sbase + C::OFF_V + s * C::KV_BYTES + c * C::KV_CH_BYTES, &tm_v, bar_vf(s), c * C::CHUNK,
                      j * C::BC, kvh);
        nv_done = j + 1;
      }
      mbar_wait_drain(bar_q, 0, p.err, WB_DRAIN);
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) {
        const int nks = nk_done > s ? (nk_done - 1 - s) / C::STAGES + 1 : 0;
        const int nvs = nv_done > s ? (nv_done - 1 - s) / C::STAGES + 1 : 0;
        if (nks > 0) mbar_wait_drain(bar_kf(s), (nks - 1) & 1, p.err, WB_DRAIN);
        if (nvs > 0) mbar_wait_drain(bar_vf(s), (nvs - 1) & 1, p.err, WB_DRAIN);
      }
    }
  } else if (warp == C::MMA_WARP || warp == C::GRAD_WARP) {
    // ------------------------------------------------------------ MMA issuers (whole warp, elected issue)
    auto wait_all = [&](uint32_t bar, uint32_t parity, int where) {
      if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err, where)) != 0;
    };
    auto commit = [&](uint32_t bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    // S_t(j) = Q_t K_j^T and dP_t(j) = dO_t V_j^T (stage s), issued by the elected lane of the caller
    constexpr uint32_t idesc_s = make_idesc(1, C::BR, C::BC, 0, 0);
    const uint64_t dq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
    const uint64_t ddo0 = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
    const uint64_t dk0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
    const uint64_t dv0 = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
    auto issue_s = [&](int t, int s) {
      const uint32_t col = t * 2 * C::BC;
      const uint64_t to = static_cast<uint64_t>((t * C::Q_BYTES) >> 4);
      const uint64_t so = static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::D / C::MMA_K; ++kk) {
        const int e = kk * C::MMA_K;
        const uint32_t oa = ((e / C::CHUNK) * C::Q_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
        const uint32_t ob = ((e / C::CHUNK) * C::KV_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
        if constexpr (C::ATMEM)
          mma_ts<0>(tmem + col, tmem + C::COL_QA + t * (C::D / 2) + kk * (C::MMA_K / 2), dk0 + so + ob, idesc_s,
                    kk > 0);
        else
          mma_ss<0>(tmem + col, dq0 + to + oa, dk0 + so + ob, idesc_s, kk > 0);
      }
    };
    auto issue_dp = [&](int t, int s) {
      const uint32_t col = t * 2 * C::BC + C::BC;
      const uint64_t to = static_cast<uint64_t>((t * C::Q_BYTES) >> 4);
      const uint64_t so = static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::D / C::MMA_K; ++kk) {
        const int e = kk * C::MMA_K;
        const uint32_t oa = ((e / C::CHUNK) * C::Q_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
        const uint32_t ob = ((e / C::CHUNK) * C::KV_CH_BYTES + (e % C::CHUNK) * 2) >> 4;
        if constexpr (C::ATMEM)
          mma_ts<0>(tmem + col, tmem + C::COL_DOA + t * (C::D / 2) + kk * (C::MMA_K / 2), dv0 + so + ob, idesc_s,
                    kk > 0);
        else
          mma_ss<0>(tmem + col, ddo0 + to + oa, dv0 + so + ob, idesc_s, kk > 0);
      }
    };
    // dQ_t += dS_t K_j, dS_t read from tensor memory
    constexpr uint32_t idesc_g = make_idesc(1, C::BR, C::D, 0, 1);  // K MN-major
    const uint64_t dkm0 = sdesc_sw128(sbase + C::OFF_K, C::KV_CH_BYTES, 1024);
    auto issue_dq = [&](int t, int s, int j) {
      const uint32_t a_tmem = tmem + t * 2 * C::BC + C::BC;  // dS over dP
      const uint64_t so = static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::BC / C::MMA_K; ++kk) {
        const uint32_t ob = (kk * C::MMA_K * 128) >> 4;
        mma_ts<0>(tmem + C::COL_DQ + t * C::D, a_tmem + kk * (C::MMA_K / 2), dkm0 + so + ob, idesc_g,
                  (j > 0 || kk > 0) ? 1u : 0u);
      }
    };
    if (warp == C::MMA_WARP) {
      bool ok = wait_all(bar_q, 0, WB_Q);
      if constexpr (C::ATMEM) {
#pragma unroll
        for (int t = 0; t < C::NQT; ++t) ok = ok && wait_all(bar_qa(t), 0, WB_Q);
      }
      // S_t(j) once K_j has landed and the warpgroup has read S_t(j-1) (it keeps P in registers)
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % C::STAGES;
        ok = wait_all(bar_kf(s), (j / C::STAGES) & 1, WB_KF);
        for (int t = 0; ok && t < C::NQT; ++t) {
          if (j > 0) ok = wait_all(bar_sr(t), (j - 1) & 1, WB_SE);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) issue_s(t, s);
          __syncwarp();
          commit(bar_sf(t));
        }
      }
      commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, p.err, WB_DRAIN);
    } else {
      // dQ_t(j) once the warpgroup has written dS_t(j) (over dP_t), then, from the same lane, dP_t(j+1)
      // into the columns dQ_t(j) reads as its A operand.  No barrier separates the two: this relies on the
      // tensor core running the MMAs one thread issues in issue order (the PTX ISA states that order for
      // MMAs into the same accumulator; these two write different ones), as the forward kernel's P V and
      // next Q K^T over the aliased S / P columns do.
      bool ok = wait_all(bar_q, 0, WB_Q);
      if constexpr (C::ATMEM) {
#pragma unroll
        for (int t = 0; t < C::NQT; ++t) ok = ok && wait_all(bar_qa(t), 0, WB_Q);
      }
      ok = ok && wait_all(bar_vf(0), 0, WB_VF);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int t = 0; t < C::NQT; ++t) {
            issue_dp(t, 0);
            mma_commit(bar_dpf(t));
          }
          mma_commit(bar_ve(0));  // V_0 is read by dP only
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % C::STAGES;
        const bool nxt = j + 1 < T;
        const int s1 = (j + 1) % C::STAGES;
        ok = wait_all(bar_kf(s), (j / C::STAGES) & 1, WB_KF);  // complete already: K_j was read by S
        if (ok && nxt) ok = wait_all(bar_vf(s1), ((j + 1) / C::STAGES) & 1, WB_VF);
        for (int t = 0; ok && t < C::NQT; ++t) {
          ok = wait_all(bar_pf(t), j & 1, WB_PF);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            issue_dq(t, s, j);
            if (nxt) {
              issue_dp(t, s1);
              mma_commit(bar_dpf(t));
            } else {
              mma_commit(bar_od(t));
            }
          }
          __syncwarp();
        }
        // K_j is read by S (complete before its dS existed) and by dQ; V_{j+1} by dP
        if (ok) {
          commit(bar_ke(s));
          if (nxt) commit(bar_ve(s1));
        }
      }
      commit(bar_drain_g);
      mbar_wait_drain(bar_drain_g, 0, p.err, WB_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups: thread = query row
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int qrow = q0 + t * C::BR + row;
    const bool in_range = qrow < p.Nq;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 2 * C::BC;
    const uint32_t tdP = tS + C::BC;
    const size_t vpair = (static_cast<size_t>(bh) * p.Nq_pad + (qrow & ~1)) * 2;  // float index of the row pair
    const float nl = in_range ? p.rowv[vpair + (qrow & 1)] : -INFINITY;
    const float ndd = in_range ? p.rowv[vpair + 2 + (qrow & 1)] : 0.f;  // -D
    const int row_lim = p.causal ? min(p.Nk, qrow + 1 + p.causal_off) : p.Nk;  // keys [0, row_lim) visible
    const uint64_t c2 = f2_pack(p.c, p.c);
    const uint64_t nl_2 = f2_pack(nl, nl);
    const uint64_t nd_2 = f2_pack(ndd, ndd);
    bool ok = true;
    if constexpr (C::ATMEM) {
      // This thread's row of Q_t and of dO_t from shared memory (128-byte swizzle: 16-byte granule g of
      // row r sits at granule g ^ (r % 8)) into its TMEM lane: 32-bit column c holds elements 2c, 2c + 1.
      bool okq = mbar_wait(bar_q, 0, abort_flag, p.err, WB_Q);
      ok = __all_sync(0xffffffffu, okq);
      if (ok) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint8_t* src = smem + (m == 0 ? C::OFF_Q : C::OFF_DO) + t * C::Q_BYTES + row * 128;
          uint32_t w[32];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + ((g ^ (row & 7)) << 4));
            w[4 * g] = x.x;
            w[4 * g + 1] = x.y;
            w[4 * g + 2] = x.z;
            w[4 * g + 3] = x.w;
          }
          tmem_st32(tmem + lane_base + (m == 0 ? C::COL_QA : C::COL_DOA) + t * (C::D / 2), w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qa(t));
      }
    }
    for (int j = 0; ok && j < T; ++j) {
      bool okw = mbar_wait(bar_sf(t), j & 1, abort_flag, p.err, WB_SF);
      ok = __all_sync(0xffffffffu, okw);
      if (!ok) break;
      tc_fence_after();
      const int valid = row_lim - j * C::BC;  // key columns of this step the row may see
      uint64_t pp[C::BC / 2];
      if (__all_sync(0xffffffffu, valid >= C::BC))
        dq_p_regs<C, false>(tS, c2, nl_2, valid, pp);
      else
        dq_p_regs<C, true>(tS, c2, nl_2, valid, pp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sr(t));  // S_t may be overwritten by the next step's S
      okw = mbar_wait(bar_dpf(t), j & 1, abort_flag, p.err, WB_SF);
      ok = __all_sync(0xffffffffu, okw);
      if (!ok) break;
      tc_fence_after();
      dq_ds_regs<C>(tdP, nd_2, pp);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pf(t));
    }
    bool okd = ok && mbar_wait(bar_od(t), 0, abort_flag, p.err, WB_OD);
    okd = __all_sync(0xffffffffu, okd);
    if (okd) {
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + C::COL_DQ + t * C::D;
      uint8_t* out = static_cast<uint8_t*>(p.dq) + (static_cast<size_t>(bh) * p.Nq + qrow) * (C::D * 2);
#pragma unroll
      for (int cc = 0; cc < C::D / 32; ++cc) {
        uint32_t a[32];
        tmem_ld32(tacc + cc * 32, a);
        tmem_wait_ld();
        reg_fence(a);
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(out + cc * 64);
          const float mul = p.scale;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 wv;
            wv.x = pack_bf16x2(__uint_as_float(a[8 * v4 + 0]) * mul, __uint_as_float(a[8 * v4 + 1]) * mul);
            wv.y = pack_bf16x2(__uint_as_float(a[8 * v4 + 2]) * mul, __uint_as_float(a[8 * v4 + 3]) * mul);
            wv.z = pack_bf16x2(__uint_as_float(a[8 * v4 + 4]) * mul, __uint_as_float(a[8 * v4 + 5]) * mul);
            wv.w = pack_bf16x2(__uint_as_float(a[8 * v4 + 6]) * mul, __uint_as_float(a[8 * v4 + 7]) * mul);
            dst[v4] = wv;
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::LOAD_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // When this grid overlaps the tail of the dK/dV grid (programmatic launch), it completes only after
  // that grid has: work enqueued after the backward sees all three gradients.
  griddep_wait();
}

}  // namespace fa
