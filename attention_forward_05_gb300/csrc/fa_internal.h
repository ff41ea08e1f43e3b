// fa_internal.h -- launch interfaces between the C ABI (fa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include <nvtx3/nvToolsExt.h>

namespace fa {

// NVTX range over one C ABI call, named after the entry point, for timeline tools (Nsight Systems and
// the like).  Header-only NVTX: without an attached tool a push or pop is a cheap no-op.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Launch with programmatic stream serialization: the kernel may start before the previous kernel in
// the stream has completed, once every CTA of that kernel has executed griddepcontrol.launch_dependents.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, int threads, int smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The C ABI's per-device check for the current device: FA_OK on an sm_103 GPU (after fetching the
// library's device error word), FA_ERR_UNSUPPORTED on any other device, FA_ERR_CUDA when a runtime
// call fails.  Allocates nothing.
int current_device_status();

struct FwdLaunch {
  const CUtensorMap* tm_q;  // 3-D maps over [B*H, N, d] (innermost d), 128-byte swizzle
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  void* o;                  // [B, H, Nq, d], same dtype as the inputs
  float* lse;               // [B, H, Nq] or nullptr
  int* err;                 // device error word
  int BH, Nq, Nk;
  int H, Hkv;               // query heads per batch, key/value heads per batch (H % Hkv == 0)
  int kv_per_split;         // keys per split, a multiple of the key tile (Nk rounded up when not split)
  int n_split;              // key splits; > 1 writes partial states to ws_o / ws_ml for fa_fwd_merge
  float* ws_o;              // [n_split][BH][Nq][d] fp32 unnormalised O
  float* ws_ml;             // [n_split][BH][Nq][2] fp32 (m in log2 units, l)
  int causal;               // 1: query row i sees keys j <= i + Nk - Nq (requires Nq <= Nk)
  float c;                  // scale * log2(e)
  float tau;                // lazy-rescale threshold in log2 units (0 = rescale whenever m grows)
  int fault;                // test-only fault injection mode (0 = none)
  cudaStream_t stream;
  int dependent = 0;        // 1: the fp32 prep kernel precedes it on `stream` (programmatic dependent launch)
  // Key-split CTAs (bf16, d = 64, no mask, n_split == 1; ks_half = 0: none): the grid is ks_whole usual
  // CTAs (units 0 .. ks_whole - 1) and then ks_count CTAs of one 128-row query tile each (tiles
  // ks_tile0 .. of the head-major list of 128-row tiles), whose two tile slots take the keys [0, ks_half)
  // and [ks_half, Nk) and merge (fa_fwd_kernel.cuh, FwdParams).
  int ks_whole = 0, ks_tile0 = 0, ks_count = 0, ks_half = 0;
};

// Tile geometry the tensor maps must be encoded with, per instantiation.
struct FwdGeometry {
  int box_cols;     // elements per 128-byte row segment (64 bf16, 32 fp32)
  int q_rows;       // rows per Q box (128)
  int kv_rows;      // rows per K box (the KV tile, Bc)
  int v_kmajor;     // 1: V is read from a key-major copy [BH, d, Nk_pad] with boxes (32 keys, d rows)
  int rows_per_cta; // query rows one CTA covers
  int ctas_per_sm;  // CTAs of this instantiation resident per SM
};

FwdGeometry fwd_geometry(int dtype_is_bf16, int d);
FwdGeometry fwd_geometry_bf16(int d);

// Merge of per-split partial states into O (dtype of the forward) and LSE:
// O = sum_s o_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s; LSE = (M + log2 L) ln 2.
// `order`: nullptr (index order) or a device int32 permutation of 0 .. n_split - 1.
cudaError_t launch_fwd_merge(const float* ws_o, const float* ws_ml, void* o, float* lse, long long rows, int d,
                             int n_split, int out_bf16, cudaStream_t stream, const int* order = nullptr);

// fp32 prep pass: qr = tf32(q), kr = tf32(k) (round to nearest), and the key-major copy
// vt[bh][c][j] = tf32(v[bh][j][c]) for j < Nk, 0 for Nk <= j < Nk_pad.
cudaError_t launch_prep_fp32(const float* q, const float* k, const float* v, float* qr, float* kr, float* vt,
                             int BH, int BHkv, int Nq, int Nk, int Nk_pad, int d, cudaStream_t stream);
cudaError_t launch_fwd_bf16_d64(const FwdLaunch& a);
cudaError_t launch_fwd_bf16_d128(const FwdLaunch& a);
cudaError_t launch_fwd_fp32_d64(const FwdLaunch& a);
cudaError_t launch_fwd_fp32_d128(const FwdLaunch& a);
// bf16 forward shaped for grouped-query decode (one query tile per CTA); see fa_fwd_decode.cu
// `sms`: the device's SM count (picks the d = 64 configuration whose CTAs start in one wave, if any)
cudaError_t launch_fwd_decode(const FwdLaunch& a, int d, int sms);
FwdGeometry fwd_geometry_decode(int d);

struct BwdLaunch {
  // maps for the dK/dV kernel: K, V boxes (64 cols, kv_keys rows); Q, dO boxes (64 cols, kv_qrows rows)
  const CUtensorMap* tm_k_kv;
  const CUtensorMap* tm_v_kv;
  const CUtensorMap* tm_q_kv;
  const CUtensorMap* tm_do_kv;
  // maps for the dQ kernel: Q, dO boxes (64 cols, q_rows rows); K, V boxes (64 cols, q_keys rows)
  const CUtensorMap* tm_q_q;
  const CUtensorMap* tm_do_q;
  const CUtensorMap* tm_k_q;
  const CUtensorMap* tm_v_q;
  const void* q;            // [BH, Nq, d] (read directly by the fp32 kernels; bf16 reads through the maps)
  const void* k;            // [BHkv, Nk, d]
  const void* v;
  const void* o;            // [BH, Nq, d] forward output, in the inputs' dtype
  const void* dout;         // [BH, Nq, d]
  const float* lse;         // [BH, Nq] natural-log LSE of the forward
  void* dq;                 // [BH, Nq, d]
  void* dk;                 // [BHkv, Nk, d]
  void* dv;
  float* rowv;              // bf16: workspace [BH][Nq_pad/2][4]: (-L log2 e, -D) interleaved by row pairs;
                            // fp32: [BH][Nq_pad] of -L log2 e
  float* rowv2;             // fp32: [BH][Nq_pad] of -D
  int* err;
  int BH, BHkv, H, Hkv, Nq, Nk, Nq_pad, d;
  int causal;
  float c;                  // scale * log2(e)
  float scale;
  int fault;                // test-only fault injection mode for the dK/dV kernel (0 = none)
  cudaStream_t stream;
};

struct BwdGeometry {
  int kv_keys;   // keys per dK/dV CTA
  int kv_qrows;  // query rows per dK/dV step
  int q_rows;    // query rows per dQ tile
  int q_keys;    // keys per dQ step
  int nq_align;  // Nq_pad is Nq rounded up to this
};

BwdGeometry bwd_geometry(int d);
// prep pass, then dK/dV, then dQ, in stream order
cudaError_t launch_bwd_bf16(const BwdLaunch& a);
// fp32 tensors, fp32 arithmetic on the CUDA cores (fa_bwd_fp32.cu); the same three launches.  Nq_pad
// must be a multiple of bwd_fp32_nq_align().
cudaError_t launch_bwd_fp32(const BwdLaunch& a);
int bwd_fp32_nq_align();

struct DecodeLaunch {
  const void* q;            // [BH, d] bf16
  const void* k;            // [BH, Nk, d] bf16
  const void* v;
  void* o;                  // [BH, d] bf16
  float* lse;               // [BH] or nullptr
  float* ws;                // workspace: m [BH*splits], l [BH*splits], o [BH*splits*d]
  const int* order;         // [splits] or nullptr
  int BH, Nk, d, splits;
  float c;                  // scale * log2(e)
  cudaStream_t stream;
};

cudaError_t launch_decode(const DecodeLaunch& a);

// Merge of per-(head, chunk) decode states in `order` (or 0..splits-1): o = sum w o_s / sum w l_s.
cudaError_t launch_decode_merge(const float* ws_m, const float* ws_l, const float* ws_o, const int* order, void* o,
                                float* lse, int BH, int splits, int d, cudaStream_t stream);

struct DecodeGqaLaunch {
  const void* q;            // [B, H, d] bf16
  const void* k;            // [B, Hkv, Nk, d] bf16
  const void* v;
  void* o;                  // [B, H, d] bf16
  float* lse;               // [B, H] or nullptr
  float* ws;                // m [B*H*splits], l [B*H*splits], o [B*H*splits*d]
  const int* order;         // [splits] or nullptr
  int* err;                 // device error word
  int B, H, Hkv, Nk, d, splits;
  float c;                  // scale * log2(e)
  cudaStream_t stream;
};

// 1 when one CTA can serve a group of this many query heads per key/value head (1, 2, 4 or a
// multiple of 8).
int decode_gqa_supported_group(int group);
cudaError_t launch_decode_gqa(const DecodeGqaLaunch& a);

}  // namespace fa
