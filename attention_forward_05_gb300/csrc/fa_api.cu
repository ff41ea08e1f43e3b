// fa_api.cu -- the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, workspace handling, kernel launches and status codes.
// Host code only (plus the device error word).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

__device__ int g_fa_err;  // device error word: 0, or DEV_TIMEOUT | wait site

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_cc_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
int g_sms[kMaxDevices] = {};    // multiprocessor count
std::atomic<int> g_fault{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local int t_last_cuda = 0;  // last CUDA error seen by this host thread inside the library

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e) {
  t_last_cuda = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// Per-device setup: checks the device is sm_103 and fetches the error word's address.
int device_setup(int* dev_out, int** err_out, int* sms_out = nullptr) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_cc_ok[dev] == 0) {
    int major = 0, minor = 0;
    if ((ce = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (ce = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(ce);
    g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    if ((ce = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(ce);
  }
  if (g_cc_ok[dev] != 1) return FA_ERR_UNSUPPORTED;
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if ((ce = cudaGetSymbolAddress(&p, g_fa_err)) != cudaSuccess) return cuda_fail(ce);
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    ce = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorSymbolNotFound);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *dev_out = dev;
  *err_out = g_err_ptr[dev];
  if (sms_out) *sms_out = g_sms[dev];
  return FA_OK;
}

}  // namespace

namespace fa {
int current_device_status() {
  int dev = 0;
  int* err = nullptr;
  return device_setup(&dev, &err);
}
}  // namespace fa

namespace {

// 3-D tiled map over a contiguous [BH, rows, inner] tensor: dims (inner, rows, BH),
// box (box_cols, box_rows, 1), 128-byte swizzle, out-of-bounds elements read as zero.
int encode_map(CUtensorMap* map, const void* base, bool bf16, int BH, int rows, int inner, int box_cols,
               int box_rows) {
  const cuuint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * esz, static_cast<cuuint64_t>(rows) * inner * esz};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda = 100000 + static_cast<int>(r);  // driver result codes are reported offset by 100000
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

constexpr long long kMaxElems = 1LL << 40;

// Lazy rescale threshold of the forward kernels (log2 units): a row's reference maximum moves only
// when a score exceeds it by more than this, so P <= 2^32.  P is bf16 (tf32 on the fp32 path) and the
// accumulators fp32, all with fp32's exponent range: 2^32 costs no precision, and O stays finite for
// any |v| below 2^(127 - 32 - log2 Nk).  A larger threshold rescales O less often: with the peaked
// d = 128 inputs 8 corrected O in a third of the warp-steps, and 32 measured 5% faster.
constexpr float kLazyTau = 32.0f;

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_debug_set_fault(int mode) {
  if (mode < 0 || mode > 1) return FA_ERR_INVALID_ARG;
  g_fault.store(mode);
  return FA_OK;
}

}  // extern "C"

namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Work split and workspace layout of one forward call.
struct FwdPlan {
  int n_split = 1, kv_per_split = 0, nk_pad = 0;
  size_t off_qr = 0, off_kr = 0, off_vt = 0, off_wo = 0, off_wml = 0, total = 0;
};

// Validates the forward arguments that do not involve pointers.  sms = 0 means "device unknown"
// (only allowed when kv_splits != 0).
int plan_fwd(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype, int causal, int kv_splits, int sms,
             FwdPlan* pl) {
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;  // the first Nq - Nk rows would see no key
  if (kv_splits < 0) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * static_cast<long long>(Nq > Nk ? Nq : Nk) * d > kMaxElems) return FA_ERR_INVALID_ARG;
  const bool bf16 = dtype == FA_BF16;
  const fa::FwdGeometry geo = fa::fwd_geometry(bf16 ? 1 : 0, d);
  const long long tiles = (Nk + geo.kv_rows - 1) / geo.kv_rows;
  long long n = kv_splits;
  if (n == 0) {  // automatic: split the keys only when the query tiles cannot fill the GPU
    if (sms <= 0) return FA_ERR_INVALID_ARG;
    const long long ctas = ((Nq + geo.rows_per_cta - 1) / geo.rows_per_cta) * BH;
    const long long slots = static_cast<long long>(sms) * geo.ctas_per_sm;
    n = 1;
    if (2 * ctas < slots) {
      n = (slots + ctas - 1) / ctas;
      const long long most = tiles / 2 > 1 ? tiles / 2 : 1;  // keep >= 2 key tiles per split
      if (n > most) n = most;
      if (n > 64) n = 64;
    }
  }
  if (n > tiles) return FA_ERR_INVALID_ARG;
  const long long per = ((tiles + n - 1) / n) * geo.kv_rows;
  pl->kv_per_split = static_cast<int>(per);
  pl->n_split = static_cast<int>((Nk + per - 1) / per);  // every split owns at least one key
  size_t off = 0;
  if (geo.v_kmajor) {
    pl->nk_pad = (Nk + 3) & ~3;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    pl->off_qr = off;
    off += round256(static_cast<size_t>(BH) * Nq * d * sizeof(float));
    pl->off_kr = off;
    off += round256(static_cast<size_t>(BHkv) * Nk * d * sizeof(float));
    pl->off_vt = off;
    off += round256(static_cast<size_t>(BHkv) * d * pl->nk_pad * sizeof(float));
  }
  if (pl->n_split > 1) {
    pl->off_wo = off;
    off += round256(static_cast<size_t>(pl->n_split) * BH * Nq * d * sizeof(float));
    pl->off_wml = off;
    off += round256(static_cast<size_t>(pl->n_split) * BH * Nq * 2 * sizeof(float));
  }
  pl->total = off;
  return FA_OK;
}

// The last, partial wave of a d = 64 bf16 forward without mask or key splits.  When the CTA units (256
// query rows) do not fill whole waves of two CTAs per SM and what is left is at most one CTA per SM,
// those CTAs would each run alone on an SM through all the key tiles.  Their rows are taken instead by
// key-split CTAs: one 128-row query tile each, its two tile slots over the two halves of the keys,
// merged inside the CTA at the end (twice as many CTAs, chains of half the length).
void plan_key_split(long long BH, int Nq, int Nk, int sms, const fa::FwdGeometry& geo, fa::FwdLaunch* a) {
  if (sms <= 0 || geo.rows_per_cta != 256 || geo.ctas_per_sm != 2 || geo.kv_rows != 64) return;
  const long long per_head = (Nq + 255) / 256, per_head1 = (Nq + 127) / 128;
  const long long units = per_head * BH, slots = 2LL * sms;
  const long long rest = units % slots;
  const long long tiles = (Nk + 63) / 64;
  if (units < slots || rest == 0 || rest > sms || tiles < 8) return;
  const long long u0 = units - rest;  // first unit of the last wave: head u0 / per_head, block u0 % per_head
  const long long first = (u0 / per_head) * per_head1 + 2 * (u0 % per_head);
  const long long count = BH * per_head1 - first;
  if (u0 + count > 0x7FFFFFFFLL) return;
  a->ks_whole = static_cast<int>(u0);
  a->ks_tile0 = static_cast<int>(first);
  a->ks_count = static_cast<int>(count);
  a->ks_half = static_cast<int>((tiles + 1) / 2 * 64);
}

}  // namespace

extern "C" {

size_t fa_fwd_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype, int causal, int kv_splits) {
  int sms = 0;
  if (kv_splits == 0) {
    int dev = 0;
    int* err = nullptr;
    if (device_setup(&dev, &err, &sms) != FA_OK) return 0;
  }
  FwdPlan pl;
  if (plan_fwd(B, H, Hkv, Nq, Nk, d, dtype, causal, kv_splits, sms, &pl) != FA_OK) return 0;
  return pl.total;
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
              int Nk, int d, float scale, int dtype, int causal, int kv_splits, void* workspace,
              size_t workspace_bytes, fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_fwd_ex");
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  FwdPlan pl;
  int rc = plan_fwd(B, H, Hkv, Nq, Nk, d, dtype, causal, kv_splits == 0 ? 1 : kv_splits, 0, &pl);
  if (rc != FA_OK) return rc;  // argument errors are reported before touching the device

  int dev = 0, sms = 0;
  int* err = nullptr;
  rc = device_setup(&dev, &err, &sms);
  if (rc != FA_OK) return rc;
  if (kv_splits == 0 && (rc = plan_fwd(B, H, Hkv, Nq, Nk, d, dtype, causal, 0, sms, &pl)) != FA_OK) return rc;
  if (workspace && workspace_bytes < pl.total) return FA_ERR_INVALID_ARG;

  const bool bf16 = (dtype == FA_BF16);
  const int BH = B * H, BHkv = B * Hkv;
  const fa::FwdGeometry geo = fa::fwd_geometry(bf16 ? 1 : 0, d);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool own_ws = false;
  if (ws == nullptr && pl.total > 0) {
    void* wp = nullptr;
    cudaError_t ea = cudaMallocAsync(&wp, pl.total, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
    ws = static_cast<char*>(wp);
    own_ws = true;
  }
  auto fail = [&](cudaError_t e) {
    if (own_ws) cudaFreeAsync(ws, st);
    return e != cudaSuccess ? cuda_fail(e) : FA_ERR_CUDA;
  };

  CUtensorMap tq, tk, tv;
  if (geo.v_kmajor) {  // fp32: tf32-rounded Q and K, key-major tf32 V^T (tf32 MMA operands are K-major)
    float* qr = reinterpret_cast<float*>(ws + pl.off_qr);
    float* kr = reinterpret_cast<float*>(ws + pl.off_kr);
    float* vt = reinterpret_cast<float*>(ws + pl.off_vt);
    cudaError_t ea = fa::launch_prep_fp32(static_cast<const float*>(q), static_cast<const float*>(k),
                                          static_cast<const float*>(v), qr, kr, vt, BH, BHkv, Nq, Nk, pl.nk_pad, d,
                                          st);
    if (ea != cudaSuccess) return fail(ea);
    if (encode_map(&tq, qr, false, BH, Nq, d, geo.box_cols, geo.q_rows) != FA_OK ||
        encode_map(&tk, kr, false, BHkv, Nk, d, geo.box_cols, geo.kv_rows) != FA_OK ||
        encode_map(&tv, vt, false, BHkv, d, pl.nk_pad, 32, d) != FA_OK)
      return fail(cudaSuccess);
  } else if (encode_map(&tq, q, bf16, BH, Nq, d, geo.box_cols, geo.q_rows) != FA_OK ||
             encode_map(&tk, k, bf16, BHkv, Nk, d, geo.box_cols, geo.kv_rows) != FA_OK ||
             encode_map(&tv, v, bf16, BHkv, Nk, d, geo.box_cols, geo.kv_rows) != FA_OK) {
    return fail(cudaSuccess);
  }

  fa::FwdLaunch a;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.o = o;
  a.lse = lse;
  a.err = err;
  a.BH = BH;
  a.Nq = Nq;
  a.Nk = Nk;
  a.H = H;
  a.Hkv = Hkv;
  a.kv_per_split = pl.kv_per_split;
  a.n_split = pl.n_split;
  a.ws_o = pl.n_split > 1 ? reinterpret_cast<float*>(ws + pl.off_wo) : nullptr;
  a.ws_ml = pl.n_split > 1 ? reinterpret_cast<float*>(ws + pl.off_wml) : nullptr;
  a.causal = causal;
  a.c = scale * 1.4426950408889634f;
  a.tau = kLazyTau;
  a.fault = g_fault.exchange(0);
  a.stream = st;
  a.dependent = geo.v_kmajor ? 1 : 0;  // the fp32 prep kernel was the last launch on `st`
  if (bf16 && d == 64 && !causal && kv_splits == 0 && pl.n_split == 1) plan_key_split(BH, Nq, Nk, sms, geo, &a);
  cudaError_t e;
  if (bf16)
    e = (d == 64) ? fa::launch_fwd_bf16_d64(a) : fa::launch_fwd_bf16_d128(a);
  else
    e = (d == 64) ? fa::launch_fwd_fp32_d64(a) : fa::launch_fwd_fp32_d128(a);
  if (e == cudaSuccess && pl.n_split > 1)
    e = fa::launch_fwd_merge(a.ws_o, a.ws_ml, o, lse, static_cast<long long>(BH) * Nq, d, pl.n_split, bf16 ? 1 : 0,
                             st);
  if (own_ws) {
    cudaError_t e2 = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// Per-device copy streams and events for fa_fwd_host, created on first use.  The mutex keeps one
// host thread's enqueue sequence (which re-records the shared events) whole.
constexpr int kHostMaxChunks = 16;
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in_end = nullptr, ev_in[kHostMaxChunks] = {},
              ev_done[kHostMaxChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.ev_start, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.ev_end, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.ev_in_end, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e);
    for (int i = 0; i < kHostMaxChunks; ++i)
      if ((e = cudaEventCreateWithFlags(&hp.ev_in[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&hp.ev_done[i], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

// Chunks of fa_fwd_host, in key/value-head units.  The host link (about 200 GB/s each way) moves
// the inputs slower than the forward consumes them, so what shows besides the copies is the first
// chunk's copy in and the last chunk's compute and copy out.  A chunk launches `unit_ctas` CTAs per
// unit; `wave` units fill the SMs' CTA slots once.  The chunks are about one wave each, the last
// half a wave: small enough to start early and end soon, large enough that the forward keeps up with
// the copies.  Measured end to end on both prefill problems: 16 MB chunks (the d = 128 forward at
// under a wave per launch) 696 TFLOP/s; one-wave chunks 757-767; two-wave 752; three-wave 711; a
// half-wave last chunk 777.  Writes bounds[0 .. n] and returns n.
constexpr int kHostRestWaves = 1;
int host_chunks(long long units, long long unit_ctas, long long slots, long long* bounds) {
  const long long wave = slots / unit_ctas > 1 ? slots / unit_ctas : 1;
  const long long half = wave / 2 > 1 ? wave / 2 : 1;
  const long long last = units < half ? units : half;
  const long long rest = units - last;
  long long n_rest = 0;
  if (rest > 0) {
    const long long per = kHostRestWaves * wave;
    n_rest = (rest + per / 2) / per;
    if (n_rest < 1) n_rest = 1;
    if (n_rest > kHostMaxChunks - 1) n_rest = kHostMaxChunks - 1;
  }
  bounds[0] = 0;
  for (long long i = 1; i <= n_rest; ++i) bounds[i] = rest * i / n_rest;
  bounds[n_rest + 1] = units;
  return static_cast<int>(n_rest + 1);
}

// Device layout of fa_fwd_host's workspace: q, k, v, o, lse, each 256-byte aligned.
struct HostLayout {
  size_t q = 0, k = 0, v = 0, o = 0, lse = 0, total = 0;
};
HostLayout host_layout(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype) {
  const size_t esz = dtype == FA_BF16 ? 2 : 4;
  const size_t nq = static_cast<size_t>(B) * H * Nq * d * esz, nkv = static_cast<size_t>(B) * Hkv * Nk * d * esz;
  HostLayout l;
  l.q = 0;
  l.k = l.q + round256(nq);
  l.v = l.k + round256(nkv);
  l.o = l.v + round256(nkv);
  l.lse = l.o + round256(nq);
  l.total = l.lse + round256(static_cast<size_t>(B) * H * Nq * sizeof(float));
  return l;
}

}  // namespace

extern "C" {

size_t fa_fwd_host_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype, int causal) {
  FwdPlan pl;
  if (plan_fwd(B, H, Hkv, Nq, Nk, d, dtype, causal, 1, 0, &pl) != FA_OK) return 0;
  return host_layout(B, H, Hkv, Nq, Nk, d, dtype).total;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
                int Nk, int d, float scale, int dtype, int causal, void* workspace, size_t workspace_bytes,
                fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_fwd_host");
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  FwdPlan pl;
  int rc = plan_fwd(B, H, Hkv, Nq, Nk, d, dtype, causal, 1, 0, &pl);
  if (rc != FA_OK) return rc;
  const HostLayout lay = host_layout(B, H, Hkv, Nq, Nk, d, dtype);
  if (workspace && workspace_bytes < lay.total) return FA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int* err = nullptr;
  if ((rc = device_setup(&dev, &err, &sms)) != FA_OK) return rc;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool own_ws = false;
  if (ws == nullptr) {
    void* wp = nullptr;
    cudaError_t ea = cudaMallocAsync(&wp, lay.total, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
    ws = static_cast<char*>(wp);
    own_ws = true;
  }
  HostPipe* hp = nullptr;
  std::lock_guard<std::mutex> lk(g_pipe[dev].mu);
  if ((rc = host_pipe(dev, &hp)) != FA_OK) {
    if (own_ws) cudaFreeAsync(ws, st);
    return rc;
  }
  // Chunks of whole key/value heads (each with its H / Hkv query heads): q, k, v, o and lse of a chunk
  // are contiguous ranges.
  const size_t esz = dtype == FA_BF16 ? 2 : 4;
  const int G = H / Hkv;
  const long long units = static_cast<long long>(B) * Hkv;
  const size_t q_unit = static_cast<size_t>(G) * Nq * d * esz, kv_unit = static_cast<size_t>(Nk) * d * esz;
  const fa::FwdGeometry geo = fa::fwd_geometry(dtype == FA_BF16 ? 1 : 0, d);
  const long long unit_ctas = static_cast<long long>(G) * ((Nq + geo.rows_per_cta - 1) / geo.rows_per_cta);
  long long bounds[kHostMaxChunks + 1];
  const int n = host_chunks(units, unit_ctas, static_cast<long long>(sms) * geo.ctas_per_sm, bounds);
  cudaError_t e = cudaEventRecord(hp->ev_start, st);  // device buffers may still be in use by earlier work
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->s_in, hp->ev_start, 0);
  int status = FA_OK;
  for (int c = 0; c < n && e == cudaSuccess && status == FA_OK; ++c) {
    const long long u0 = bounds[c], u1 = bounds[c + 1];
    const size_t nu = static_cast<size_t>(u1 - u0);
    char* dq = ws + lay.q + u0 * q_unit;
    char* dk = ws + lay.k + u0 * kv_unit;
    char* dv = ws + lay.v + u0 * kv_unit;
    char* dout = ws + lay.o + u0 * q_unit;
    float* dl = reinterpret_cast<float*>(ws + lay.lse) + u0 * G * Nq;
    if ((e = cudaMemcpyAsync(dq, static_cast<const char*>(q) + u0 * q_unit, nu * q_unit, cudaMemcpyHostToDevice,
                             hp->s_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk, static_cast<const char*>(k) + u0 * kv_unit, nu * kv_unit, cudaMemcpyHostToDevice,
                             hp->s_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv, static_cast<const char*>(v) + u0 * kv_unit, nu * kv_unit, cudaMemcpyHostToDevice,
                             hp->s_in)) != cudaSuccess ||
        (e = cudaEventRecord(hp->ev_in[c], hp->s_in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, hp->ev_in[c], 0)) != cudaSuccess)
      break;
    status = fa_fwd_ex(dq, dk, dv, dout, dl, 1, static_cast<int>(nu) * G, static_cast<int>(nu), Nq, Nk, d, scale,
                       dtype, causal, 0, nullptr, 0, stream);
    if (status != FA_OK) break;
    if ((e = cudaEventRecord(hp->ev_done[c], st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->s_out, hp->ev_done[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<char*>(o) + u0 * q_unit, dout, nu * q_unit, cudaMemcpyDeviceToHost,
                             hp->s_out)) != cudaSuccess)
      break;
    if (lse && (e = cudaMemcpyAsync(lse + u0 * G * Nq, dl, nu * G * Nq * sizeof(float), cudaMemcpyDeviceToHost,
                                    hp->s_out)) != cudaSuccess)
      break;
  }
  // The caller's stream waits for the last copy out (later work on it sees finished host buffers) and
  // for every copy in: after an error part-way through a chunk, copies already queued on s_in may not
  // yet be covered by an ev_in event, and the workspace must outlive them.
  cudaError_t e2 = cudaEventRecord(hp->ev_end, hp->s_out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, hp->ev_end, 0);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(hp->ev_in_end, hp->s_in);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, hp->ev_in_end, 0);
  if (e == cudaSuccess) e = e2;
  if (own_ws) {
    e2 = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = e2;
  }
  if (status != FA_OK) return status;
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
           float scale, int dtype, fa_stream_t stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, H, Nq, Nk, d, scale, dtype, 0, 0, nullptr, 0, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128)) return 0;
  const long long align = fa::bwd_geometry(d).nq_align;
  const long long nq_pad = (Nq + align - 1) / align * align;
  return 2 * round256(static_cast<size_t>(B) * H * nq_pad * sizeof(float));
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int dtype, int causal,
           void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_bwd");
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * static_cast<long long>(Nq > Nk ? Nq : Nk) * d > kMaxElems) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_bytes(B, H, Nq, d);
  if (workspace && workspace_bytes < need) return FA_ERR_INVALID_ARG;

  int dev = 0;
  int* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != FA_OK) return rc;
  const fa::BwdGeometry geo = fa::bwd_geometry(d);
  const int nq_pad = (Nq + geo.nq_align - 1) / geo.nq_align * geo.nq_align;
  const int BHi = B * H, BHkv = B * Hkv;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool own_ws = false;
  if (ws == nullptr) {
    void* wp = nullptr;
    cudaError_t ea = cudaMallocAsync(&wp, need, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
    ws = static_cast<char*>(wp);
    own_ws = true;
  }
  auto fail = [&](cudaError_t e) {
    if (own_ws) cudaFreeAsync(ws, st);
    return e != cudaSuccess ? cuda_fail(e) : FA_ERR_CUDA;
  };
  fa::BwdLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.rowv = reinterpret_cast<float*>(ws);
  a.rowv2 = reinterpret_cast<float*>(ws + round256(static_cast<size_t>(BHi) * nq_pad * sizeof(float)));
  a.err = err;
  a.BH = BHi;
  a.BHkv = BHkv;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.Nq_pad = nq_pad;
  a.d = d;
  a.causal = causal;
  a.c = scale * 1.4426950408889634f;
  a.scale = scale;
  a.fault = g_fault.exchange(0);  // consumed by either dtype; only the bf16 kernels have waits to fault
  a.stream = st;
  if (dtype == FA_FP32) {
    cudaError_t e = nq_pad % fa::bwd_fp32_nq_align() == 0 ? fa::launch_bwd_fp32(a) : cudaErrorInvalidValue;
    if (own_ws) {
      cudaError_t e2 = cudaFreeAsync(ws, st);
      if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }
  CUtensorMap kk, vk, qk, dok, qq, doq, kq, vq;
  if (encode_map(&kk, k, true, BHkv, Nk, d, 64, geo.kv_keys) != FA_OK ||
      encode_map(&vk, v, true, BHkv, Nk, d, 64, geo.kv_keys) != FA_OK ||
      encode_map(&qk, q, true, BHi, Nq, d, 64, geo.kv_qrows) != FA_OK ||
      encode_map(&dok, dout, true, BHi, Nq, d, 64, geo.kv_qrows) != FA_OK ||
      encode_map(&qq, q, true, BHi, Nq, d, 64, geo.q_rows) != FA_OK ||
      encode_map(&doq, dout, true, BHi, Nq, d, 64, geo.q_rows) != FA_OK ||
      encode_map(&kq, k, true, BHkv, Nk, d, 64, geo.q_keys) != FA_OK ||
      encode_map(&vq, v, true, BHkv, Nk, d, 64, geo.q_keys) != FA_OK)
    return fail(cudaSuccess);
  a.tm_k_kv = &kk;
  a.tm_v_kv = &vk;
  a.tm_q_kv = &qk;
  a.tm_do_kv = &dok;
  a.tm_q_q = &qq;
  a.tm_do_q = &doq;
  a.tm_k_q = &kq;
  a.tm_v_q = &vq;
  cudaError_t e = fa::launch_bwd_bf16(a);
  if (own_ws) {
    cudaError_t e2 = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

size_t fa_decode_workspace_bytes(int B, int H, int d, int splits) {
  if (B < 1 || H < 1 || splits < 1 || (d != 64 && d != 128)) return 0;
  const size_t n = static_cast<size_t>(B) * H * splits;
  return ((n * (2 + d) * sizeof(float)) + 255) & ~static_cast<size_t>(255);
}

int fa_decode_splitkv_ex(const void* q, const void* k, const void* v, void* o, int B, int H, int Nk, int d,
                         int splits, float scale, void* workspace, size_t workspace_bytes, const int* merge_order,
                         float* lse, fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_decode_splitkv_ex");
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (merge_order && (reinterpret_cast<uintptr_t>(merge_order) & 3u)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nk < 1 || Nk >= (1 << 30)) return FA_ERR_INVALID_ARG;
  if (splits < 1 || splits > Nk) return FA_ERR_INVALID_ARG;
  if (splits > 4096) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH * splits > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * static_cast<long long>(Nk) * d > kMaxElems) return FA_ERR_INVALID_ARG;
  const size_t need = fa_decode_workspace_bytes(B, H, d, splits);
  if (workspace && (!aligned16(workspace) || workspace_bytes < need)) return FA_ERR_INVALID_ARG;

  int dev = 0;
  int* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != FA_OK) return rc;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* ws = workspace;
  if (ws == nullptr) {
    cudaError_t ea = cudaMallocAsync(&ws, need, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
  }
  fa::DecodeLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.ws = static_cast<float*>(ws);
  a.order = merge_order;
  a.BH = static_cast<int>(BH);
  a.Nk = Nk;
  a.d = d;
  a.splits = splits;
  a.c = scale * 1.4426950408889634f;
  a.stream = st;
  cudaError_t e = fa::launch_decode(a);
  if (workspace == nullptr) {
    cudaError_t e2 = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// Groups of at least this many query heads per key/value head decode on the tensor cores: the group's
// queries are the rows of a bf16 forward (one 128-row query tile per CTA) over the head's keys, split
// into the decode's chunks.
// FA_GQA_TC_MIN_GROUP overrides it in tuning builds.
#ifndef FA_GQA_TC_MIN_GROUP
#define FA_GQA_TC_MIN_GROUP 4
#endif
constexpr int kGqaTensorMinGroup = FA_GQA_TC_MIN_GROUP;

// Grouped-query decode through the forward kernel in split mode: the G = H / Hkv query heads of a
// key/value head are contiguous in q, so q is a [B*Hkv, G, d] prefill over that head's keys; chunk s
// covers keys [s*L, (s+1)*L) with L a whole number of key tiles, and the forward merge combines the
// chunks in merge_order.  ws holds the fp32 states: O [splits][B*H][d], then (m, l) [splits][B*H].
cudaError_t gqa_decode_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int Hkv, int Nk, int d, int splits, int L, float scale, char* ws,
                               const int* merge_order, int* err, int sms, cudaStream_t st) {
  const fa::FwdGeometry geo = fa::fwd_geometry_decode(d);
  const int G = H / Hkv, BHkv = B * Hkv;
  CUtensorMap tq, tk, tv;
  if (encode_map(&tq, q, true, BHkv, G, d, geo.box_cols, geo.q_rows) != FA_OK ||
      encode_map(&tk, k, true, BHkv, Nk, d, geo.box_cols, geo.kv_rows) != FA_OK ||
      encode_map(&tv, v, true, BHkv, Nk, d, geo.box_cols, geo.kv_rows) != FA_OK)
    return cudaErrorInvalidValue;
  const size_t rows = static_cast<size_t>(B) * H;
  fa::FwdLaunch a;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.o = o;
  a.lse = lse;
  a.err = err;
  a.BH = BHkv;
  a.Nq = G;
  a.Nk = Nk;
  a.H = Hkv;
  a.Hkv = Hkv;
  a.kv_per_split = L;
  a.n_split = splits;
  a.ws_o = splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  a.ws_ml = splits > 1 ? reinterpret_cast<float*>(ws + round256(static_cast<size_t>(splits) * rows * d * sizeof(float)))
                       : nullptr;
  a.causal = 0;
  a.c = scale * 1.4426950408889634f;
  a.tau = kLazyTau;
  a.fault = 0;
  a.stream = st;
  cudaError_t e = fa::launch_fwd_decode(a, d, sms);
  if (e == cudaSuccess && splits > 1)
    e = fa::launch_fwd_merge(a.ws_o, a.ws_ml, o, lse, static_cast<long long>(rows), d, splits, 1, st, merge_order);
  return e;
}

}  // namespace

extern "C" {

int fa_decode_splitkv_gqa(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int Nk, int d,
                          int splits, float scale, void* workspace, size_t workspace_bytes, const int* merge_order,
                          float* lse, fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_decode_splitkv_gqa");
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (merge_order && (reinterpret_cast<uintptr_t>(merge_order) & 3u)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Nk < 1 || Nk >= (1 << 30)) return FA_ERR_INVALID_ARG;
  if (splits < 1 || splits > Nk) return FA_ERR_INVALID_ARG;
  if (splits > 4096) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!fa::decode_gqa_supported_group(H / Hkv)) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH * splits > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hkv * static_cast<long long>(Nk) * d > kMaxElems) return FA_ERR_INVALID_ARG;
  const size_t need = fa_decode_workspace_bytes(B, H, d, splits);
  if (workspace && (!aligned16(workspace) || workspace_bytes < need)) return FA_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  int* err = nullptr;
  int rc = device_setup(&dev, &err, &sms);
  if (rc != FA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* ws = workspace;
  if (ws == nullptr) {
    cudaError_t ea = cudaMallocAsync(&ws, need, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
  }
  const int L = (Nk + splits - 1) / splits;
  const int tile = fa::fwd_geometry_decode(d).kv_rows;
  cudaError_t e;
  if (H / Hkv >= kGqaTensorMinGroup && L % tile == 0 && static_cast<long long>(splits - 1) * L < Nk) {
    e = gqa_decode_forward(q, k, v, o, lse, B, H, Hkv, Nk, d, splits, L, scale, static_cast<char*>(ws), merge_order,
                           err, sms, st);
    if (workspace == nullptr) {
      cudaError_t e2 = cudaFreeAsync(ws, st);
      if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }
  fa::DecodeGqaLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.ws = static_cast<float*>(ws);
  a.order = merge_order;
  a.err = err;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nk = Nk;
  a.d = d;
  a.splits = splits;
  a.c = scale * 1.4426950408889634f;
  a.stream = st;
  e = fa::launch_decode_gqa(a);
  if (workspace == nullptr) {
    cudaError_t e2 = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, int B, int H, int Nk, int d, int splits,
                      fa_stream_t stream) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return fa_decode_splitkv_ex(q, k, v, o, B, H, Nk, d, splits, 1.0f / std::sqrt(static_cast<float>(d)), nullptr, 0,
                              nullptr, nullptr, stream);
}

int fa_last_cuda_error(void) { return t_last_cuda; }

const char* fa_last_cuda_error_string(void) {
  if (t_last_cuda >= 100000) return "CUDA driver error (tensor-map encoding); code = value - 100000";
  return cudaGetErrorString(static_cast<cudaError_t>(t_last_cuda));
}

int fa_check_device_error(void) {
  int dev = 0;
  int* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != FA_OK) return rc;
  int h = 0;
  cudaError_t ce = cudaDeviceSynchronize();
  if (ce != cudaSuccess) return cuda_fail(ce);
  if ((ce = cudaMemcpyFromSymbol(&h, g_fa_err, sizeof(int))) != cudaSuccess) return cuda_fail(ce);
  if (h != 0) {
    const int zero = 0;
    if ((ce = cudaMemcpyToSymbol(g_fa_err, &zero, sizeof(int))) != cudaSuccess) return cuda_fail(ce);
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"
