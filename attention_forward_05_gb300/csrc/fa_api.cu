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
std::atomic<int> g_fault{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local int t_last_cuda = 0;  // last CUDA error seen by this host thread inside the library

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e) {
  t_last_cuda = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// Per-device setup: checks the device is sm_103 and fetches the error word's address.
int device_setup(int* dev_out, int** err_out) {
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
  return FA_OK;
}

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

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
           float scale, int dtype, fa_stream_t stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * static_cast<long long>(Nq > Nk ? Nq : Nk) * d > kMaxElems) return FA_ERR_INVALID_ARG;
  const bool bf16 = (dtype == FA_BF16);

  int dev = 0;
  int* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != FA_OK) return rc;

  const fa::FwdGeometry geo = fa::fwd_geometry(bf16 ? 1 : 0, d);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  void* ws = nullptr;  // fp32 path only: tf32-rounded Q and K, key-major tf32 V^T (stream-ordered)
  if (geo.v_kmajor) {
    const int nk_pad = (Nk + 3) & ~3;  // row stride of V^T must be a multiple of 16 bytes
    const size_t qb = (static_cast<size_t>(BH) * Nq * d * sizeof(float) + 255) & ~static_cast<size_t>(255);
    const size_t kb = (static_cast<size_t>(BH) * Nk * d * sizeof(float) + 255) & ~static_cast<size_t>(255);
    const size_t vb = static_cast<size_t>(BH) * d * nk_pad * sizeof(float);
    cudaError_t ea = cudaMallocAsync(&ws, qb + kb + vb, st);
    if (ea != cudaSuccess) return cuda_fail(ea);
    float* qr = static_cast<float*>(ws);
    float* kr = reinterpret_cast<float*>(static_cast<char*>(ws) + qb);
    float* vt = reinterpret_cast<float*>(static_cast<char*>(ws) + qb + kb);
    ea = fa::launch_prep_fp32(static_cast<const float*>(q), static_cast<const float*>(k),
                              static_cast<const float*>(v), qr, kr, vt, static_cast<int>(BH), Nq, Nk, nk_pad, d, st);
    if (ea != cudaSuccess ||
        encode_map(&tq, qr, false, static_cast<int>(BH), Nq, d, geo.box_cols, geo.q_rows) != FA_OK ||
        encode_map(&tk, kr, false, static_cast<int>(BH), Nk, d, geo.box_cols, geo.kv_rows) != FA_OK ||
        encode_map(&tv, vt, false, static_cast<int>(BH), d, nk_pad, 32, d) != FA_OK) {
      cudaFreeAsync(ws, st);
      return ea != cudaSuccess ? cuda_fail(ea) : FA_ERR_CUDA;
    }
  } else if (encode_map(&tq, q, bf16, static_cast<int>(BH), Nq, d, geo.box_cols, geo.q_rows) != FA_OK ||
             encode_map(&tk, k, bf16, static_cast<int>(BH), Nk, d, geo.box_cols, geo.kv_rows) != FA_OK ||
             encode_map(&tv, v, bf16, static_cast<int>(BH), Nk, d, geo.box_cols, geo.kv_rows) != FA_OK) {
    return FA_ERR_CUDA;
  }

  fa::FwdLaunch a;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.o = o;
  a.lse = lse;
  a.err = err;
  a.BH = static_cast<int>(BH);
  a.Nq = Nq;
  a.Nk = Nk;
  a.c = scale * 1.4426950408889634f;
  a.tau = 8.0f;
  a.fault = g_fault.exchange(0);
  a.stream = st;
  cudaError_t e;
  if (bf16)
    e = (d == 64) ? fa::launch_fwd_bf16_d64(a) : fa::launch_fwd_bf16_d128(a);
  else
    e = (d == 64) ? fa::launch_fwd_fp32_d64(a) : fa::launch_fwd_fp32_d128(a);
  if (ws != nullptr) {
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
