// fa_decode_noalloc.cu -- split-KV decode that allocates no device memory.
//
// fa_decode_splitkv keeps its fp32 partial states (m, l, o per chunk) in a
// workspace taken with cudaMallocAsync.  Some callers cannot allocate device
// memory at call time: serving processes that reserve nearly all HBM for
// their KV cache up front and run with allocation disabled afterwards, and
// runtimes whose memory manager must own every allocation.  cudaMalloc can
// also block on the device, which such callers cannot afford on their hot
// path.  This entry point serves them: its scratch is a fixed array in the
// library's device image, so a call only launches the two decode kernels.
//
// Costs and rules that come with the fixed array:
//   * Every GPU on which the library is loaded holds FA_DECODE_NOALLOC_SCRATCH_BYTES
//     of device memory for the array until the process exits.
//   * A request whose partial states do not fit is rejected with
//     FA_ERR_UNSUPPORTED before anything is launched.
//   * All calls share the one array.  Two calls whose kernels overlap on the
//     GPU (different streams, no ordering between them) race on it; order such
//     calls, e.g. issue them on one stream.
//   * The array keeps whatever the previous call left.  Nothing needs clearing:
//     the split kernel writes every partial state the merge kernel then reads.
//   * The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current); make that first call
//     before any stream capture.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = FA_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, int B, int H, int Nk,
                                         int d, int splits, fa_stream_t stream) {
  const fa::NvtxRange nvtx_range("fa_decode_splitkv_noalloc");
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nk < 1 || Nk >= (1 << 30)) return FA_ERR_INVALID_ARG;
  if (splits < 1 || splits > Nk) return FA_ERR_INVALID_ARG;
  if (splits > 4096) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH * splits > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * static_cast<long long>(Nk) * d > (1LL << 40)) return FA_ERR_INVALID_ARG;
  if (fa_decode_workspace_bytes(B, H, d, splits) > kScratchBytes) return FA_ERR_UNSUPPORTED;

  // the same device check as every other entry point: sm_103 only, FA_ERR_UNSUPPORTED elsewhere
  const int dev_status = fa::current_device_status();
  if (dev_status != FA_OK) return dev_status;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return FA_ERR_CUDA;
  fa::DecodeLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = nullptr;
  a.ws = static_cast<float*>(ws);
  a.order = nullptr;
  a.BH = static_cast<int>(BH);
  a.Nk = Nk;
  a.d = d;
  a.splits = splits;
  a.c = (1.0f / std::sqrt(static_cast<float>(d))) * 1.4426950408889634f;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return fa::launch_decode(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
