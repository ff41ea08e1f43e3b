// fa_fwd_fp32.cu -- fp32-input instantiations (operands multiplied as TF32).
//   d = 64 : Bc = 128, two query tiles per CTA, 2-stage ring (192 KB shared)
//   d = 128: Bc = 64, one query tile per CTA, 2-stage ring (192 KB shared)
// A prep pass runs first: tf32 tensor-core operands must be K-major, so P V
// reads V from a key-major copy; and the tensor core truncates fp32 operands
// to tf32, a one-sided error that biases every score, so the prep pass also
// rounds Q, K and V to the nearest tf32 value (cvt.rna) once.
#include "fa_fwd_kernel.cuh"

namespace fa {

using CfgF32D64 = FwdCfg<float, 64, 128, 2, 2>;
using CfgF32D128 = FwdCfg<float, 128, 64, 1, 2>;

cudaError_t launch_fwd_fp32_d64(const FwdLaunch& a) { return launch_fwd<CfgF32D64>(a); }
cudaError_t launch_fwd_fp32_d128(const FwdLaunch& a) { return launch_fwd<CfgF32D128>(a); }

FwdGeometry fwd_geometry(int dtype_is_bf16, int d) {
  if (dtype_is_bf16) return fwd_geometry_bf16(d);
  if (d == 64) return FwdGeometry{32, 128, CfgF32D64::BC, 1, CfgF32D64::BR * CfgF32D64::NQT, CfgF32D64::MINB};
  return FwdGeometry{32, 128, CfgF32D128::BC, 1, CfgF32D128::BR * CfgF32D128::NQT, CfgF32D128::MINB};
}

__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// The prep pass, one launch: CTAs [0, n_tr) transpose V in 32 x 32 blocks (staged through shared
// memory so that both the read of V rows and the write of V^T rows are coalesced; block t covers key
// rows 32 (t % n_kb) .. and columns 32 (t / n_kb % (d / 32)) .. of head t / (n_kb d / 32)); the rest
// copy Q and K rounded to the nearest tf32 value (n4q, n4k float4s, 16-byte aligned pointers).
__global__ void __launch_bounds__(256) prep_fp32_kernel(const float* __restrict__ v, float* __restrict__ vt,
                                                        const float4* __restrict__ q, float4* __restrict__ qr,
                                                        size_t n4q, const float4* __restrict__ k,
                                                        float4* __restrict__ kr, size_t n4k, int Nk, int Nk_pad,
                                                        int d, int n_kb, long long n_tr) {
  griddep_launch_dependents();  // the forward may do its set-up; it waits for this grid's outputs
  if (static_cast<long long>(blockIdx.x) < n_tr) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int ncb = d / 32;
    const long long t = blockIdx.x;
    const int kb = static_cast<int>(t % n_kb);
    const int cb = static_cast<int>((t / n_kb) % ncb);
    const long long bh = t / (static_cast<long long>(n_kb) * ncb);
    const int j0 = kb * 32, c0 = cb * 32;
    const float* vb = v + static_cast<size_t>(bh) * Nk * d;
    float* tb = vt + static_cast<size_t>(bh) * d * Nk_pad;
    for (int r = ty; r < 32; r += 8) {
      const int j = j0 + r;
      tile[r][tx] = (j < Nk) ? round_tf32(vb[static_cast<size_t>(j) * d + c0 + tx]) : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
      const int j = j0 + tx;
      if (j < Nk_pad) tb[static_cast<size_t>(c0 + r) * Nk_pad + j] = tile[tx][r];
    }
    return;
  }
  const size_t n4 = n4q + n4k;
  const size_t stride = (gridDim.x - static_cast<size_t>(n_tr)) * blockDim.x;
  for (size_t i = (blockIdx.x - static_cast<size_t>(n_tr)) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = i < n4q ? q[i] : k[i - n4q];
    a.x = round_tf32(a.x);
    a.y = round_tf32(a.y);
    a.z = round_tf32(a.z);
    a.w = round_tf32(a.w);
    if (i < n4q)
      qr[i] = a;
    else
      kr[i - n4q] = a;
  }
}

cudaError_t launch_prep_fp32(const float* q, const float* k, const float* v, float* qr, float* kr, float* vt,
                             int BH, int BHkv, int Nq, int Nk, int Nk_pad, int d, cudaStream_t stream) {
  const int n_kb = (Nk_pad + 31) / 32;
  const long long n_tr = static_cast<long long>(n_kb) * (d / 32) * BHkv;
  if (n_tr <= 0 || d % 32 != 0) return cudaErrorInvalidValue;
  const size_t nq4 = static_cast<size_t>(BH) * Nq * d / 4, nk4 = static_cast<size_t>(BHkv) * Nk * d / 4;
  const size_t n4 = nq4 + nk4;
  const long long n_round = static_cast<long long>(n4 / 256 + 1 < 4096 ? n4 / 256 + 1 : 4096);
  const long long grid = n_tr + n_round;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  prep_fp32_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      v, vt, reinterpret_cast<const float4*>(q), reinterpret_cast<float4*>(qr), nq4,
      reinterpret_cast<const float4*>(k), reinterpret_cast<float4*>(kr), nk4, Nk, Nk_pad, d, n_kb, n_tr);
  return cudaGetLastError();
}

}  // namespace fa
