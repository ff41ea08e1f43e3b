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

// One 32 x 32 block per CTA, staged through shared memory so that both the
// read of V rows and the write of V^T rows are coalesced.
__global__ void __launch_bounds__(256) transpose_v_kernel(const float* __restrict__ v, float* __restrict__ vt,
                                                          int Nk, int Nk_pad, int d, int n_kb) {
  __shared__ float tile[32][33];
  const int bh = blockIdx.x / n_kb;
  const int j0 = (blockIdx.x % n_kb) * 32;
  const int c0 = blockIdx.y * 32;
  const float* vb = v + static_cast<size_t>(bh) * Nk * d;
  float* tb = vt + static_cast<size_t>(bh) * d * Nk_pad;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int j = j0 + r;
    tile[r][threadIdx.x] = (j < Nk) ? round_tf32(vb[static_cast<size_t>(j) * d + c0 + threadIdx.x]) : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int j = j0 + threadIdx.x;
    if (j < Nk_pad) tb[static_cast<size_t>(c0 + r) * Nk_pad + j] = tile[threadIdx.x][r];
  }
}

// Element-wise round-to-nearest tf32 copy (n a multiple of 4, 16-byte aligned pointers).
__global__ void __launch_bounds__(256) round_tf32_kernel(const float4* __restrict__ x, float4* __restrict__ y,
                                                         size_t n4) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 a = x[i];
    a.x = round_tf32(a.x);
    a.y = round_tf32(a.y);
    a.z = round_tf32(a.z);
    a.w = round_tf32(a.w);
    y[i] = a;
  }
}

cudaError_t launch_prep_fp32(const float* q, const float* k, const float* v, float* qr, float* kr, float* vt,
                             int BH, int BHkv, int Nq, int Nk, int Nk_pad, int d, cudaStream_t stream) {
  const int n_kb = (Nk_pad + 31) / 32;
  const long long gx = static_cast<long long>(n_kb) * BHkv;
  if (gx <= 0 || gx > 0x7FFFFFFFLL || d % 32 != 0) return cudaErrorInvalidValue;
  transpose_v_kernel<<<dim3(static_cast<unsigned>(gx), d / 32), dim3(32, 8), 0, stream>>>(v, vt, Nk, Nk_pad, d,
                                                                                         n_kb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t nq4 = static_cast<size_t>(BH) * Nq * d / 4, nk4 = static_cast<size_t>(BHkv) * Nk * d / 4;
  const unsigned gq = static_cast<unsigned>(nq4 / 256 + 1 < 4096 ? nq4 / 256 + 1 : 4096);
  const unsigned gk = static_cast<unsigned>(nk4 / 256 + 1 < 4096 ? nk4 / 256 + 1 : 4096);
  round_tf32_kernel<<<gq, 256, 0, stream>>>(reinterpret_cast<const float4*>(q), reinterpret_cast<float4*>(qr), nq4);
  round_tf32_kernel<<<gk, 256, 0, stream>>>(reinterpret_cast<const float4*>(k), reinterpret_cast<float4*>(kr), nk4);
  return cudaGetLastError();
}

}  // namespace fa
