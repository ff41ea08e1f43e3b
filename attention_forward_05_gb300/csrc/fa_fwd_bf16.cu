// fa_fwd_bf16.cu -- bf16 instantiations of the fused forward kernel.
// Template arguments: head dim, key tile Bc, 128-row query tiles per CTA, K/V ring stages, CTAs per SM,
// softmax warpgroups per tile, P handed over in two halves.
//   d = 64 : Bc = 64, two query tiles per CTA, 4-stage K/V ring (96 KB shared), 2 CTAs/SM
//            (four softmax warpgroups per SM: the d = 64 softmax is as costly as its MMAs)
//   d = 128: Bc = 128, two query tiles per CTA, 2-stage K/V ring (192 KB shared), 1 CTA/SM; P is handed
//            to the MMA warp in two halves, so P V of the first 64 keys overlaps the second half's exps
#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

using CfgBf16D64 = FwdCfg<__nv_bfloat16, 64, 64, 2, 4, 2, false>;
using CfgBf16D128 = FwdCfg<__nv_bfloat16, 128, 128, 2, 2, 1, true>;

cudaError_t launch_fwd_bf16_d64(const FwdLaunch& a) { return launch_fwd<CfgBf16D64>(a); }
cudaError_t launch_fwd_bf16_d128(const FwdLaunch& a) { return launch_fwd<CfgBf16D128>(a); }
FwdGeometry fwd_geometry_bf16(int d) {
  if (d == 64)
    return FwdGeometry{64, 128, CfgBf16D64::BC, 0, CfgBf16D64::BR * CfgBf16D64::NQT, CfgBf16D64::MINB};
  return FwdGeometry{64, 128, CfgBf16D128::BC, 0, CfgBf16D128::BR * CfgBf16D128::NQT, CfgBf16D128::MINB};
}

}  // namespace fa
