// fa_fwd_bf16.cu -- bf16 instantiations of the fused forward kernel.
// Template arguments: head dim, key tile Bc, 128-row query tiles per CTA, K/V ring stages, CTAs per SM.
//   d = 64 : Bc = 64, two query tiles per CTA, 4-stage K/V ring (96 KB shared), 2 CTAs/SM
//            (four softmax warpgroups per SM: the d = 64 softmax is as costly as its MMAs)
//   d = 128: Bc = 128, two query tiles per CTA, 2-stage K/V ring (192 KB shared), 1 CTA/SM; P is handed
//            to the MMA warp in two halves, so P V of the first 64 keys overlaps the second half's exps
// Compiler definitions FA_D64_{BC,NQT,STAGES,MINB,SPLIT,PV2} / FA_D128_{...} override the
// tile configuration for tuning builds.
#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

#ifndef FA_D64_BC
#define FA_D64_BC 64
#endif
#ifndef FA_D64_NQT
#define FA_D64_NQT 2
#endif
#ifndef FA_D64_STAGES
#define FA_D64_STAGES 4
#endif
#ifndef FA_D64_MINB
#define FA_D64_MINB 2
#endif
#ifndef FA_D128_BC
#define FA_D128_BC 128
#endif
#ifndef FA_D128_NQT
#define FA_D128_NQT 2
#endif
#ifndef FA_D128_STAGES
#define FA_D128_STAGES 2
#endif
#ifndef FA_D128_MINB
#define FA_D128_MINB 1
#endif
#ifndef FA_D64_SPLIT
#define FA_D64_SPLIT 1
#endif
#ifndef FA_D128_SPLIT
#define FA_D128_SPLIT 1
#endif
#ifndef FA_D64_PV2
#define FA_D64_PV2 0
#endif
#ifndef FA_D128_PV2
#define FA_D128_PV2 1
#endif

namespace fa {

using CfgBf16D64 = FwdCfg<__nv_bfloat16, 64, FA_D64_BC, FA_D64_NQT, FA_D64_STAGES, FA_D64_MINB, FA_D64_SPLIT,
                          FA_D64_PV2 != 0>;
using CfgBf16D128 = FwdCfg<__nv_bfloat16, 128, FA_D128_BC, FA_D128_NQT, FA_D128_STAGES, FA_D128_MINB, FA_D128_SPLIT,
                           FA_D128_PV2 != 0>;

cudaError_t launch_fwd_bf16_d64(const FwdLaunch& a) { return launch_fwd<CfgBf16D64>(a); }
cudaError_t launch_fwd_bf16_d128(const FwdLaunch& a) { return launch_fwd<CfgBf16D128>(a); }
FwdGeometry fwd_geometry_bf16(int d) {
  if (d == 64)
    return FwdGeometry{64, 128, CfgBf16D64::BC, 0, CfgBf16D64::BR * CfgBf16D64::NQT, CfgBf16D64::MINB};
  return FwdGeometry{64, 128, CfgBf16D128::BC, 0, CfgBf16D128::BR * CfgBf16D128::NQT, CfgBf16D128::MINB};
}

}  // namespace fa
