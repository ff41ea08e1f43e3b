// fa_fwd_decode.cu -- instantiations of the fused forward kernel shaped for grouped-query decode.
//
// A grouped-query decode step is a forward with the group's G query heads as the query rows of one
// 128-row tile (G <= 128 real rows) over one key/value head's keys, split into chunks and merged
// ("CS349E 第 11 讲 01_online_softmax.py", demo 2: split-KV states and their merge).  With so few
// real rows the work per key is small, so these configurations keep one query tile per CTA and
// more CTAs per SM than the prefill ones, to have enough K/V copies in flight:
//   d = 64 : Bc = 64, one query tile, 3-stage K/V ring (64 KB shared), 3 CTAs/SM; a grid that a fourth
//            CTA per SM would start in one wave (and three would not) takes a 2-stage ring with 4 CTAs/SM
//            instead: its CTAs then all run at once rather than leaving a short second wave
//   d = 128: Bc = 64, one query tile, 2-stage K/V ring (96 KB shared), 2 CTAs/SM (tensor memory allows
//            no more)
#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

using CfgDecD64 = FwdCfg<__nv_bfloat16, 64, 64, 1, 3, 3>;
using CfgDecD64OneWave = FwdCfg<__nv_bfloat16, 64, 64, 1, 2, 4>;
using CfgDecD128 = FwdCfg<__nv_bfloat16, 128, 64, 1, 2, 2>;

cudaError_t launch_fwd_decode(const FwdLaunch& a, int d, int sms) {
  if (d != 64) return launch_fwd<CfgDecD128>(a);
  const long long ctas = static_cast<long long>(a.BH) * a.n_split * ((a.Nq + CfgDecD64::BR - 1) / CfgDecD64::BR);
  if (ctas > static_cast<long long>(CfgDecD64::MINB) * sms && ctas <= static_cast<long long>(CfgDecD64OneWave::MINB) * sms)
    return launch_fwd<CfgDecD64OneWave>(a);
  return launch_fwd<CfgDecD64>(a);
}

// The two d = 64 configurations share Bc and the tile boxes.
static_assert(CfgDecD64OneWave::BC == CfgDecD64::BC && CfgDecD64OneWave::NQT == CfgDecD64::NQT, "same geometry");

FwdGeometry fwd_geometry_decode(int d) {
  if (d == 64)
    return FwdGeometry{64, 128, CfgDecD64::BC, 0, CfgDecD64::BR * CfgDecD64::NQT, CfgDecD64::MINB};
  return FwdGeometry{64, 128, CfgDecD128::BC, 0, CfgDecD128::BR * CfgDecD128::NQT, CfgDecD128::MINB};
}

}  // namespace fa
