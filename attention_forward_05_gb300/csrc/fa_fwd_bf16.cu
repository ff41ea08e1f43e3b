// fa_fwd_bf16.cu -- bf16 instantiations of the fused forward kernel.
//   d = 64 : Bc = 128, two 128-row query tiles per CTA, 4-stage K/V ring (160 KB shared)
//   d = 128: Bc = 128, two 128-row query tiles per CTA, 2-stage K/V ring (192 KB shared)
#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

using CfgBf16D64 = FwdCfg<__nv_bfloat16, 64, 128, 2, 4>;
using CfgBf16D128 = FwdCfg<__nv_bfloat16, 128, 128, 2, 2>;

cudaError_t launch_fwd_bf16_d64(const FwdLaunch& a) { return launch_fwd<CfgBf16D64>(a); }
cudaError_t launch_fwd_bf16_d128(const FwdLaunch& a) { return launch_fwd<CfgBf16D128>(a); }

}  // namespace fa
