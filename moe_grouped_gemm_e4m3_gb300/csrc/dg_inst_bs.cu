// dg_inst_bs.cu — instantiations of the block-scaled (packed UE8M0) GEMM kernel: dense,
// contiguous and masked forms, BF16 and FP32 D.
#include "dg_launch.h"

namespace dg {
cudaError_t launch_bs(const LaunchArgs& a, Mode mode) {
  switch (mode) {
    case kDense: return a.out_f32 ? launch_bs_instance<kDense, true>(a) : launch_bs_instance<kDense, false>(a);
    case kContiguous:
      return a.out_f32 ? launch_bs_instance<kContiguous, true>(a) : launch_bs_instance<kContiguous, false>(a);
    default: return a.out_f32 ? launch_bs_instance<kMasked, true>(a) : launch_bs_instance<kMasked, false>(a);
  }
}
int cluster_capacity_bs(Mode mode, bool out_f32, int cluster) {
  const size_t smem = BsSmemPlan::kDynamicBytes;
  if (mode == kDense)
    return out_f32 ? clusters_resident(fp8_gemm_bs_kernel<kDense, true>, BsRoles::kThreads, smem, cluster)
                   : clusters_resident(fp8_gemm_bs_kernel<kDense, false>, BsRoles::kThreads, smem, cluster);
  if (mode == kContiguous)
    return out_f32 ? clusters_resident(fp8_gemm_bs_kernel<kContiguous, true>, BsRoles::kThreads, smem, cluster)
                   : clusters_resident(fp8_gemm_bs_kernel<kContiguous, false>, BsRoles::kThreads, smem, cluster);
  return 0;
}
}  // namespace dg
