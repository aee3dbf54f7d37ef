// dg_inst_bs_kgrouped.cu — instantiations of the block-scaled (packed UE8M0) K-grouped GEMM
// (groups along K, MN-major A and B; BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_bs_kgrouped(const LaunchArgs& a) {
  return a.out_f32 ? launch_bs_instance<kKGrouped, true>(a) : launch_bs_instance<kKGrouped, false>(a);
}
}  // namespace dg
