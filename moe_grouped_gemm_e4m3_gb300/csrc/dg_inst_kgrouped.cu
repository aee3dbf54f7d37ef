// dg_inst_kgrouped.cu — instantiations of the GEMM kernel for the K-grouped form (BN 128/256, BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_kgrouped(const LaunchArgs& a) { return launch_mode<kKGrouped>(a); }
}  // namespace dg
