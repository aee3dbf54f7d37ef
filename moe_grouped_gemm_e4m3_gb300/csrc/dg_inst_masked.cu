// dg_inst_masked.cu — instantiations of the GEMM kernel for the masked form (BN 128/256, BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_masked(const LaunchArgs& a) { return launch_mode<kMasked>(a); }
}  // namespace dg
