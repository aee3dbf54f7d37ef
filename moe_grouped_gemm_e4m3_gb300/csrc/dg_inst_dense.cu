// dg_inst_dense.cu — instantiations of the GEMM kernel for the dense form (BN 128/256, BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_dense(const LaunchArgs& a) { return launch_mode<kDense>(a); }
}  // namespace dg
