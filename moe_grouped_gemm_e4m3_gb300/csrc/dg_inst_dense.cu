// dg_inst_dense.cu — instantiations of the GEMM kernel for the dense form (BN 128/256, BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_dense(const LaunchArgs& a) { return launch_mode<kDense>(a); }
int cluster_capacity_dense(int block_n, bool out_f32, int cluster) {
  return cluster_capacity_mode<kDense>(block_n, out_f32, cluster);
}
}  // namespace dg
