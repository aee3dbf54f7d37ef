// dg_inst_contiguous.cu — instantiations of the GEMM kernel for the contiguous form (BN 128/256, BF16/FP32 D).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_contiguous(const LaunchArgs& a) { return launch_mode<kContiguous>(a); }
int cluster_capacity_contiguous(int block_n, bool out_f32, int cluster) {
  return cluster_capacity_mode<kContiguous>(block_n, out_f32, cluster);
}
}  // namespace dg
