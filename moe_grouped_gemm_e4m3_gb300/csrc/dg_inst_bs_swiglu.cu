// dg_inst_bs_swiglu.cu — instantiations of the block-scaled (packed UE8M0) masked GEMM fused with
// SwiGLU (BF16/FP32 H).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_bs_swiglu(const LaunchArgs& a) {
  return a.out_f32 ? launch_bs_instance<kMasked, true, true>(a) : launch_bs_instance<kMasked, false, true>(a);
}
}  // namespace dg
