// dg_inst_swiglu.cu — instantiations of the masked GEMM fused with SwiGLU (BN 256, BF16/FP32 H).
#include "dg_launch.h"

namespace dg {
cudaError_t launch_masked_swiglu(const LaunchArgs& a) {
  return a.out_f32 ? launch_instance<256, kMasked, true, true>(a) : launch_instance<256, kMasked, false, true>(a);
}
}  // namespace dg
