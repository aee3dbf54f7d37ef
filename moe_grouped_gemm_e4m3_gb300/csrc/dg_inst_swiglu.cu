// dg_inst_swiglu.cu — instantiations of the masked GEMM fused with SwiGLU (BN 256): BF16/FP32 H, or
// H as FP8 codes with 1x128-group scales.
#include "dg_launch.h"

namespace dg {
cudaError_t launch_masked_swiglu(const LaunchArgs& a, bool fp8_h) {
  if (fp8_h) return launch_instance<256, kMasked, false, kSwigluFp8>(a);
  return a.out_f32 ? launch_instance<256, kMasked, true, kSwiglu>(a) : launch_instance<256, kMasked, false, kSwiglu>(a);
}
}  // namespace dg
