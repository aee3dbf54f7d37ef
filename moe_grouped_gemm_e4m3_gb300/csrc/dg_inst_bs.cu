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
}  // namespace dg
