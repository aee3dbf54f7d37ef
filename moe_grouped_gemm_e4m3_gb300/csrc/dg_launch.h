// dg_launch.h — host-side interface between the C-ABI layer (dg_api.cu) and the per-mode kernel
// instantiations (dg_inst_*.cu), which are compiled as separate translation units in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_kernel.cuh"

namespace dg {

struct LaunchArgs {
  CUtensorMap tmA, tmB, tmD;
  GemmParams p;
  int block_n;   // 128 or 256
  bool out_f32;
  int grid;
  cudaStream_t stream;
};

// Pipeline depth per tile width (shared-memory plan of the kernel).
constexpr int stages_for(int block_n) { return block_n == 256 ? 4 : 6; }

cudaError_t launch_dense(const LaunchArgs& a);
cudaError_t launch_contiguous(const LaunchArgs& a);
cudaError_t launch_masked(const LaunchArgs& a);

// Launches one instantiation; sets its dynamic shared-memory limit on first use per device.
template <int BN, Mode MODE, bool OUT_F32>
cudaError_t launch_instance(const LaunchArgs& a) {
  constexpr int STAGES = stages_for(BN);
  using Plan = SmemPlan<BN, STAGES>;
  auto kernel = fp8_gemm_kernel<BN, STAGES, MODE, OUT_F32>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Plan::kDynamicBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  kernel<<<a.grid, Threads<BN>::kCount, Plan::kDynamicBytes, a.stream>>>(a.tmA, a.tmB, a.tmD, a.p);
  return cudaGetLastError();
}

template <Mode MODE>
cudaError_t launch_mode(const LaunchArgs& a) {
  if (a.block_n == 256) {
    return a.out_f32 ? launch_instance<256, MODE, true>(a) : launch_instance<256, MODE, false>(a);
  }
  return a.out_f32 ? launch_instance<128, MODE, true>(a) : launch_instance<128, MODE, false>(a);
}

}  // namespace dg
