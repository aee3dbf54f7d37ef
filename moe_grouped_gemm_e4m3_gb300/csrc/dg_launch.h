// dg_launch.h — host-side interface between the C-ABI layer (dg_api.cu) and the per-mode kernel
// instantiations (dg_inst_*.cu), which are compiled as separate translation units in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_kernel.cuh"
#include "dg_kernel_bs.cuh"

namespace dg {

struct LaunchArgs {
  CUtensorMap tmA, tmB, tmD;
  GemmParams p;
  int block_n;   // 128 or 256
  bool out_f32;
  int grid;
  int cluster;   // > 1: launch as clusters of this many CTAs (cluster split-K)
  bool pdl;      // programmatic dependent launch (dg_set_pdl): may start before the previous kernel ends
  cudaStream_t stream;
};

// Pipeline depth per tile width (shared-memory plan of the kernel).
constexpr int stages_for(int block_n) { return block_n == 256 ? 4 : 6; }

// Columns per epilogue warp: 128 for wide tiles (8 epilogue warps), 64 for narrow ones (also 8,
// so that more warps hide the TMEM-load latency of the promotion).
constexpr int epi_cols_for(int block_n) { return block_n == 256 ? 128 : 64; }

// TMEM accumulator buffers in the ring: as many as the 512 TMEM columns hold.
constexpr int tmem_bufs_for(int block_n) { return 512 / block_n; }

cudaError_t launch_dense(const LaunchArgs& a);
cudaError_t launch_contiguous(const LaunchArgs& a);
cudaError_t launch_masked(const LaunchArgs& a);
// The K-grouped form (groups along K; FP32-scale kernel, MN-major A and B).
cudaError_t launch_kgrouped(const LaunchArgs& a);
// The masked form fused with SwiGLU (block_n 256, FP32-scale kernel); fp8_h: H as FP8 codes and
// 1x128-group scales.
cudaError_t launch_masked_swiglu(const LaunchArgs& a, bool fp8_h = false);
// The block-scaled kernel for packed UE8M0 scales (block_n is always 256).
cudaError_t launch_bs(const LaunchArgs& a, Mode mode);
// The block-scaled masked form fused with SwiGLU.
cudaError_t launch_bs_swiglu(const LaunchArgs& a);
// The block-scaled K-grouped form (MN-major A and B).
cudaError_t launch_bs_kgrouped(const LaunchArgs& a);
// FP32 scale factors to packed UE8M0 words (dg_sf_transform.cu). A: [G][nkb][ldsa] ->
// [G][ceil(nkb/4)][ldsa]; B: [rows][nkb] -> [rows][ceil(nkb/4)] (rows = G * nnb).
cudaError_t launch_sf_pack_a(const float* sf, int32_t* out, int G, int nkb, int ldsa, int* status, int sms,
                             cudaStream_t stream);
cudaError_t launch_sf_pack_b(const float* sf, int32_t* out, long long rows, int nkb, int* status, int sms,
                             cudaStream_t stream);
// A's scales row-major [G][M][nkb] -> MN-major [G][nkb][ldsa] (rows m >= M zero).
cudaError_t launch_sf_a_to_mn_major(const float* in, float* out, int G, int M, int nkb, int ldsa, cudaStream_t stream);
// How many clusters of `cluster` CTAs of the dense / contiguous instantiation for (block_n,
// out_f32) can be resident at once (0 if the query fails).
int cluster_capacity_dense(int block_n, bool out_f32, int cluster);
int cluster_capacity_contiguous(int block_n, bool out_f32, int cluster);
// The same for the block-scaled kernel (dense or contiguous).
int cluster_capacity_bs(Mode mode, bool out_f32, int cluster);

// Launches `kernel` on a 1-D grid of `grid` CTAs: as clusters of `cluster` CTAs when cluster > 1,
// and with programmatic stream serialization when pdl is set (the kernels wait for the previous
// kernel's results with griddepcontrol.wait before their first global read).
template <typename Kernel>
cudaError_t launch_kernel(Kernel kernel, const LaunchArgs& a, int threads, size_t smem_bytes) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (a.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)a.cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (a.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, a.tmA, a.tmB, a.tmD, a.p);
}

// Resident clusters of `cluster` CTAs of `kernel` (an occupancy query; nothing runs; 0 on error).
template <typename Kernel>
int clusters_resident(Kernel kernel, int threads, size_t smem_bytes, int cluster) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();   // clear the error: the caller falls back to the global split-K
    return 0;
  }
  return n;
}

// Launches one instantiation; sets its dynamic shared-memory limit on first use per device.
template <int BN, Mode MODE, bool OUT_F32, int SWIGLU = 0>
cudaError_t launch_instance(const LaunchArgs& a) {
  constexpr int STAGES = stages_for(BN);
  constexpr int EPI_COLS = epi_cols_for(BN);
  constexpr int NBUF = tmem_bufs_for(BN);
  using R = Roles<BN, EPI_COLS>;
  using Plan = SmemPlan<BN, STAGES, R::kEpiWarps, NBUF>;
  auto kernel = fp8_gemm_kernel<BN, EPI_COLS, STAGES, NBUF, MODE, OUT_F32, SWIGLU>;
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
  return launch_kernel(kernel, a, R::kThreads, Plan::kDynamicBytes);
}

// Resident clusters of `cluster` CTAs for one instantiation (an occupancy query; nothing runs).
template <int BN, Mode MODE, bool OUT_F32>
int cluster_capacity_instance(int cluster) {
  constexpr int STAGES = stages_for(BN);
  constexpr int EPI_COLS = epi_cols_for(BN);
  constexpr int NBUF = tmem_bufs_for(BN);
  using R = Roles<BN, EPI_COLS>;
  using Plan = SmemPlan<BN, STAGES, R::kEpiWarps, NBUF>;
  return clusters_resident(fp8_gemm_kernel<BN, EPI_COLS, STAGES, NBUF, MODE, OUT_F32, false>, R::kThreads,
                           Plan::kDynamicBytes, cluster);
}

template <Mode MODE>
int cluster_capacity_mode(int block_n, bool out_f32, int cluster) {
  if (block_n == 256)
    return out_f32 ? cluster_capacity_instance<256, MODE, true>(cluster) : cluster_capacity_instance<256, MODE, false>(cluster);
  return out_f32 ? cluster_capacity_instance<128, MODE, true>(cluster) : cluster_capacity_instance<128, MODE, false>(cluster);
}

template <Mode MODE, bool OUT_F32, bool SWIGLU = false>
cudaError_t launch_bs_instance(const LaunchArgs& a) {
  auto kernel = fp8_gemm_bs_kernel<MODE, OUT_F32, SWIGLU>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BsSmemPlan::kDynamicBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_kernel(kernel, a, BsRoles::kThreads, BsSmemPlan::kDynamicBytes);
}

template <Mode MODE>
cudaError_t launch_mode(const LaunchArgs& a) {
  if (a.block_n == 256) {
    return a.out_f32 ? launch_instance<256, MODE, true>(a) : launch_instance<256, MODE, false>(a);
  }
  return a.out_f32 ? launch_instance<128, MODE, true>(a) : launch_instance<128, MODE, false>(a);
}

}  // namespace dg
