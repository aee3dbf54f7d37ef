// dg_sf_transform.cu — scale-factor layout conversions: A's row-major FP32 scales to the MN-major
// layout, and FP32 power-of-two scales to the packed UE8M0 words of the block-scaled calls.
//
// The SM100 kernels of the pages take their scaling factors as UE8M0 codes packed four to an int32,
// and the library lists a helper that brings scale factors into that required layout ("DeepGEMM:
// İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri", tr.news.hada.io/topic?id=19459,
// § "GEMM arayüzü ve yerleşim kısıtları" and § "Yardımcı fonksiyonlar ve ortam değişkenleri").
// Two conversions. A's FP32 scales as a per-token quantiser writes them (row-major [G][M][nkb]) into the
// MN-major layout every call takes ([G][nkb][ldsa], rows m >= M zero). And this library's FP32 layouts
// into its packed layouts:
//   A: [G][nkb][ldsa] FP32 -> [G][ceil(nkb/4)][ldsa] int32 (MN-major; one thread per word, threads
//      along the row index so that reads and writes are coalesced);
//   B: [G][nnb][nkb] FP32 -> [G][nnb][ceil(nkb/4)] int32.
// Byte j of word q holds the code of K-block 4q + j; bytes past the last K-block are 127 (the scale
// 1). The code of a power of two 2^e in [2^-127, 2^127] is its FP32 exponent field (2^-127, an FP32
// subnormal, has field 0 = code 0). A zero scale (the padding rows of A's layout) packs as 127. Any
// other value — not a power of two, negative, infinite or NaN — sets kStatusBadScale in the device
// status word and packs as the code of the smallest power of two at or above its magnitude, clamped
// to [0, 254] (127 for NaN).
#include <cstdint>

#include <cuda_runtime.h>

#include "dg_launch.h"

namespace dg {

namespace {

__device__ __forceinline__ uint32_t e8m0_code(float s, int* status) {
  const uint32_t bits = __float_as_uint(s);
  const uint32_t expo = (bits >> 23) & 0xFFu, frac = bits & 0x7FFFFFu;
  if (s == 0.0f) return 127u;                                               // padding
  const bool neg = (bits >> 31) != 0u;
  if (!neg && expo > 0u && expo < 255u && frac == 0u) return expo;          // 2^(expo - 127)
  if (!neg && expo == 0u && frac == 0x400000u) return 0u;                   // 2^-127
  atomicOr(status, kStatusBadScale);
  if (expo == 255u) return frac != 0u ? 127u : 254u;                        // NaN / infinity
  if (expo == 0u) return frac > 0x400000u ? 1u : 0u;                        // subnormal magnitude
  const uint32_t up = expo + (frac != 0u ? 1u : 0u);                        // round the magnitude up
  return up > 254u ? 254u : up;
}

__global__ void sf_pack_a_kernel(const float* __restrict__ sf, int32_t* __restrict__ out, int G, int nkb,
                                 int ldsa, int* status) {
  const int nkq = (nkb + 3) / 4;
  const long long total = (long long)G * nkq * ldsa;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(i % ldsa);
    const long long gq = i / ldsa;
    const int q = (int)(gq % nkq);
    const long long g = gq / nkq;
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * q + j;
      const uint32_t c = kb < nkb ? e8m0_code(sf[(g * nkb + kb) * ldsa + m], status) : 127u;
      w |= c << (8 * j);
    }
    out[i] = (int32_t)w;
  }
}

__global__ void sf_pack_b_kernel(const float* __restrict__ sf, int32_t* __restrict__ out, long long rows, int nkb,
                                 int* status) {
  const int nkq = (nkb + 3) / 4;
  const long long total = rows * nkq;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int q = (int)(i % nkq);
    const long long r = i / nkq;
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * q + j;
      const uint32_t c = kb < nkb ? e8m0_code(sf[r * nkb + kb], status) : 127u;
      w |= c << (8 * j);
    }
    out[i] = (int32_t)w;
  }
}

// Row-major A scales [G][M][nkb] -> MN-major [G][nkb][ldsa], rows m >= M zero: one 32x32 tile of the
// (m, kb) plane per block of 32x8 threads, through shared memory so that both sides are coalesced.
__global__ void sf_a_to_mn_major_kernel(const float* __restrict__ in, float* __restrict__ out, int M, int nkb,
                                        int ldsa) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z;
  const int m0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const float* src = in + (size_t)g * M * nkb;
  float* dst = out + (size_t)g * nkb * ldsa;
  for (int r = threadIdx.y; r < 32; r += 8) {   // read rows m0 + r, columns k0 + threadIdx.x
    const int m = m0 + r, kb = k0 + threadIdx.x;
    tile[r][threadIdx.x] = (m < M && kb < nkb) ? src[(size_t)m * nkb + kb] : 0.0f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {   // write K-block k0 + r, rows m0 + threadIdx.x
    const int kb = k0 + r, m = m0 + threadIdx.x;
    if (kb < nkb && m < ldsa) dst[(size_t)kb * ldsa + m] = tile[threadIdx.x][r];
  }
}

int grid_for(long long words, int sms) {
  const long long blocks = (words + 255) / 256;
  const long long cap = 4LL * (sms > 0 ? sms : 1);
  return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_sf_pack_a(const float* sf, int32_t* out, int G, int nkb, int ldsa, int* status, int sms,
                             cudaStream_t stream) {
  const long long words = (long long)G * ((nkb + 3) / 4) * ldsa;
  if (words == 0) return cudaSuccess;
  sf_pack_a_kernel<<<grid_for(words, sms), 256, 0, stream>>>(sf, out, G, nkb, ldsa, status);
  return cudaGetLastError();
}

cudaError_t launch_sf_a_to_mn_major(const float* in, float* out, int G, int M, int nkb, int ldsa, cudaStream_t stream) {
  if ((long long)G * ldsa * nkb == 0) return cudaSuccess;
  const dim3 grid((unsigned)((ldsa + 31) / 32), (unsigned)((nkb + 31) / 32), (unsigned)G);
  sf_a_to_mn_major_kernel<<<grid, dim3(32, 8), 0, stream>>>(in, out, M, nkb, ldsa);
  return cudaGetLastError();
}

cudaError_t launch_sf_pack_b(const float* sf, int32_t* out, long long rows, int nkb, int* status, int sms,
                             cudaStream_t stream) {
  const long long words = rows * ((nkb + 3) / 4);
  if (words == 0) return cudaSuccess;
  sf_pack_b_kernel<<<grid_for(words, sms), 256, 0, stream>>>(sf, out, rows, nkb, status);
  return cudaGetLastError();
}

}  // namespace dg
