// dg_api.cu — the C ABI of libdg (declared in include/dg.h): argument validation, tile
// configuration, TMA descriptor encoding, the split-K workspace, the device status word and the
// launch of the sm_103a kernels. No GEMM arithmetic happens on the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "dg.h"
#include "dg_launch.h"

static_assert(dg::kStatusTimeout == DG_DEV_TIMEOUT, "status bit mismatch");
static_assert(dg::kStatusBadGroup == DG_DEV_BAD_GROUP_INDEX, "status bit mismatch");
static_assert(dg::kStatusBadMaskedM == DG_DEV_BAD_MASKED_M, "status bit mismatch");
static_assert(dg::kStatusBadScale == DG_DEV_BAD_SCALE, "status bit mismatch");

// The device status word: one per device context, read and cleared by dg_get_device_status().
__device__ int g_dg_device_status;

namespace {

thread_local std::string t_last_error;

dg_status fail(dg_status s, const std::string& msg) {
  t_last_error = msg;
  return s;
}

dg_status fail_cuda(cudaError_t e, const char* what) {
  return fail(DG_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 16;
// Most K ranges a tile of a last, partial wave is cut into (the kernel decides per launch whether
// splitting pays). DG_TAIL_SPLITS sets the initial value and
// dg_set_tail_splits() changes it; 1 switches the tail split off.
constexpr int kTailSplits = 4;
std::atomic<int> g_tail_splits{-1};   // -1: not yet initialised from DG_TAIL_SPLITS

int clamp_tail_splits(int x) { return x < 1 ? 1 : (x > kMaxSplits ? kMaxSplits : x); }

// Split-K inside thread-block clusters (dense and contiguous, FP32 scales): on unless
// DG_CLUSTER_SPLIT=0 or dg_set_cluster_split(0).
std::atomic<int> g_cluster_split{-1};
bool cluster_split_setting() {
  int v = g_cluster_split.load();
  if (v < 0) {
    const char* e = std::getenv("DG_CLUSTER_SPLIT");
    int expected = -1;
    g_cluster_split.compare_exchange_strong(expected, (e && std::atoi(e) == 0) ? 0 : 1);
    v = g_cluster_split.load();
  }
  return v != 0;
}

// Pairs of CTAs sharing B tiles through TMA multicast (dense and contiguous, FP32 scales, BN = 256,
// no split-K): off unless DG_PAIR_B=1 or dg_set_pair_b(1). Measured on GB300, the FP32-scale kernel
// is bound by its per-K-block TMEM round trip, not by the L2 feed that pairing relieves, and paired
// launches lose the tail split: 4096x7168x16384 397 us single, 419 us paired.
// Programmatic dependent launch: off unless DG_PDL=1 or dg_set_pdl(1).
std::atomic<int> g_pdl{-1};
bool pdl_setting() {
  int v = g_pdl.load();
  if (v < 0) {
    const char* e = std::getenv("DG_PDL");
    int expected = -1;
    g_pdl.compare_exchange_strong(expected, (e && std::atoi(e) != 0) ? 1 : 0);
    v = g_pdl.load();
  }
  return v != 0;
}

std::atomic<int> g_pair_b{-1};
bool pair_b_setting() {
  int v = g_pair_b.load();
  if (v < 0) {
    const char* e = std::getenv("DG_PAIR_B");
    int expected = -1;
    g_pair_b.compare_exchange_strong(expected, (e && std::atoi(e) != 0) ? 1 : 0);
    v = g_pair_b.load();
  }
  return v != 0;
}

// Largest cluster of the cluster split-K: the portable limit.
constexpr int kMaxClusterSplit = 8;

// Resident clusters of `splits` CTAs for an instantiation, queried once per device.
int cluster_capacity(int mode, int block_n, bool out_f32, int splits, bool block_scaled) {
  static std::mutex mu;
  static int cache[kMaxDevices][2][2][2][2][kMaxClusterSplit + 1];
  static bool have[kMaxDevices][2][2][2][2][kMaxClusterSplit + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (splits < 2 || splits > kMaxClusterSplit || (mode != dg::kDense && mode != dg::kContiguous)) return 0;
  const int k = block_scaled ? 1 : 0, m = mode == dg::kDense ? 0 : 1, f = out_f32 ? 1 : 0;
  const int b = block_n == 256 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev][k][m][b][f][splits]) {
    int n;
    if (block_scaled)
      n = dg::cluster_capacity_bs(static_cast<dg::Mode>(mode), out_f32, splits);
    else
      n = m == 0 ? dg::cluster_capacity_dense(block_n, out_f32, splits)
                 : dg::cluster_capacity_contiguous(block_n, out_f32, splits);
    cache[dev][k][m][b][f][splits] = n;
    have[dev][k][m][b][f][splits] = true;
  }
  return cache[dev][k][m][b][f][splits];
}

// Time limit of the kernels' pipeline waits, in microseconds, carried in bits 8..31 of the kernel
// flags word: default 2 s; DG_WAIT_LIMIT_US sets the initial value, dg_set_wait_limit_us() changes it.
constexpr long long kDefaultWaitLimitUs = 2000000;
constexpr long long kMaxWaitLimitUs = (1LL << (32 - dg::kWaitLimitShift)) - 1;   // ~16.7 s
std::atomic<long long> g_wait_limit_us{-1};   // -1: not yet initialised from DG_WAIT_LIMIT_US

long long clamp_wait_limit(long long us) {
  return us < 0 ? kDefaultWaitLimitUs : (us > kMaxWaitLimitUs ? kMaxWaitLimitUs : us);
}

long long wait_limit_setting() {
  long long v = g_wait_limit_us.load();
  if (v < 0) {
    const char* e = std::getenv("DG_WAIT_LIMIT_US");
    long long expected = -1;
    g_wait_limit_us.compare_exchange_strong(expected, clamp_wait_limit(e ? std::atoll(e) : kDefaultWaitLimitUs));
    v = g_wait_limit_us.load();
  }
  return v;
}

// The wait limit's bits of the kernel flags word.
int wait_limit_flags() { return (int)((uint32_t)wait_limit_setting() << dg::kWaitLimitShift); }

int tail_splits_setting() {
  int v = g_tail_splits.load();
  if (v < 0) {
    const char* e = std::getenv("DG_TAIL_SPLITS");
    int expected = -1;
    g_tail_splits.compare_exchange_strong(expected, clamp_tail_splits(e ? std::atoi(e) : kTailSplits));
    v = g_tail_splits.load();
  }
  return v;
}

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int* status = nullptr;      // device address of g_dg_device_status
  float* workspace = nullptr; // split-K partial tiles
  size_t workspace_floats = 0;
  int* counters = nullptr;    // split-K arrival counters
  size_t counter_count = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<int> g_num_sms_cap{-1};  // -1: not yet initialised from DG_NUM_SMS; 0: no cap

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int num_sms_cap() {
  int c = g_num_sms_cap.load();
  if (c < 0) {
    const char* env = std::getenv("DG_NUM_SMS");
    int v = env ? std::atoi(env) : 0;
    if (v < 0) v = 0;
    int expected = -1;
    g_num_sms_cap.compare_exchange_strong(expected, v);
    c = g_num_sms_cap.load();
  }
  return c;
}

// State of the current device, initialised on first use.
dg_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DG_ERR_UNSUPPORTED, "device ordinal beyond 64");
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(DG_ERR_UNSUPPORTED, "libdg is built for sm_103a (GB300); this device is sm_" +
                                          std::to_string(major) + std::to_string(minor));
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_dg_device_status)) != cudaSuccess)
      return fail_cuda(e, "cudaGetSymbolAddress(status)");
    st.status = static_cast<int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return DG_OK;
}

int effective_sms(const DeviceState& st) {
  const int cap = num_sms_cap();
  return (cap > 0 && cap < st.sm_count) ? cap : st.sm_count;
}

// ---------------------------------------------------------------------------------------------
// Tile configuration: a static heuristic keyed on the problem shape and the SM count.

struct Config {
  int block_n;
  int stages;
  int splits;
  int kb_per_split;
  int tiles;       // output tiles (masked: upper bound)
  int grid;
  int raster_m;
};

Config choose_config(int mode, int rows, int N, int K, int G, int num_sms, bool block_scaled = false) {
  // Cost model calibrated on GB300 (sm_103a), times in microseconds per CTA:
  //  * compute: one K-block (BM=128, BK=128) costs ~0.55 (BN=256) or ~0.50 (BN=128: an N=128 MMA
  //    takes as long as an N=256 one, for half the work);
  //  * memory: a CTA streams ~48 GB/s when its operands come from HBM; operands shared by other
  //    tiles in flight (A across n-blocks, B across m-blocks) come from L2 and cost no HBM time;
  //  * split-K: the last split reads every partial tile back, ~0.6 (BN=128) / ~1.0 (BN=256) per split;
  //  * a tile's prologue/epilogue: ~1.5;
  //  * the block-scaled kernel (packed UE8M0 scales) has no per-K-block promotion: ~0.30 per
  //    K-block, BN = 256 only.
  // Split-K is considered only while all units fit in one wave (more waves never shorten the
  // critical path). The HBM time of the operands bounds the estimate from below.
  constexpr double kTileUs = 1.5, kCtaGBs = 48.0, kHbmGBs = 6000.0;
  Config c{};
  const int nkb = ceil_div(K, 128);
  const int rows_total = rows * (mode == dg::kMasked ? G : 1);
  const int m_blocks = ceil_div(rows, 128) * (mode == dg::kMasked ? G : 1);
  const double bytes = (double)rows_total * K + (double)(mode == dg::kDense ? 1 : G) * N * K + 2.0 * rows_total * N;
  int bn = N > 128 ? 256 : 128;
  int best_s = 1;
  double best_t = 1e300;
  const int max_s = (mode == dg::kMasked) ? 1 : kMaxSplits;
  if (block_scaled) bn = 256;
  for (int cand_bn = 128; cand_bn <= 256; cand_bn += 128) {
    if (cand_bn == 256 && N <= 128 && !block_scaled) continue;
    if (cand_bn == 128 && block_scaled) continue;
    const int n_blocks = ceil_div(N, cand_bn);
    const int tiles = m_blocks * n_blocks;
    const double t_compute = block_scaled ? 0.30 : (cand_bn == 256 ? 0.55 : 0.50);
    const double t_red = cand_bn == 256 ? 1.0 : 0.6;
    for (int s = 1; s <= max_s; ++s) {
      const int kps = ceil_div(nkb, s);
      const int se = ceil_div(nkb, kps);
      if (se != s) continue;
      const long long units = (long long)tiles * se;
      if (se > 1 && units > num_sms) break;
      const long long active = units < num_sms ? units : num_sms;
      // unique HBM bytes per K-block of one tile: its share of A and of B
      const double a_kb = (double)(rows < 128 ? rows : 128) * 128.0 / n_blocks;
      const double b_kb = (double)cand_bn * 128.0 / (m_blocks < 16 ? m_blocks : 16);
      const double cta_gbs = kCtaGBs < kHbmGBs / active ? kCtaGBs : kHbmGBs / active;
      const double t_mem = (a_kb + b_kb) / (cta_gbs * 1e3);
      const double t_kb = t_compute > t_mem ? t_compute : t_mem;
      const double waves = (double)((units + num_sms - 1) / num_sms);
      double t = waves * (kps * t_kb + kTileUs) + (se > 1 ? t_red * se : 0.0);
      const double t_hbm = bytes / (kHbmGBs * 1e3);
      if (t < t_hbm) t = t_hbm;
      if (t < best_t - 1e-9) { best_t = t; best_s = se; bn = cand_bn; }
    }
  }
  const int tiles = m_blocks * ceil_div(N, bn);
  // Tuning overrides (environment): DG_BLOCK_N in {128, 256} and DG_SPLITS >= 1 (dense and
  // contiguous only; a split that would exceed one wave of units is still allowed here).
  int bn_final = bn, tiles_final = tiles;
  if (const char* e = block_scaled ? nullptr : std::getenv("DG_BLOCK_N")) {
    const int v = std::atoi(e);
    if (v == 128 || v == 256) { bn_final = v; tiles_final = m_blocks * ceil_div(N, v); }
  }
  if (mode != dg::kMasked) {
    if (const char* e = std::getenv("DG_SPLITS")) {
      const int v = std::atoi(e);
      if (v >= 1 && v <= kMaxSplits) best_s = v < nkb ? v : nkb;
    }
  }
  c.kb_per_split = ceil_div(nkb, best_s);
  c.splits = ceil_div(nkb, c.kb_per_split);
  c.block_n = bn_final;
  c.stages = block_scaled ? dg::BsSmemPlan::kStages : dg::stages_for(bn_final);
  c.tiles = tiles_final;
  const long long units = (long long)tiles_final * c.splits;
  c.grid = (int)(units < num_sms ? units : num_sms);
  if (c.grid < 1) c.grid = 1;
  const int mb = ceil_div(rows, 128);
  c.raster_m = mb < 16 ? (mb > 0 ? mb : 1) : 16;
  return c;
}

// Split-K in clusters needs every tile's cluster resident at once. When the chosen split count does
// not fit, one or two fewer splits may; take the largest that does. The exchange through
// distributed shared memory then saves more than the longer K range of each CTA costs: on
// 64x2112x7168, 7 splits through the global workspace versus 6 in clusters. An explicit DG_SPLITS is
// left alone.
void fit_cluster_splits(Config& c, int mode, int K, bool block_scaled, bool out_f32) {
  if ((mode != dg::kDense && mode != dg::kContiguous) || c.splits < 3) return;
  if (!cluster_split_setting() || std::getenv("DG_SPLITS")) return;
  if (c.splits <= kMaxClusterSplit && cluster_capacity(mode, c.block_n, out_f32, c.splits, block_scaled) >= c.tiles)
    return;
  const int nkb = ceil_div(K, 128);
  for (int s = c.splits - 1; s >= 2 && s >= c.splits - 2; --s) {
    const int kps = ceil_div(nkb, s), eff = ceil_div(nkb, kps);
    if (eff >= 2 && eff <= kMaxClusterSplit && cluster_capacity(mode, c.block_n, out_f32, eff, block_scaled) >= c.tiles) {
      c.splits = eff;
      c.kb_per_split = kps;
      c.grid = c.tiles * eff;
      return;
    }
  }
}

// Whether a call with this configuration runs its split-K in clusters: dense or contiguous (either
// kernel), 2..8 splits, one work unit per CTA, and every tile's cluster resident at once.
bool use_cluster_split(const Config& c, int mode, bool out_f32, bool block_scaled, bool swiglu) {
  return !swiglu && (mode == dg::kDense || mode == dg::kContiguous) && c.splits > 1 &&
         c.splits <= kMaxClusterSplit && cluster_split_setting() && c.grid == c.tiles * c.splits &&
         cluster_capacity(mode, c.block_n, out_f32, c.splits, block_scaled) >= c.tiles;
}

// Whether a call with this configuration runs as pairs of CTAs sharing B (kFlagPairB): dense or
// contiguous with FP32 scales and K-major operands, BN = 256, no split-K, at least two 128-row
// blocks, and clusters of 2 can be resident. Returns the resident clusters of 2 (0: no pairing).
int pair_clusters(const Config& c, int mode, int rows, bool out_f32, bool block_scaled, bool swiglu, bool mn_layout) {
  if (!pair_b_setting() || block_scaled || swiglu || mn_layout) return 0;
  if ((mode != dg::kDense && mode != dg::kContiguous) || c.block_n != 256 || c.splits != 1 || ceil_div(rows, 128) < 2)
    return 0;
  return cluster_capacity(mode, 256, out_f32, 2, false);
}

// Read on every call (a debugging aid), so that a process can switch it on and off.
bool print_configs() {
  const char* e = std::getenv("DG_PRINT_CONFIGS");
  return e && std::atoi(e) != 0;
}

// ---------------------------------------------------------------------------------------------
// TMA descriptors

dg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapL2promotion promo,
                    const char* what, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DG_ERR_CUDA, std::string("cuTensorMapEncodeTiled(") + what + ") failed: " + std::to_string((int)r));
  return DG_OK;
}

// Grows the split-K workspace of the device to at least `floats` partial values and `counters`
// arrival counters (new counters are zeroed on `stream`).
dg_status ensure_workspace(DeviceState& st, size_t floats, size_t counters, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  cudaError_t e;
  if (st.workspace_floats < floats) {
    if (st.workspace) cudaFree(st.workspace);
    st.workspace = nullptr;
    st.workspace_floats = 0;
    if ((e = cudaMalloc(&st.workspace, floats * sizeof(float))) != cudaSuccess) return fail_cuda(e, "cudaMalloc(workspace)");
    st.workspace_floats = floats;
  }
  if (st.counter_count < counters) {
    if (st.counters) cudaFree(st.counters);
    st.counters = nullptr;
    st.counter_count = 0;
    if ((e = cudaMalloc(&st.counters, counters * sizeof(int))) != cudaSuccess) return fail_cuda(e, "cudaMalloc(counters)");
    if ((e = cudaMemsetAsync(st.counters, 0, counters * sizeof(int), stream)) != cudaSuccess)
      return fail_cuda(e, "cudaMemsetAsync(counters)");
    st.counter_count = counters;
  }
  return DG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The allocation-free call's fixed split-K scratch: its capacity, and the device address of the
// array on the current device (the array and this lookup are defined with the entry point at the end
// of this file).
constexpr size_t kNoAllocCounterBytes = 4096 * sizeof(int);   // 4096 output tiles
constexpr size_t kNoAllocWorkspaceBytes = size_t(20) << 20;   // 20 MiB of FP32 partials
dg_status noalloc_scratch(void** out);

// Common implementation of the six GEMM entry points.
//   mode dense: rows = M, G = 1;  contiguous: rows = M_total;  masked: rows = M_max (per group).
//   sA/sB are FP32 scales, or (block_scaled) packed UE8M0 words: sA [G][ceil(nkb/4)][ldsa] and
//   sB [G][nnb][ceil(nkb/4)] int32.
//   C (dense, FP32 D only): D = C + A·Bᵀ. C may be D itself; otherwise it is copied into D first.
//   noalloc (dense, BF16, FP32 scales only): split-K scratch comes from the fixed array of the
//   allocation-free entry point instead of the lazily grown workspace; a shape that needs more
//   than it holds returns DG_ERR_UNSUPPORTED.
dg_status run_gemm(int mode, bool out_f32, const uint8_t* A, const void* sA, const uint8_t* B, const void* sB,
                   const int32_t* idx, void* D, int rows, int N, int K, int G, cudaStream_t stream,
                   bool block_scaled = false, const float* C = nullptr, bool accumulate = false,
                   bool swiglu = false, bool a_mn = false, bool b_mn = false, bool noalloc = false,
                   float* h_scales = nullptr) {
  t_last_error.clear();
  // h_scales: the fused SwiGLU writes H as FP8 codes (D, bytes) and these 1x128-group scales
  const bool quant_h = h_scales != nullptr;
  if (quant_h && (!swiglu || out_f32 || block_scaled))
    return fail(DG_ERR_INVALID_ARG, "FP8 H: the fused SwiGLU with FP32 scales");
  if (quant_h && !aligned(h_scales, 4)) return fail(DG_ERR_ALIGNMENT, "sH must be 4-byte aligned");
  if (rows < 0 || N < 0 || K < 0 || G < 0) return fail(DG_ERR_INVALID_ARG, "negative size");
  if (mode != dg::kDense && G < 1 && rows > 0) {
    if (G == 0) return DG_OK;
  }
  if (accumulate && (!C || !out_f32 || mode != dg::kDense))
    return fail(DG_ERR_INVALID_ARG, "the accumulating form needs a C pointer and FP32 D (dense only)");
  if (swiglu && (mode != dg::kMasked || accumulate))
    return fail(DG_ERR_INVALID_ARG, "the fused SwiGLU form is masked and not accumulating");
  if (swiglu && N % 256 != 0)
    return fail(DG_ERR_ALIGNMENT, "fused SwiGLU: B must hold 2I rows per group with I a multiple of 128");
  if ((a_mn || b_mn) && mode != dg::kDense)
    return fail(DG_ERR_INVALID_ARG, "the NN/TN/TT layouts are dense");
  if (rows == 0 || N == 0 || G == 0) return DG_OK;
  if (K == 0) return fail(DG_ERR_INVALID_ARG, "K must be positive");
  if (!A || !sA || !B || !sB || !D) return fail(DG_ERR_INVALID_ARG, "null tensor pointer");
  if (a_mn && rows % 16 != 0) return fail(DG_ERR_ALIGNMENT, "A stored [K,M]: M must be a multiple of 16");
  if (b_mn && N % 16 != 0) return fail(DG_ERR_ALIGNMENT, "B stored [K,N]: N must be a multiple of 16");
  if (mode != dg::kDense && !idx) return fail(DG_ERR_INVALID_ARG, mode == dg::kMasked ? "null masked_m" : "null m_indices");
  if (K % 16 != 0) return fail(DG_ERR_ALIGNMENT, "K must be a multiple of 16 (16-byte rows of E4M3 A and B)");
  if (N % (out_f32 ? 4 : 8) != 0)
    return fail(DG_ERR_ALIGNMENT, out_f32 ? "N must be a multiple of 4 (16-byte rows of FP32 D)"
                                          : "N must be a multiple of 8 (16-byte rows of BF16 D)");
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
    return fail(DG_ERR_ALIGNMENT, "A, B and D must be 16-byte aligned");
  if (!aligned(sA, 4) || !aligned(sB, 4) || (idx && !aligned(idx, 4)))
    return fail(DG_ERR_ALIGNMENT, "sA, sB and index tensors must be 4-byte aligned");
  if (accumulate) {
    if (!aligned(C, 16)) return fail(DG_ERR_ALIGNMENT, "C must be 16-byte aligned");
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(C), d0 = reinterpret_cast<uintptr_t>(D);
    const uintptr_t bytes = (uintptr_t)rows * (uintptr_t)N * sizeof(float);
    if (c0 != d0 && c0 < d0 + bytes && d0 < c0 + bytes)
      return fail(DG_ERR_INVALID_ARG, "C and D overlap without being the same matrix");
  }
  const long long rows_total = (long long)rows * (mode == dg::kMasked ? G : 1);
  const long long b_rows = (long long)N * (mode == dg::kDense ? 1 : G);
  if (rows_total > INT_MAX - 256 || b_rows > INT_MAX - 256 || K > INT_MAX - 256)
    return fail(DG_ERR_UNSUPPORTED, "a tensor extent exceeds 2^31 - 257");

  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  const int sms = effective_sms(*st);
  Config cfg = choose_config(mode, rows, N, K, mode == dg::kDense ? 1 : G, sms, block_scaled);
  if (!swiglu) fit_cluster_splits(cfg, mode, K, block_scaled, out_f32);
  const int d_cols = swiglu ? N / 2 : N;   // width of D (fused SwiGLU: H has I = N/2 columns)
  if (swiglu) {
    // one tile = 128 gate rows + 128 up rows of B; no host split-K (the tail split may still apply)
    cfg.block_n = 256;
    cfg.stages = block_scaled ? dg::BsSmemPlan::kStages : dg::stages_for(256);
    cfg.splits = 1;
    cfg.kb_per_split = ceil_div(K, 128);
    cfg.tiles = ceil_div(rows, 128) * G * (d_cols / 128);
    cfg.grid = cfg.tiles < sms ? cfg.tiles : sms;
    if (cfg.grid < 1) cfg.grid = 1;
  }
  if ((long long)cfg.tiles * cfg.splits > INT_MAX / 2) return fail(DG_ERR_UNSUPPORTED, "too many tiles");

  dg::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  dg::GemmParams& p = a.p;
  p.M = rows;
  p.N = N;
  p.K = K;
  p.G = mode == dg::kDense ? 1 : G;
  p.nkb = ceil_div(K, 128);
  p.nnb = ceil_div(N, 128);
  p.ldsa = dg_get_tma_aligned_size(rows, 4);
  p.num_m_blocks = ceil_div(rows, 128);
  p.num_n_blocks = swiglu ? d_cols / 128 : ceil_div(N, cfg.block_n);
  p.swiglu_i = swiglu ? d_cols : 0;
  p.flags = (a_mn ? dg::kFlagAMN : 0) | (b_mn ? dg::kFlagBMN : 0) | (accumulate ? dg::kFlagAccumulate : 0) |
            wait_limit_flags();
  p.num_splits = cfg.splits;
  p.kb_per_split = cfg.kb_per_split;
  p.num_tiles = mode == dg::kMasked ? 0 : cfg.tiles;   // masked: counted on the device
  p.raster_m = (int16_t)cfg.raster_m;
  // Tail split (no host split-K; the fused SwiGLU included: its split-K step reduces the gate and
  // up partials before H is formed): the workspace holds at most one wave of split units, the
  // counters one per CTA.
  const bool tail = cfg.splits == 1 && tail_splits_setting() > 1;
  p.tail_splits = (int16_t)(tail ? tail_splits_setting() : 1);
  // (the block-scaled kernel reads these as its packed UE8M0 words)
  p.sA = static_cast<const float*>(sA);
  p.sB = static_cast<const float*>(sB);
  p.m_indices = mode == dg::kContiguous ? idx : nullptr;
  p.masked_m = mode == dg::kMasked ? idx : nullptr;
  p.D = D;
  p.status = st->status;
  if (quant_h) p.h_scales = h_scales;   // (masked: no m_indices)
  if (accumulate && static_cast<const void*>(C) != D) {
    cudaError_t ce = cudaMemcpyAsync(D, C, (size_t)rows * N * sizeof(float), cudaMemcpyDeviceToDevice, stream);
    if (ce != cudaSuccess) return fail_cuda(ce, "cudaMemcpyAsync(C -> D)");
  }
  // Split-K in clusters: the splits of a tile are one cluster of CTAs that reduce through
  // distributed shared memory (no workspace, no counters) when every tile's cluster can be resident
  // at once and each CTA gets exactly one work unit.
  const bool cluster = use_cluster_split(cfg, mode, out_f32, block_scaled, swiglu);
  // Pairs of CTAs share B tiles (kFlagPairB): the persistent units are pairs of 128-row blocks by
  // BN columns, walked by clusters of 2; no tail split.
  const int pair_cap = cluster ? 0 : pair_clusters(cfg, mode, rows, out_f32, block_scaled, swiglu, a_mn || b_mn);
  const bool pair = pair_cap > 0;
  if (pair) {
    const int m_pairs = ceil_div(ceil_div(rows, 128), 2);
    const long long units = (long long)m_pairs * ceil_div(N, cfg.block_n);
    p.flags |= dg::kFlagPairB;
    p.num_tiles = (int)units;
    p.raster_m = (int16_t)(m_pairs < 8 ? m_pairs : 8);
    p.tail_splits = 1;
    a.cluster = 2;
    cfg.grid = 2 * (int)(units < pair_cap ? units : pair_cap);
  }
  if (cluster) {
    p.flags |= dg::kFlagClusterSplit;
    a.cluster = cfg.splits;
  } else if (!pair && (cfg.splits > 1 || tail)) {
    const size_t floats = cfg.splits > 1 ? (size_t)cfg.tiles * cfg.splits * 128 * cfg.block_n
                                         : (size_t)cfg.grid * 128 * cfg.block_n;
    const size_t counters = cfg.splits > 1 ? (size_t)cfg.tiles : (size_t)cfg.grid;
    if (noalloc) {
      if (counters * sizeof(int) > kNoAllocCounterBytes || floats * sizeof(float) > kNoAllocWorkspaceBytes)
        return fail(DG_ERR_UNSUPPORTED,
                    "dg_fp8_gemm_nt_noalloc: this shape needs " + std::to_string(floats * sizeof(float)) +
                        " bytes of split-K partials and " + std::to_string(counters) + " counters; the fixed scratch holds " +
                        std::to_string(kNoAllocWorkspaceBytes) + " bytes and " +
                        std::to_string(kNoAllocCounterBytes / sizeof(int)) + " counters (use dg_fp8_gemm_nt)");
      void* scratch = nullptr;
      if ((s = noalloc_scratch(&scratch)) != DG_OK) return s;
      unsigned char* base = static_cast<unsigned char*>(scratch);
      p.counters = reinterpret_cast<int*>(base);
      p.workspace = reinterpret_cast<float*>(base + kNoAllocCounterBytes);
      // The array keeps whatever the previous call left; the arrival counters must start at zero.
      const cudaError_t me = cudaMemsetAsync(p.counters, 0, counters * sizeof(int), stream);
      if (me != cudaSuccess) return fail_cuda(me, "cudaMemsetAsync(noalloc counters)");
    } else {
      if ((s = ensure_workspace(*st, floats, counters, stream)) != DG_OK) return s;
      p.workspace = st->workspace;
      p.counters = st->counters;
    }
  }

  if (a_mn) {   // A stored [K, M]: M contiguous
    if ((s = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)rows_total, (uint64_t)K, (uint64_t)rows_total,
                       128, 128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A")) != DG_OK)
      return s;
  } else if ((s = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)K, (uint64_t)rows_total, (uint64_t)K,
                            128, 128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A")) != DG_OK) {
    return s;
  }
  if (b_mn) {   // B stored [K, N]: N contiguous, boxes of 128 N-bytes x 128 K-rows
    if ((s = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)b_rows, (uint64_t)K, (uint64_t)b_rows, 128,
                       128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B")) != DG_OK)
      return s;
  } else if ((s = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)K, (uint64_t)b_rows, (uint64_t)K, 128,
                            (uint32_t)(swiglu ? 128 : (pair ? cfg.block_n / 2 : cfg.block_n)),
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B")) != DG_OK) {
    return s;
  }
  if (quant_h) {   // (FP8 H is written with plain stores; the map only has to be valid)
    s = encode_2d(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_UINT8, D, (uint64_t)d_cols, (uint64_t)rows_total, (uint64_t)d_cols,
                  32, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE, "H");
  } else if (out_f32) {
    s = encode_2d(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, (uint64_t)d_cols, (uint64_t)rows_total,
                  (uint64_t)d_cols * 4, 16, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE, "D", CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    s = encode_2d(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)d_cols, (uint64_t)rows_total,
                  (uint64_t)d_cols * 2, 32, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE, "D", CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (s != DG_OK) return s;

  a.block_n = cfg.block_n;
  a.out_f32 = out_f32;
  a.grid = cfg.grid;
  a.stream = stream;
  a.pdl = pdl_setting();
  if (print_configs()) {
    static const char* names[3] = {"dense", "contiguous", "masked"};
    std::fprintf(stderr, "[dg] %s%s%s%s rows=%d N=%d K=%d G=%d: BM=128 BN=%d stages=%d splits=%d%s grid=%d tiles=%d\n",
                 names[mode], block_scaled ? "/ue8m0" : "", swiglu ? "/swiglu" : "", out_f32 ? "/f32" : "", rows, N, K,
                 p.G, cfg.block_n, cfg.stages, cfg.splits, cluster ? " (cluster)" : (pair ? " (pairs sharing B)" : ""),
                 cfg.grid, cfg.tiles);
  }
  cudaError_t e;
  if (swiglu) {
    e = block_scaled ? dg::launch_bs_swiglu(a) : dg::launch_masked_swiglu(a, quant_h);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return DG_OK;
  }
  if (block_scaled) {
    e = dg::launch_bs(a, static_cast<dg::Mode>(mode));
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return DG_OK;
  }
  switch (mode) {
    case dg::kDense: e = dg::launch_dense(a); break;
    case dg::kContiguous: e = dg::launch_contiguous(a); break;
    default: e = dg::launch_masked(a); break;
  }
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return DG_OK;
}

// The K-grouped GEMM: A stored [K_total, M], B stored [K_total, N] (both MN-major), D [G, M, N];
// group g sums the K-blocks [offsets[g], offsets[g+1]) / 128 (offsets on the device).
// block_scaled: sA/sB are packed UE8M0 words (sA [ceil(nkb/4)][ldsa], sB [ceil(N/128)][ceil(nkb/4)],
// nkb = K_total/128), run on the block-scaled kernel (BN = 256).
dg_status run_k_grouped(bool out_f32, const uint8_t* A, const void* sA, const uint8_t* B, const void* sB,
                        const int32_t* offsets, void* D, int G, int M, int N, int K_total, cudaStream_t stream,
                        bool block_scaled = false) {
  t_last_error.clear();
  if (G < 0 || M < 0 || N < 0 || K_total < 0) return fail(DG_ERR_INVALID_ARG, "negative size");
  if (G == 0 || M == 0 || N == 0) return DG_OK;
  if (!A || !sA || !B || !sB || !offsets || !D) return fail(DG_ERR_INVALID_ARG, "null pointer");
  if (M % 16 != 0 || N % 16 != 0)
    return fail(DG_ERR_ALIGNMENT, "K-grouped: M and N must be multiples of 16 (A [K,M], B [K,N] rows)");
  if (K_total % 128 != 0) return fail(DG_ERR_ALIGNMENT, "K-grouped: K_total must be a multiple of 128");
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
    return fail(DG_ERR_ALIGNMENT, "A, B and D must be 16-byte aligned");
  if (!aligned(sA, 4) || !aligned(sB, 4) || !aligned(offsets, 4))
    return fail(DG_ERR_ALIGNMENT, "sA, sB and offsets must be 4-byte aligned");
  if ((long long)G * M > INT_MAX - 256 || K_total > INT_MAX - 256 || N > INT_MAX - 256)
    return fail(DG_ERR_UNSUPPORTED, "a tensor extent exceeds 2^31 - 257");
  if (K_total == 0) {   // every group is empty: D = 0
    const cudaError_t e = cudaMemsetAsync(D, 0, (size_t)G * M * N * (out_f32 ? 4 : 2), stream);
    return e == cudaSuccess ? DG_OK : fail_cuda(e, "cudaMemsetAsync(D)");
  }
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  const int sms = effective_sms(*st);
  const int bn = (block_scaled || N > 128) ? 256 : 128;
  const int mb = ceil_div(M, 128), nb = ceil_div(N, bn);
  if ((long long)G * mb * nb > INT_MAX / 2) return fail(DG_ERR_UNSUPPORTED, "too many tiles");
  const int tiles = G * mb * nb;

  dg::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  dg::GemmParams& p = a.p;
  p.M = M;
  p.N = N;
  p.K = K_total;
  p.G = G;
  p.nkb = K_total / 128;
  p.nnb = ceil_div(N, 128);
  p.ldsa = dg_get_tma_aligned_size(M, 4);
  p.num_m_blocks = mb;
  p.num_n_blocks = nb;
  p.num_splits = 1;
  p.kb_per_split = p.nkb;
  p.num_tiles = tiles;
  p.raster_m = (int16_t)(mb < 16 ? mb : 16);
  p.tail_splits = 1;   // every group's K range comes from its offsets
  p.sA = static_cast<const float*>(sA);   // (packed UE8M0 words when block_scaled)
  p.sB = static_cast<const float*>(sB);
  p.D = D;
  p.status = st->status;
  p.flags = dg::kFlagAMN | dg::kFlagBMN | wait_limit_flags();
  p.m_indices = offsets;   // the K offsets of the groups
  if ((s = encode_2d(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)M, (uint64_t)K_total, (uint64_t)M, 128, 128,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A")) != DG_OK)
    return s;
  if ((s = encode_2d(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)N, (uint64_t)K_total, (uint64_t)N, 128, 128,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B")) != DG_OK)
    return s;
  const uint64_t d_rows = (uint64_t)G * M;
  if (out_f32)
    s = encode_2d(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, (uint64_t)N, d_rows, (uint64_t)N * 4, 16, 32,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, "D", CU_TENSOR_MAP_SWIZZLE_64B);
  else
    s = encode_2d(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, d_rows, (uint64_t)N * 2, 32, 32,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, "D", CU_TENSOR_MAP_SWIZZLE_64B);
  if (s != DG_OK) return s;
  a.block_n = bn;
  a.out_f32 = out_f32;
  a.grid = tiles < sms ? tiles : sms;
  a.stream = stream;
  a.pdl = pdl_setting();
  if (print_configs())
    std::fprintf(stderr, "[dg] k-grouped%s%s G=%d M=%d N=%d K_total=%d: BM=128 BN=%d grid=%d tiles=%d\n",
                 block_scaled ? "/ue8m0" : "", out_f32 ? "/f32" : "", G, M, N, K_total, bn, a.grid, tiles);
  const cudaError_t e = block_scaled ? dg::launch_bs_kgrouped(a) : dg::launch_kgrouped(a);
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return DG_OK;
}

}  // namespace

extern "C" {

dg_status dg_fp8_gemm_nt(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D, int M,
                         int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_gemm_nt_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D, int M,
                             int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_grouped_contiguous(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                    const int32_t* m_indices, uint16_t* D, int M_total, int N, int K, int G,
                                    dg_stream_t stream) {
  return run_gemm(dg::kContiguous, false, A, sA, B, sB, m_indices, D, M_total, N, K, G,
                  static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_grouped_contiguous_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                        const int32_t* m_indices, float* D, int M_total, int N, int K, int G,
                                        dg_stream_t stream) {
  return run_gemm(dg::kContiguous, true, A, sA, B, sB, m_indices, D, M_total, N, K, G,
                  static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                const int32_t* masked_m, uint16_t* D, int G, int M_max, int N, int K,
                                dg_stream_t stream) {
  return run_gemm(dg::kMasked, false, A, sA, B, sB, masked_m, D, M_max, N, K, G, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_grouped_masked_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                    const int32_t* masked_m, float* D, int G, int M_max, int N, int K,
                                    dg_stream_t stream) {
  return run_gemm(dg::kMasked, true, A, sA, B, sB, masked_m, D, M_max, N, K, G, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_gemm_nt_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, uint16_t* D,
                               int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true);
}

dg_status dg_fp8_gemm_nt_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, float* D,
                                   int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true);
}

dg_status dg_fp8_grouped_contiguous_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                          const int32_t* m_indices, uint16_t* D, int M_total, int N, int K, int G,
                                          dg_stream_t stream) {
  return run_gemm(dg::kContiguous, false, A, sA, B, sB, m_indices, D, M_total, N, K, G,
                  static_cast<cudaStream_t>(stream), true);
}

dg_status dg_fp8_grouped_contiguous_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                              const int32_t* sB, const int32_t* m_indices, float* D, int M_total,
                                              int N, int K, int G, dg_stream_t stream) {
  return run_gemm(dg::kContiguous, true, A, sA, B, sB, m_indices, D, M_total, N, K, G,
                  static_cast<cudaStream_t>(stream), true);
}

dg_status dg_fp8_grouped_masked_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                      const int32_t* masked_m, uint16_t* D, int G, int M_max, int N, int K,
                                      dg_stream_t stream) {
  return run_gemm(dg::kMasked, false, A, sA, B, sB, masked_m, D, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  true);
}

dg_status dg_fp8_grouped_masked_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                          const int32_t* masked_m, float* D, int G, int M_max, int N, int K,
                                          dg_stream_t stream) {
  return run_gemm(dg::kMasked, true, A, sA, B, sB, masked_m, D, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  true);
}

dg_status dg_fp8_k_grouped_gemm_tn_contiguous(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                              const int32_t* k_offsets, uint16_t* D, int G, int M, int N,
                                              int K_total, dg_stream_t stream) {
  return run_k_grouped(false, A, sA, B, sB, k_offsets, D, G, M, N, K_total, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_k_grouped_gemm_tn_contiguous_f32(const uint8_t* A, const float* sA, const uint8_t* B,
                                                  const float* sB, const int32_t* k_offsets, float* D, int G, int M,
                                                  int N, int K_total, dg_stream_t stream) {
  return run_k_grouped(true, A, sA, B, sB, k_offsets, D, G, M, N, K_total, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                    const int32_t* sB, const int32_t* k_offsets, uint16_t* D, int G,
                                                    int M, int N, int K_total, dg_stream_t stream) {
  return run_k_grouped(false, A, sA, B, sB, k_offsets, D, G, M, N, K_total, static_cast<cudaStream_t>(stream), true);
}

dg_status dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                        const int32_t* sB, const int32_t* k_offsets, float* D, int G,
                                                        int M, int N, int K_total, dg_stream_t stream) {
  return run_k_grouped(true, A, sA, B, sB, k_offsets, D, G, M, N, K_total, static_cast<cudaStream_t>(stream), true);
}

dg_status dg_transform_sf_into_ue8m0_a(const float* sA, int32_t* sA_packed, int G, int M, int K, dg_stream_t stream) {
  if (!sA || !sA_packed) return fail(DG_ERR_INVALID_ARG, "null pointer");
  if (G < 1 || M < 1 || K < 1) return fail(DG_ERR_INVALID_ARG, "G, M and K must be positive");
  if (!aligned(sA, 4) || !aligned(sA_packed, 4)) return fail(DG_ERR_ALIGNMENT, "scale arrays must be 4-byte aligned");
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  const int nkb = ceil_div(K, 128), ldsa = dg_get_tma_aligned_size(M, 4);
  const cudaError_t e = dg::launch_sf_pack_a(sA, sA_packed, G, nkb, ldsa, st->status, effective_sms(*st),
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "UE8M0 packing (A) launch");
}

dg_status dg_transform_sf_a_into_mn_major(const float* sA_rows, float* sA, int G, int M, int K, dg_stream_t stream) {
  if (!sA_rows || !sA) return fail(DG_ERR_INVALID_ARG, "null pointer");
  if (G < 1 || M < 1 || K < 1) return fail(DG_ERR_INVALID_ARG, "G, M and K must be positive");
  if (!aligned(sA_rows, 4) || !aligned(sA, 4)) return fail(DG_ERR_ALIGNMENT, "scale arrays must be 4-byte aligned");
  if (G > 65535) return fail(DG_ERR_UNSUPPORTED, "more than 65535 groups");
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  const cudaError_t e = dg::launch_sf_a_to_mn_major(sA_rows, sA, G, M, ceil_div(K, 128), dg_get_tma_aligned_size(M, 4),
                                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "scale transpose launch");
}

dg_status dg_transform_sf_into_ue8m0_b(const float* sB, int32_t* sB_packed, int G, int N, int K, dg_stream_t stream) {
  if (!sB || !sB_packed) return fail(DG_ERR_INVALID_ARG, "null pointer");
  if (G < 1 || N < 1 || K < 1) return fail(DG_ERR_INVALID_ARG, "G, N and K must be positive");
  if (!aligned(sB, 4) || !aligned(sB_packed, 4)) return fail(DG_ERR_ALIGNMENT, "scale arrays must be 4-byte aligned");
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  const int nkb = ceil_div(K, 128);
  const long long rows = (long long)G * ceil_div(N, 128);
  const cudaError_t e = dg::launch_sf_pack_b(sB, sB_packed, rows, nkb, st->status, effective_sms(*st),
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "UE8M0 packing (B) launch");
}

dg_status dg_fp8_gemm_nn(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D, int M,
                         int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, false, true);
}

dg_status dg_fp8_gemm_nn_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D, int M,
                             int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, false, true);
}

dg_status dg_fp8_gemm_tn(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D, int M,
                         int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, true, true);
}

dg_status dg_fp8_gemm_tn_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D, int M,
                             int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, true, true);
}

dg_status dg_fp8_gemm_tt(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D, int M,
                         int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, true, false);
}

dg_status dg_fp8_gemm_tt_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D, int M,
                             int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, true, false);
}

dg_status dg_fp8_gemm_nn_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, uint16_t* D,
                               int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, false, true);
}

dg_status dg_fp8_gemm_nn_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, float* D,
                                   int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, false, true);
}

dg_status dg_fp8_gemm_tn_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, uint16_t* D,
                               int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, true, true);
}

dg_status dg_fp8_gemm_tn_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, float* D,
                                   int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, true, true);
}

dg_status dg_fp8_gemm_tt_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, uint16_t* D,
                               int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, true, false);
}

dg_status dg_fp8_gemm_tt_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB, float* D,
                                   int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  nullptr, false, false, true, false);
}

dg_status dg_fp8_grouped_masked_swiglu(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                       const int32_t* masked_m, uint16_t* H, int G, int M_max, int N, int K,
                                       dg_stream_t stream) {
  return run_gemm(dg::kMasked, false, A, sA, B, sB, masked_m, H, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  false, nullptr, false, true);
}

dg_status dg_fp8_grouped_masked_swiglu_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                           const int32_t* masked_m, float* H, int G, int M_max, int N, int K,
                                           dg_stream_t stream) {
  return run_gemm(dg::kMasked, true, A, sA, B, sB, masked_m, H, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  false, nullptr, false, true);
}

dg_status dg_fp8_grouped_masked_swiglu_fp8(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                           const int32_t* masked_m, uint8_t* Hq, float* sH, int G, int M_max, int N,
                                           int K, dg_stream_t stream) {
  if (!sH) return fail(DG_ERR_INVALID_ARG, "null sH");
  return run_gemm(dg::kMasked, false, A, sA, B, sB, masked_m, Hq, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  false, nullptr, false, true, false, false, false, sH);
}

dg_status dg_fp8_grouped_masked_swiglu_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                             const int32_t* masked_m, uint16_t* H, int G, int M_max, int N, int K,
                                             dg_stream_t stream) {
  return run_gemm(dg::kMasked, false, A, sA, B, sB, masked_m, H, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  true, nullptr, false, true);
}

dg_status dg_fp8_grouped_masked_swiglu_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                 const int32_t* sB, const int32_t* masked_m, float* H, int G,
                                                 int M_max, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kMasked, true, A, sA, B, sB, masked_m, H, M_max, N, K, G, static_cast<cudaStream_t>(stream),
                  true, nullptr, false, true);
}

dg_status dg_fp8_gemm_nt_acc_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, const float* C,
                                 float* D, int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  C, true);
}

dg_status dg_fp8_gemm_nt_ue8m0_acc_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                       const float* C, float* D, int M, int N, int K, dg_stream_t stream) {
  return run_gemm(dg::kDense, true, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), true,
                  C, true);
}

int dg_get_tma_aligned_size(int x, int elem_bytes) {
  if (x < 0 || (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 && elem_bytes != 16)) return -1;
  const int per = 16 / elem_bytes;
  return (x + per - 1) / per * per;
}

int dg_get_mk_alignment_for_contiguous_layout(void) { return 128; }

void dg_set_num_sms(int n) {
  num_sms_cap();  // make sure the environment default has been read first
  g_num_sms_cap.store(n > 0 ? n : 0);
}

int dg_set_pair_b(int on) {
  const int prev = pair_b_setting() ? 1 : 0;
  g_pair_b.store(on ? 1 : 0);
  return prev;
}

int dg_set_pdl(int on) {
  const int prev = pdl_setting() ? 1 : 0;
  g_pdl.store(on ? 1 : 0);
  return prev;
}

int dg_get_pdl(void) { return pdl_setting() ? 1 : 0; }

int dg_set_cluster_split(int on) {
  const int prev = cluster_split_setting() ? 1 : 0;
  g_cluster_split.store(on ? 1 : 0);
  return prev;
}

long long dg_set_wait_limit_us(long long us) {
  const long long prev = wait_limit_setting();
  g_wait_limit_us.store(clamp_wait_limit(us));
  return prev;
}

int dg_set_tail_splits(int n) {
  const int prev = tail_splits_setting();
  g_tail_splits.store(n > 0 ? clamp_tail_splits(n) : kTailSplits);
  return prev;
}

int dg_get_num_sms(void) {
  DeviceState* st = nullptr;
  if (device_state(&st) != DG_OK) {
    const int cap = num_sms_cap();
    return cap > 0 ? cap : 0;
  }
  return effective_sms(*st);
}

dg_status dg_get_device_status(int* code, dg_stream_t stream) {
  t_last_error.clear();
  if (!code) return fail(DG_ERR_INVALID_ARG, "null code");
  *code = 0;
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  int v = 0;
  if ((e = cudaMemcpy(&v, st->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e, "cudaMemcpy(status)");
  if (v != 0) {
    if ((e = cudaMemset(st->status, 0, sizeof(int))) != cudaSuccess) return fail_cuda(e, "cudaMemset(status)");
    if ((v & DG_DEV_TIMEOUT) && st->counters) {
      // an abandoned split-K tile can leave its arrival counter non-zero
      std::lock_guard<std::mutex> lock(g_mutex);
      if ((e = cudaMemset(st->counters, 0, st->counter_count * sizeof(int))) != cudaSuccess)
        return fail_cuda(e, "cudaMemset(counters)");
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    *code = v;
    return fail(DG_ERR_DEVICE_STATUS, "device status word 0x" + std::to_string(v));
  }
  return DG_OK;
}

const char* dg_last_error_string(void) { return t_last_error.c_str(); }

namespace {

dg_status query_config(int mode, int M, int N, int K, int G, int* cfg, bool block_scaled) {
  t_last_error.clear();
  if (!cfg || mode < 0 || mode > 2 || M < 0 || N < 0 || K <= 0 || G < 0) return fail(DG_ERR_INVALID_ARG, "bad query");
  DeviceState* st = nullptr;
  int sms = num_sms_cap();
  if (device_state(&st) == DG_OK) sms = effective_sms(*st);
  if (sms <= 0) sms = 152;  // no device: report the GB300 configuration
  Config c = choose_config(mode, M, N, K, mode == 0 ? 1 : G, sms, block_scaled);
  int block_m = 128;
  if (st) {
    fit_cluster_splits(c, mode, K, block_scaled, false);
    const int cap = use_cluster_split(c, mode, false, block_scaled, false)
                        ? 0 : pair_clusters(c, mode, M, false, block_scaled, false, false);
    if (cap > 0) {   // pairs of CTAs: 256 rows (two CTAs of 128) by BN columns per unit
      const long long units = (long long)ceil_div(ceil_div(M, 128), 2) * ceil_div(N, c.block_n);
      c.grid = 2 * (int)(units < cap ? units : cap);
      block_m = 256;
    }
  }
  cfg[0] = block_m;
  cfg[1] = c.block_n;
  cfg[2] = c.stages;
  cfg[3] = c.splits;
  cfg[4] = c.grid;
  cfg[5] = c.tiles;
  return DG_OK;
}

}  // namespace

dg_status dg_query_config(int mode, int M, int N, int K, int G, int out_f32, int* cfg) {
  (void)out_f32;  // the configuration never depends on the output type
  return query_config(mode, M, N, K, G, cfg, false);
}

dg_status dg_query_config_ue8m0(int mode, int M, int N, int K, int G, int out_f32, int* cfg) {
  (void)out_f32;
  return query_config(mode, M, N, K, G, cfg, true);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Allocation-free dense GEMM.
//
// Some callers cannot let a library call cudaMalloc: frameworks whose caching allocator already
// owns the device memory (a foreign cudaMalloc can fail or fragment their pool), and serving loops
// that must never block on the implicit device synchronisation cudaMalloc/cudaFree may perform.
// dg_fp8_gemm_nt_noalloc serves them: the split-K partials and arrival counters live in the
// fixed array below, which every device that loads libdg holds until the process exits.

// Layout: [counters: 4096 int][workspace: 20 MiB of float]. Shared by every call on a device.
// Split-K uses at most one wave of 128x256 FP32 partial tiles (128 KiB each): 160 of them fit.
static __device__ __align__(256) unsigned char g_dg_noalloc_scratch[kNoAllocCounterBytes + kNoAllocWorkspaceBytes];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the array's name is
// only a host-side stand-in, so its device address is looked up once per device, with that device
// current, and cached.
dg_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DG_ERR_UNSUPPORTED, "device ordinal beyond 64");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dg_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(noalloc scratch)");
    if (!p) return fail(DG_ERR_CUDA, "cudaGetSymbolAddress returned a null scratch address");
    g_noalloc_scratch_ptr[dev] = p;
  }
  *out = g_noalloc_scratch_ptr[dev];
  return DG_OK;
}

}  // namespace

// The allocation-free dense GEMM: the same validation, schedule and kernels as dg_fp8_gemm_nt (one
// shared code path), with any split-K scratch taken from the fixed array above.
extern "C" dg_status dg_fp8_gemm_nt_noalloc(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                            uint16_t* D, int M, int N, int K, dg_stream_t stream) {
  t_last_error.clear();
  // The array is looked up first, so that every call, even one that needs no scratch, performs the
  // per-device set-up (the first call on a device belongs before any stream capture).
  void* scratch = nullptr;
  const dg_status s = noalloc_scratch(&scratch);
  if (s != DG_OK) return s;
  return run_gemm(dg::kDense, false, A, sA, B, sB, nullptr, D, M, N, K, 1, static_cast<cudaStream_t>(stream), false,
                  nullptr, false, false, false, false, true);
}
