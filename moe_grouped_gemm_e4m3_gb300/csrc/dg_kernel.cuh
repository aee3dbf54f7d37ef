// dg_kernel.cuh — the FP8 (E4M3) fine-grained-scaled GEMM kernel for GB300 (sm_103a).
//
// What it computes (DeepGEMM pages: "DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM
// çekirdekleri", tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları" and
// § "Dense ve Grouped GEMM"; DeepSeek-V3 Technical Report § 3.3.2 for the scale granularity):
//
//     D[m,n] = Σ_kb sA[m,kb]·sB[n/128,kb]·P_kb[m,n],   P_kb = Σ_{k in 128-deep slice kb} A[m,k]·B[n,k]
//
// with P_kb produced by the tensor core and promoted, after scaling, into an FP32 accumulator on
// CUDA cores (the two-level accumulation of the "DeepGEMM" first-release summary,
// tr.news.hada.io/topic?id=19444, and "DeepSeek AI libera DeepGEMM", 7minutos.es, § "Detalles y
// beneficios técnicos").
//
// GB300 design (one persistent CTA per SM, warp-specialised; the pages' Hopper design — wgmma,
// register accumulators, FFMA yield-bit interleaving — is prior art, not the blueprint):
//   * producer warp: TMA loads of 128x128-byte A tiles and BNx128-byte B tiles (128-byte swizzle)
//     into a STAGES-deep shared-memory ring guarded by full/empty mbarriers;
//   * two MMA warps: one thread of each issues 4 tcgen05.mma.kind::f8f6f4 (K = 32 each) per
//     128-deep K-block, alternating K-blocks, into a ring of TMEM accumulators (128 lanes x BN FP32
//     columns each), a fresh accumulator per K-block; tcgen05.commit then frees the smem stage and
//     publishes the TMEM buffer. (Each tcgen05 instruction holds its issuing thread for about 50
//     cycles: one thread alone cannot issue a K-block's waits, MMAs and commits in the 512 cycles
//     the tensor core takes to run it.)
//   * epilogue warps (BN/32 of them; warp w owns TMEM lanes 32*(w%4).. and 128 columns
//     starting at 128*(w/4)): tcgen05.ld the K-block's partial, scale it by sA·sB and add it into
//     128 FP32 registers per thread with packed fma.rn.f32x2; release the TMEM buffer right after
//     the loads so the tensor core runs ahead by one K-block;
//   * after the last K-block of a tile: round to BF16 (or keep FP32), write 32x64 (32x32 for FP32)
//     boxes into a 128-byte-swizzled staging buffer and TMA-store them (tails clipped by TMA);
//     rows that must stay untouched (masked tail, contiguous padding) are stored with predicated
//     plain stores instead;
//   * split-K: each split writes its FP32 partial tile to a workspace; the last split to arrive
//     (per-tile counter) sums all partials in split order 0..S-1 — deterministic — and stores.
//
// Tiles: BM = 128 rows (tensor-core M), BN in {128, 256} columns, BK = 128 (one scale block).
// Every pipeline wait is bounded (see mbar_wait); on a timeout the kernel records
// DG_DEV_TIMEOUT, stops issuing, drains its own in-flight copies and MMAs, frees TMEM, returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "dg_ptx.cuh"

namespace dg {

// kKGrouped: groups along K (A stored [K_total, M], B stored [K_total, N], D [G, M, N]); every group
// covers all M x N tiles over its own K-block range.
enum Mode : int { kDense = 0, kContiguous = 1, kMasked = 2, kKGrouped = 3 };

constexpr int kStatusBadGroup = 0x1;
constexpr int kStatusBadMaskedM = 0x2;
constexpr int kStatusBadScale = 0x8;   // a scale packed as UE8M0 was not a power of two (dg_sf_transform.cu)

// Kept at 128 bytes: a larger parameter block made ptxas spill the contiguous form's epilogue.
struct GemmParams {
  int M;             // dense: M; contiguous: M_total; masked: M_max (rows per group)
  int N, K, G;
  int nkb;           // ceil(K / 128): K-blocks (= scale blocks along K)
  int nnb;           // ceil(N / 128): scale blocks along N
  int ldsa;          // row stride of the MN-major A scales (M or M_max rounded up to 4)
  int num_m_blocks;  // ceil(M / 128)
  int num_n_blocks;  // ceil(N / BN)
  int num_splits;    // split-K factor of every tile (1: none; see Sched)
  int kb_per_split;  // K-blocks per split (the last split may get fewer)
  int num_tiles;     // output tiles (dense/contiguous/K-grouped); masked: counted on device
  int16_t raster_m;     // m-blocks per rasterisation group
  int16_t tail_splits;  // most K ranges a tile of a last, partial wave may be cut into (1: never)
  const float* sA;           // block-scaled kernel: the packed UE8M0 words (uint32) instead
  const float* sB;           // block-scaled kernel: the packed UE8M0 words (uint32) instead
  union {
    const int32_t* m_indices;  // K-grouped: the [G+1] K offsets of the groups (K is then K_total)
    float* h_scales;           // fused SwiGLU with FP8 H (masked): the scales of H, [G][I/128][ldsa]
  };
  const int32_t* masked_m;
  void* D;           // row-major, row stride N elements (used by predicated stores)
  float* workspace;  // split-K partial tiles
  int* counters;     // split-K arrival counter per output tile (zero between calls)
  int* status;       // device status word
  int flags;         // kFlag* bits below; bits 8..31: wait limit in microseconds
  int swiglu_i;      // fused SwiGLU: I, the width of H; B holds 2I rows per group (gate, then up)
};

static_assert(sizeof(GemmParams) <= 128, "keep the kernel parameter block at 128 bytes (register allocation)");

constexpr int kFlagAccumulate = 0x1;  // FP32 D only: add the product onto D (D = C + A·Bᵀ, D holding C)
constexpr int kFlagAMN = 0x2;         // dense layouts: A stored [K, M] (MN-major)
constexpr int kFlagBMN = 0x4;         // dense layouts: B stored [K, N] (MN-major)
// Split-K inside a thread-block cluster (dense and contiguous): one work unit per CTA, the splits
// of a tile are the CTAs of one cluster (rank = split), and they reduce through distributed
// shared memory instead of the global workspace.
constexpr int kFlagClusterSplit = 0x8;
// Pairs of CTAs (clusters of 2) over pairs of 128-row blocks that use the same B tile (dense and
// contiguous, BN = 256, no split-K): each CTA loads its own A tile and half of the B tile,
// which TMA multicasts into both CTAs' shared memory, so each SM pulls a third less from L2 per
// K-block. Every MMA commit then releases the stage in both CTAs (empty barriers count 2).
constexpr int kFlagPairB = 0x10;
// The SWIGLU template argument: 0 no SwiGLU; kSwiglu H = silu(gate)·up stored as BF16/FP32;
// kSwigluFp8 H quantised to FP8 for the down projection: each row's 128 columns of a tile (one 1x128
// group) get the codes e4m3_rne(clamp(h · (448/amax), ±448)) and the dequantisation scale amax/448
// (factor and scale 1 where amax = 0).
// D then points to the codes [G·M_max, I] (bytes) and h_scales to the scales [G][I/128][ldsa]
// (the MN-major LHS scale layout of the masked GEMM). A separate instantiation: holding a row's 128
// H values until their amax is known raises the epilogue's register pressure.
constexpr int kSwiglu = 1;
constexpr int kSwigluFp8 = 2;
// Bits 8..31 of the flags word hold the time limit of the pipeline waits in microseconds
// (kWaitLimitShift, mbar_wait).

struct Tile {
  int g;          // group
  int m_blk;      // 128-row block within the group (contiguous/dense: within A)
  int n_blk;      // BN-column block
  int split;      // K split
  int splits;     // K splits of this tile (1: computed whole)
  int out_idx;    // index of the split tile (split-K workspace / counters)
  int a_row;      // first row of the tile in A's 2-D view (also D's)
  int rows;       // rows of the tile that exist for this group (<= 128)
  int kb0, kb1;   // K-block range
  bool skip;      // nothing to compute (all-padding block, bad group)
  bool shared;    // pair mode: both CTAs of the pair use this B tile (each loads half of it)
};

// Pair mode: this CTA's rank in its cluster of 2 (0 otherwise). A 1-D cluster of 2 holds the blocks
// 2c and 2c + 1.
__device__ __forceinline__ int pair_rank(const GemmParams& p) {
  return (p.flags & kFlagPairB) ? (int)(blockIdx.x & 1) : 0;
}

// ---------------------------------------------------------------------------------------------
// Tile scheduling. Every role walks the same sequence of linear tile ids (blockIdx.x, then +grid)
// and decodes them identically, so the roles agree on every tile without talking to each other.

// Clamped valid-row count of masked group g.
__device__ __forceinline__ int masked_rows(const GemmParams& p, int g) {
  int v = __ldg(p.masked_m + g);
  return v < 0 ? 0 : (v > p.M ? p.M : v);
}

// Number of (m, n) tiles of the masked problem (warp-cooperative; all lanes return the total).
__device__ __forceinline__ int masked_total_tiles(const GemmParams& p, int lane, bool report) {
  int total = 0;
  for (int g0 = 0; g0 < p.G; g0 += 32) {
    const int g = g0 + lane;
    int cnt = 0;
    if (g < p.G) {
      const int raw = __ldg(p.masked_m + g);
      if (report && (raw < 0 || raw > p.M)) atomicOr(p.status, kStatusBadMaskedM);
      cnt = ((masked_rows(p, g) + 127) / 128) * p.num_n_blocks;
    }
    total += __reduce_add_sync(0xffffffffu, cnt);
  }
  return total;
}

// Work units of the persistent loop. Output tiles [0, whole) of the linear order run whole; every
// later tile is cut into `splits` K ranges of `kps` K-blocks, and the last range to finish reduces
// the partial tiles (split-K). Unit ids: tiles first, then the ranges of each split tile in turn.
struct Sched {
  int whole;   // tiles computed whole
  int splits;  // K ranges per remaining tile
  int kps;     // K-blocks per range
  int units;   // whole + (tiles - whole) * splits
};

// A host-chosen split (num_splits > 1) applies to every tile. Otherwise, with TAIL and
// tail_splits > 1, the last partial wave (tiles % grid, at most half the grid) is split along K when
// the K-blocks it saves outweigh the exchange. Model on GB300, in ns: a K-block KB_NS (534 with
// CUDA-core promotion, 300 block-scaled); publishing a partial 2500 (BN=256) / 1600 (BN=128);
// reducing, per split, 1000 / 600.
template <int BN, bool TAIL, int KB_NS>
__device__ __forceinline__ Sched make_sched(const GemmParams& p, int tiles, int grid) {
  Sched s;
  if (p.num_splits > 1) {
    s.whole = 0;
    s.splits = p.num_splits;
    s.kps = p.kb_per_split;
  } else {
    s.whole = tiles;
    s.splits = 1;
    s.kps = p.nkb;
    const int rem = tiles % grid;
    if (TAIL && p.tail_splits > 1 && rem > 0 && 2 * rem <= grid) {
      constexpr int kPub = BN == 256 ? 2500 : 1600, kRed = BN == 256 ? 1000 : 600, kKb = KB_NS;
      int best_gain = 0;
      for (int S = 2; S <= p.tail_splits && S * rem <= grid; ++S) {
        const int kps = (p.nkb + S - 1) / S;
        const int eff = (p.nkb + kps - 1) / kps;   // ranges that are not empty
        const int gain = (p.nkb - kps) * kKb - (kPub + eff * kRed);
        if (eff > 1 && gain > best_gain) {
          best_gain = gain;
          s.whole = tiles - rem;
          s.splits = eff;
          s.kps = kps;
        }
      }
    }
  }
  s.units = s.whole + (tiles - s.whole) * s.splits;
  return s;
}

// Decodes work unit t (warp-cooperative for masked and contiguous modes).
template <int BN, Mode MODE>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, const Sched& sc, int t, int lane) {
  Tile tile;
  tile.skip = false;
  tile.shared = false;
  int u;   // output tile
  if (t < sc.whole) {
    u = t;
    tile.split = 0;
    tile.splits = 1;
    tile.out_idx = 0;
    tile.kb0 = 0;
    tile.kb1 = p.nkb;
  } else {
    const int v = t - sc.whole;
    u = sc.whole + v / sc.splits;
    tile.split = v % sc.splits;
    tile.splits = sc.splits;
    tile.out_idx = u - sc.whole;
    tile.kb0 = tile.split * sc.kps;
    tile.kb1 = min(p.nkb, tile.kb0 + sc.kps);
  }
  if (tile.kb1 <= tile.kb0) tile.skip = true;
  if constexpr (MODE == kMasked) {
    // u -> (g, m_blk, n_blk): groups in order, within a group m fastest so the (at most two for
    // decode-sized groups) m-blocks that share a B tile run side by side.
    int base = 0;
    tile.g = -1;
    for (int g0 = 0; g0 < p.G; g0 += 32) {
      const int g = g0 + lane;
      const int rows = g < p.G ? masked_rows(p, g) : 0;
      const int mb = (rows + 127) / 128;
      const int cnt = mb * p.num_n_blocks;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int chunk_total = __shfl_sync(0xffffffffu, incl, 31);
      if (u < base + chunk_total) {
        const unsigned hit = __ballot_sync(0xffffffffu, base + incl > u);
        const int L = __ffs(hit) - 1;
        const int excl = __shfl_sync(0xffffffffu, incl - cnt, L);
        const int mbL = __shfl_sync(0xffffffffu, mb, L);
        const int rowsL = __shfl_sync(0xffffffffu, rows, L);
        const int local = u - base - excl;
        tile.g = g0 + L;
        tile.m_blk = local % mbL;
        tile.n_blk = local / mbL;
        tile.rows = min(128, rowsL - tile.m_blk * 128);
        tile.a_row = tile.g * p.M + tile.m_blk * 128;
        break;
      }
      base += chunk_total;
    }
    if (tile.g < 0) tile.skip = true;
  } else {
    // u -> (m_blk, n_blk) rasterised in groups of raster_m m-blocks: the CTAs running at the same
    // time cover raster_m m-blocks x (grid / raster_m) n-blocks, so A and B tiles are re-read
    // from L2 rather than HBM.
    int v = u;   // tile within its group (K-grouped) or within the problem
    if constexpr (MODE == kKGrouped) {
      // one K group per block of num_m_blocks x num_n_blocks tiles
      const int tiles_per_group = p.num_m_blocks * p.num_n_blocks;
      tile.g = u / tiles_per_group;
      v = u - tile.g * tiles_per_group;
    }
    // pair mode: the rasterised unit is a pair of m-blocks (2j, 2j+1), rank r of the cluster takes 2j+r
    const bool pair = BN == 256 && (MODE == kDense || MODE == kContiguous) && (p.flags & kFlagPairB);
    const int m_units = pair ? (p.num_m_blocks + 1) / 2 : p.num_m_blocks;
    const int per_group = p.raster_m * p.num_n_blocks;
    const int grp = v / per_group;
    const int first_m = grp * p.raster_m;
    const int gsz = min(m_units - first_m, p.raster_m);
    const int local = v % per_group;
    const int m_unit = first_m + local % gsz;
    tile.m_blk = pair ? 2 * m_unit + (int)(blockIdx.x & 1) : m_unit;
    tile.n_blk = local / gsz;
    tile.a_row = tile.m_blk * 128;
    tile.rows = min(128, p.M - tile.a_row);   // pair mode: <= 0 for a second block past M
    tile.shared = pair;
    if constexpr (MODE != kKGrouped) tile.g = 0;
    if constexpr (MODE == kContiguous) {
      // A block's group is the largest valid index among its rows (padding rows are -1).
      // Rows with an index outside [-1, G) are flagged and never stored.
      auto block_group = [&](int m_blk) -> int {
        int mx = -1;
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = m_blk * 128 + lane * 4 + i;
          if (r < p.M) {
            const int idx = __ldg(p.m_indices + r);
            if (idx >= 0 && idx < p.G) mx = max(mx, idx);
            bad |= (idx < -1 || idx >= p.G);
          }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kStatusBadGroup);
        return (int)__reduce_max_sync(0xffffffffu, (unsigned)(mx + 1)) - 1;
      };
      if (pair) {
        // Both CTAs of the pair decide alike: they share B when the two blocks have one group (or
        // one of them is all padding, which computes with the other's B and stores nothing);
        // otherwise each loads its own group's whole B tile. Nothing to do when both are padding.
        const int g0 = block_group(2 * m_unit), g1 = block_group(2 * m_unit + 1);
        const int g_own = (blockIdx.x & 1) ? g1 : g0, g_other = (blockIdx.x & 1) ? g0 : g1;
        tile.g = g_own >= 0 ? g_own : g_other;
        tile.shared = g0 < 0 || g1 < 0 || g0 == g1;
        if (g0 < 0 && g1 < 0) tile.skip = true;
      } else {
        tile.g = block_group(tile.m_blk);
        if (tile.g < 0) tile.skip = true;        // all padding (or all invalid): nothing to do
      }
    }
    if constexpr (MODE == kKGrouped) {
      // the group's K-block range; an empty range still stores its (zero) tile. Offsets that are
      // not multiples of 128, decrease or pass k_total are flagged and the group is left untouched.
      const int k0 = __ldg(p.m_indices + tile.g), k1 = __ldg(p.m_indices + tile.g + 1);
      if ((k0 | k1) % 128 != 0 || k0 < 0 || k1 < k0 || k1 > p.K) {
        tile.skip = true;
        if (lane == 0 && tile.m_blk == 0 && tile.n_blk == 0) atomicOr(p.status, kStatusBadGroup);
      }
      tile.kb0 = k0 / 128;
      tile.kb1 = k1 / 128;
      tile.a_row = tile.g * p.M + tile.m_blk * 128;   // the tile's first row of D [G*M, N]
    }
  }
  return tile;
}

// ---------------------------------------------------------------------------------------------
// Warp roles, register split and shared-memory plan.
//
// Epilogue warps come first, 4 per EPI_COLS-wide column group (one per 32-lane TMEM quadrant);
// then one more warpgroup holds the producer warp, the two MMA-issuing warps and an idle warp, so
// that every warpgroup is whole and can rebalance registers with setmaxnreg.

template <int BN, int EPI_COLS>
struct Roles {
  static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
  static_assert(EPI_COLS == 64 || EPI_COLS == 128, "EPI_COLS must be 64 or 128");
  static_assert(BN % EPI_COLS == 0, "EPI_COLS must divide BN");
  static constexpr int kEpiWarps = 4 * (BN / EPI_COLS);
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kProducerWarp = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + 1;    // allocates TMEM; issues the even K-blocks
  static constexpr int kMmaWarp2 = kEpiWarps + 2;   // issues the odd K-blocks
  static constexpr int kWarps = kEpiWarps + 4;
  static constexpr int kThreads = kWarps * 32;
  // Registers per thread at launch (65536 per SM, allocated for whole 4-warp groups).
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8 > 255 ? 255 : (65536 / kThreads) / 8 * 8;
  // With more than 8 warps the launch budget is too small for 128 accumulators per epilogue
  // thread: shift registers from the producer/MMA warpgroup (56) to the epilogue warpgroups.
  static constexpr bool kRebalance = kThreads > 256;
  // (BN = 128 epilogue warps hold 64 accumulators, so the producer and MMA warps get more there)
  static constexpr int kOtherRegs = BN == 128 ? 80 : 56;
  static constexpr int kEpiRegs = ((kLaunchRegs * kThreads - kOtherRegs * 128) / kEpiThreads) / 8 * 8;
  static_assert(!kRebalance || kEpiRegs * kEpiThreads + kOtherRegs * 128 <= kLaunchRegs * kThreads,
                "register split exceeds the launch budget");
  static_assert(!kRebalance || kEpiRegs <= 256, "setmaxnreg limit");
};

template <int BN, int STAGES, int EPI_WARPS, int NBUF>
struct SmemPlan {
  static constexpr uint32_t kABytes = 128 * 128;
  static constexpr uint32_t kBBytes = BN * 128;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kStagingBox = 32 * 64;         // one 32-row x 64-byte swizzled box
  static constexpr uint32_t kStagingPerWarp = 2 * kStagingBox;  // double-buffered
  static constexpr uint32_t kStagingOff = STAGES * kStageBytes;
  static constexpr uint32_t kBarOff = kStagingOff + EPI_WARPS * kStagingPerWarp;
  static constexpr uint32_t kNumBars = 2 * STAGES + 2 * NBUF + 2 + 8;   // + fused-SwiGLU hand-over
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStashOff = kMiscOff + 64;                 // per epilogue warp: its tile
  static constexpr uint32_t kBytes = kStashOff + EPI_WARPS * 64;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kDynamicBytes <= 232448, "shared memory plan exceeds 227 KB");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

// silu(x) = x / (1 + e^-x), the gate function of SwiGLU, with the fast exponential and division
// (relative error ~1e-6). For x below about -87 the denominator overflows and the quotient is -0, the
// function's limit. (An IEEE-rounded division or reciprocal there takes a slow special-case path:
// it made the fused kernel 50% slower than the GEMM alone on decode-sized outputs.)
__device__ __forceinline__ float silu_f32(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------------------------
// The kernel.
//
// TMEM holds a ring of NBUF accumulator buffers of BN FP32 columns (NBUF * BN <= 512), one per
// K-block in flight. The MMA of K-block kb writes buffer kb % NBUF while the epilogue promotes
// earlier K-blocks out of the others; an epilogue warp releases a buffer as soon as its last TMEM
// load has landed, before the FMAs that consume it. The ring's depth is what hides the round trip
// "MMA done -> commit -> epilogue loads -> release -> next MMA into that buffer".

//
// SWIGLU (masked form only, BN = 256): the tile's 256 B rows are 128 gate rows (block n of [0, I))
// and the 128 up rows I + 128·n ..; the epilogue pairs the two halves and stores
// H = silu(gate)·up, 128 columns of the [G·M_max, I] output per tile.

template <int BN, int EPI_COLS, int STAGES, int NBUF, Mode MODE, bool OUT_F32, int SWIGLU>
__global__ void __launch_bounds__(Roles<BN, EPI_COLS>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using R = Roles<BN, EPI_COLS>;
  using Plan = SmemPlan<BN, STAGES, R::kEpiWarps, NBUF>;
  constexpr int kEpiWarps = R::kEpiWarps;
  // cluster split-K (kFlagClusterSplit) is compiled into the dense and contiguous forms only
  constexpr bool kClusterCapable = (MODE == kDense || MODE == kContiguous) && !SWIGLU;
  constexpr int kChunks = EPI_COLS / 32;   // 32-column TMEM loads per epilogue thread and K-block
  constexpr uint32_t kTmemCols = NBUF * BN;
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocation: power of two");
  constexpr uint32_t kIdesc = make_idesc_e4m3_f32(128, BN);
  static_assert(kChunks % 2 == 0, "TMEM loads go in pairs");
  // Two MMA issuers take alternate K-blocks, and each waits on its stages' full barriers and its
  // TMEM buffers' empty barriers by phase parity. With even STAGES and NBUF every stage and buffer
  // belongs to one issuer, whose consecutive uses are one phase apart. With an odd count both
  // issuers would share a stage, and one could wait for the use two phases ahead while the barrier
  // is still one phase behind: the parity test would pass early and the ring would lose step.
  static_assert(STAGES % 2 == 0 && NBUF % 2 == 0, "stage and TMEM-buffer counts must be even (two issuers)");
  static_assert(!SWIGLU || (BN == 256 && EPI_COLS == 128 && MODE == kMasked), "fused SwiGLU: masked, BN = 256");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Plan::kBarOff);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;        // [buffer]: the K-block's partial is in TMEM
  uint64_t* tempty_bar = tfull_bar + NBUF;         // [buffer]: every epilogue warp has loaded it
  uint64_t* epi_arrive_bar = tempty_bar + NBUF;       // split-K: all epilogue warps published a partial
  uint64_t* epi_release_bar = epi_arrive_bar + 1;  // split-K: the arrival count has been taken
  uint64_t* xfull_bar = epi_release_bar + 1;       // fused SwiGLU [quadrant]: up values are in the buffer
  uint64_t* xempty_bar = xfull_bar + 4;            // fused SwiGLU [quadrant]: the gate warp has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Plan::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 8);
  // cluster split-K: set when an epilogue warp of this CTA ends without its partial (a skipped tile,
  // or a wait that gave up); the cluster then leaves D untouched
  volatile int* no_partial = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 12);
  volatile int* sched_smem = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 16);   // Sched, 4 ints

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // pair mode (dense and contiguous, BN = 256): see kFlagPairB
  const bool pair = (BN == 256 && (MODE == kDense || MODE == kContiguous) && !SWIGLU) && (p.flags & kFlagPairB);
  // the persistent loop's first unit and stride: a pair walks the units together
  const int unit0 = pair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustep = pair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], pair ? 2 : 1);   // pair mode: released by the MMAs of both CTAs
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kEpiWarps);
    }
    mbar_init(epi_arrive_bar, kEpiWarps);
    mbar_init(epi_release_bar, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&xfull_bar[q], 1);
      mbar_init(&xempty_bar[q], 1);
    }
    *abort_flag = 0;
    *last_flag = 0;
    *no_partial = 0;
    fence_barrier_init();
  }
  if (warp == R::kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // Programmatic dependent launch: everything above reads no global memory that the previous
  // kernel in the stream may still be writing; everything below may.
  griddep_wait();
  if (warp == 0) {
    // the launch's work units, the same in every CTA (masked: tiles counted from masked_m)
    int tiles = p.num_tiles;
    if constexpr (MODE == kMasked) tiles = masked_total_tiles(p, lane, blockIdx.x == 0);
    const Sched sc = make_sched<BN, true, 534>(p, tiles, (int)gridDim.x);
    if (lane == 0) {
      sched_smem[0] = sc.whole; sched_smem[1] = sc.splits; sched_smem[2] = sc.kps; sched_smem[3] = sc.units;
    }
    if (lane < kEpiWarps) {   // and in ints 8..11 of every epilogue warp's stash
      volatile int* st = reinterpret_cast<volatile int*>(smem + Plan::kStashOff + lane * 64);
      st[8] = sc.whole; st[9] = sc.splits; st[10] = sc.kps; st[11] = sc.units;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) griddep_launch_dependents();
  // pair mode: the peer's multicast copies and MMA commits arrive on this CTA's barriers, so both
  // CTAs' barriers are initialised before either starts
  if (pair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= kEpiWarps) {
    // ================================================================== producer / MMA warpgroup
    if constexpr (R::kRebalance) setmaxnreg_dec<R::kOtherRegs>();
    const Sched sc = {sched_smem[0], sched_smem[1], sched_smem[2], sched_smem[3]};
    const int total_units = sc.units;
    if (warp == R::kProducerWarp) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t it = 0;
      bool alive = true;
      int issued_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
      // L2 hints: A tiles evict last (re-read by every n-block of the tiles in flight). With more
      // than one 128-row block, B tiles evict first: they stream past each m-block group, and A
      // then stays in L2. Measured: dense 4096x7168x16384 (A and B 64 + 117 MB) 385 -> 363 us
      // with DRAM reads 434 -> 365 MB, masked decode N=4096 103 -> 99 us, the other large shapes
      // within 1%. Two exceptions keep evict-last for B: one 128-row block (small M: B is read
      // once, and evict-last measured slightly faster, 128x32768x512 12.6 against 13.7 us), and
      // the contiguous form, where a group's B (29 MB for N=4096, K=7168) fits in L2 and serves
      // all of that group's m-blocks (evict-first doubled its DRAM reads at the same speed).
      const uint64_t policy = l2_policy_evict_last();
      const uint64_t policy_b = (MODE != kContiguous && p.M > 128) ? l2_policy_evict_first() : policy;
      for (int t = unit0; alive && t < total_units; t += ustep) {
        const Tile tile = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile.skip) continue;
        const int b_row = (MODE == kKGrouped ? 0 : tile.g * p.N) + tile.n_blk * BN;
        // Lane 0 runs the tile's K loop on its own (no warp-wide step per K-block).
        int ok = 1;
        if (lane == 0) {
          for (int kb = tile.kb0; kb < tile.kb1; ++kb, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            ok = mbar_wait(&empty_bar[s], ph ^ 1, abort_flag, p.status, p.flags);
            if (!ok) break;
            uint8_t* sa = smem + s * Plan::kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], Plan::kStageBytes);
            if (p.flags & kFlagAMN)   // A stored [K, M]: the box is 128 K-rows x 128 M-bytes
              tma_load_2d(&tmA, sa, &full_bar[s], MODE == kKGrouped ? tile.m_blk * 128 : tile.a_row, kb * 128,
                          policy);
            else
              tma_load_2d(&tmA, sa, &full_bar[s], kb * 128, tile.a_row, policy);
            if (p.flags & kFlagBMN) {  // B stored [K, N]: BN/128 boxes of 128 K-rows x 128 N-bytes, 16 KB apart
#pragma unroll
              for (int h = 0; h < BN / 128; ++h)
                tma_load_2d(&tmB, sa + Plan::kABytes + h * 128 * 128, &full_bar[s], b_row + h * 128, kb * 128,
                            policy_b);
            } else if constexpr (SWIGLU) {
              // gate rows 128·n .. and up rows I + 128·n .. (B's tensor map box is 128 rows)
              const int gate_row = tile.g * p.N + tile.n_blk * 128;
              tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], kb * 128, gate_row, policy_b);
              tma_load_2d(&tmB, sa + Plan::kABytes + 128 * 128, &full_bar[s], kb * 128, gate_row + p.swiglu_i,
                          policy_b);
            } else if (BN == 256 && pair) {
              // B's tensor map box is BN/2 rows here: the tile is two boxes, BN/2 x 128 bytes apart
              constexpr int kHalf = BN / 2;
              if (tile.shared) {
                const int r = (int)(blockIdx.x & 1);   // this CTA's half, written into both CTAs
                tma_load_2d_multicast(&tmB, sa + Plan::kABytes + r * kHalf * 128, &full_bar[s], kb * 128,
                                      b_row + r * kHalf, (uint16_t)0x3, policy_b);
              } else {
                tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], kb * 128, b_row, policy_b);
                tma_load_2d(&tmB, sa + Plan::kABytes + kHalf * 128, &full_bar[s], kb * 128, b_row + kHalf, policy_b);
              }
            } else {
              tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], kb * 128, b_row, policy_b);
            }
            issued_phase[s] = (int)ph;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { alive = false; break; }
      }
      if (!alive && lane == 0) {
        // Abandoned: let the loads already issued land before the CTA's shared memory goes away.
        for (int s = 0; s < STAGES; ++s) {
          if (issued_phase[s] < 0) continue;
          const uint32_t a = smem_u32(&full_bar[s]);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(a, (uint32_t)issued_phase[s]) && global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
      if (pair && lane == 0) {
        if (alive) {
          // Both CTAs' MMAs have released this CTA's last stages: the peer's last commits have
          // arrived on this CTA's barriers (and its copies into this CTA landed before them).
          for (int s = 0; s < STAGES; ++s) {
            if (issued_phase[s] < 0) continue;
            const uint32_t a = smem_u32(&empty_bar[s]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(a, (uint32_t)issued_phase[s]) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
          }
        } else {
          // Abandoned: the peer may have issued copies into this CTA for stages this CTA never
          // armed; give any such copy in flight time to land before the pair's final barrier.
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 50000ull) {
          }
        }
      }
    } else if (warp == R::kMmaWarp || warp == R::kMmaWarp2) {
      // ---------------------------------------------------------------- tcgen05 MMA issuers
      // Two threads issue the MMAs: issuer `me` takes the K-blocks whose running index (over all
      // of this CTA's tiles) is congruent to `me` mod 2, so each has two K-blocks of tensor time for
      // its two waits, four MMAs and two commits. Issuing one tcgen05 instruction blocks the issuing
      // thread for about 50 cycles, so one thread alone needs more time per K-block (waits,
      // 4 MMAs, 2 commits) than the tensor core takes to run it. K-blocks use separate TMEM
      // buffers and stages, so the order in which the two threads issue them does not matter;
      // each commit covers only its own thread's MMAs.
      const uint32_t me = (uint32_t)(warp - R::kMmaWarp);
      const bool a_mn = (p.flags & kFlagAMN) != 0, b_mn = (p.flags & kFlagBMN) != 0;
      const uint32_t a_addr0 = smem_u32(smem);
      const uint64_t adesc0 = a_mn ? make_sw128_mnmajor_desc(a_addr0, 128 * 128) : make_sw128_kmajor_desc(a_addr0);
      const uint64_t bdesc0 = b_mn ? make_sw128_mnmajor_desc(a_addr0 + Plan::kABytes, 128 * 128)
                                   : make_sw128_kmajor_desc(a_addr0 + Plan::kABytes);
      // one K=32 step: +32 bytes inside a K-major 128-byte row (+2 in the >>4 address field), or
      // +32 rows of 128 bytes in an MN-major tile (+256)
      const uint32_t a_step = a_mn ? 256u : 2u, b_step = b_mn ? 256u : 2u;
      const uint32_t idesc = kIdesc | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
      uint32_t acc_it = 0;   // running K-block index of the CTA (both issuers count every K-block)
      bool alive = true;
      int last_b = -1;
      uint32_t last_ph = 0;
      for (int t = unit0; alive && t < total_units; t += ustep) {
        const Tile tile = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile.skip) continue;
        const uint32_t nk = (uint32_t)(tile.kb1 - tile.kb0);
        // Lane 0 runs this issuer's K-blocks of the tile on its own (no warp-wide step per K-block).
        int ok = 1;
        if (lane == 0) {
          for (uint32_t g = acc_it + ((me - acc_it) & 1u); g < acc_it + nk; g += 2) {
            const int s = (int)(g % STAGES);
            const uint32_t ph = (g / STAGES) & 1;
            const int b = (int)(g % NBUF);
            const uint32_t aph = (g / NBUF) & 1;
            // the stage's data first (normally there long before), then the TMEM buffer, whose
            // release by the epilogue is the round trip this wait is on
            ok = mbar_wait(&full_bar[s], ph, abort_flag, p.status, p.flags) &&
                 mbar_wait(&tempty_bar[b], aph ^ 1, abort_flag, p.status, p.flags);
            if (!ok) break;
            tc_fence_after();
            const uint64_t soff = (uint64_t)((s * Plan::kStageBytes) >> 4);
            const uint64_t adesc = adesc0 + soff, bdesc = bdesc0 + soff;
            const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mma_e4m3(d_tmem, adesc + a_step * k, bdesc + b_step * k, idesc, k > 0 ? 1u : 0u);
            }
            if (pair)
              mma_commit_multicast(&empty_bar[s], (uint16_t)0x3);   // the stage is free in both CTAs' view
            else
              mma_commit(&empty_bar[s]);
            mma_commit(&tfull_bar[b]);
            last_b = b;
            last_ph = aph;
          }
        }
        acc_it += nk;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { alive = false; break; }
      }
      if (!alive && lane == 0 && last_b >= 0) {
        // Abandoned: wait for the MMAs this thread issued before TMEM is freed.
        const uint32_t a = smem_u32(&tfull_bar[last_b]);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, last_ph) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    if (kClusterCapable && (p.flags & kFlagClusterSplit)) {
      // the two cluster barriers of the epilogue's reduction, which every thread must reach
      __syncwarp();
      cluster_sync_all();
      cluster_sync_all();
    }
  } else {
    // ================================================================== epilogue warpgroups
    if constexpr (R::kRebalance) setmaxnreg_inc<R::kEpiRegs>();
    const int quad = warp % 4;              // TMEM lanes 32*quad .. 32*quad+31
    const int cgrp = warp / 4;              // columns EPI_COLS*cgrp .. of the tile
    // The tile description is parked in shared memory across the K loop, so that only the loop's
    // own values occupy registers next to the 128 accumulators and the 64 loaded partials. Ints
    // 8..11 hold the launch's Sched (whole, splits, kps, units), read where needed.
    volatile int* stash = reinterpret_cast<volatile int*>(smem + Plan::kStashOff + warp * 64);
    const int row_in_tile = quad * 32 + lane;
    uint8_t* staging = smem + Plan::kStagingOff + warp * Plan::kStagingPerWarp;
    const uint32_t staging_addr = smem_u32(staging);
    uint32_t acc_it = 0, sk_it = 0, x_it = 0;
    bool alive = true;
    uint32_t store_count = 0;   // TMA store boxes issued by this warp
    // Tile columns EPI_COLS*cgrp + i, as FP32 pairs so that each promotion step is one packed
    // fma (__ffma2_rn: two IEEE round-to-nearest FMAs in one instruction).
    float2 acc2[EPI_COLS / 2];
    float* const acc = reinterpret_cast<float*>(acc2);

    bool have_partial = false;   // cluster split: this CTA's partial tile is in acc
    for (int t = unit0; alive && t < stash[11]; t += ustep) {
      int kb_begin, kb_end;
      {
        const Sched sc = {stash[8], stash[9], stash[10], stash[11]};
        const Tile tile0 = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile0.skip) continue;
        if (lane == 0) {
          stash[0] = tile0.g; stash[1] = tile0.m_blk; stash[2] = tile0.n_blk; stash[3] = tile0.split;
          stash[4] = tile0.out_idx; stash[5] = tile0.a_row; stash[6] = tile0.rows; stash[7] = tile0.splits;
        }
        kb_begin = tile0.kb0;
        kb_end = tile0.kb1;
      }
      __syncwarp();
      // The first column of this warp (as a row of B: fused SwiGLU puts the up rows at I + 128·n).
      auto first_col = [&](int n_blk) -> int {
        return SWIGLU ? (cgrp ? p.swiglu_i : 0) + n_blk * 128 : n_blk * BN + cgrp * EPI_COLS;
      };
      // Only what the K loop needs is live across it; the rest of the tile is re-read afterwards.
      const float* sa_ptr;
      const float* sb_ptr;
      bool active, row_live;
      {
        const int g = stash[0], n_col = first_col(stash[2]);
        row_live = row_in_tile < stash[6];
        const bool col_live = n_col < p.N;
        sa_ptr = p.sA + (MODE == kMasked ? (size_t)g * p.nkb * p.ldsa : 0) + stash[1] * 128 + row_in_tile;
        sb_ptr = p.sB + ((size_t)(MODE == kKGrouped ? 0 : g) * p.nnb + (col_live ? n_col / 128 : 0)) * p.nkb;
        // Warps with no row or no column in range only keep the TMEM handshake going.
        active = col_live && __any_sync(0xffffffffu, row_live);
      }

#pragma unroll
      for (int i = 0; i < EPI_COLS; ++i) acc[i] = 0.0f;

      // Scales: K-block kb uses sA[m,kb]·sB[nb,kb]. The pair for kb + 1 is requested at the top of
      // step kb, before its wait, and moved into place at the end of it, so a global load has the
      // step's wait, TMEM loads and FMAs to land. (A K-grouped tile can have an empty K range: it
      // stores zeros and reads no scale.)
      auto fetch_sa = [&](int kb) -> float {
        return (active && row_live && kb < kb_end) ? __ldg(sa_ptr + (size_t)kb * p.ldsa) : 0.0f;
      };
      auto fetch_sb = [&](int kb) -> float { return (active && kb < kb_end) ? __ldg(sb_ptr + kb) : 0.0f; };
      float sa_cur = fetch_sa(kb_begin), sb_cur = fetch_sb(kb_begin);

      for (int kb = kb_begin; kb < kb_end; ++kb, ++acc_it) {
        const int b = acc_it % NBUF;
        const uint32_t aph = (acc_it / NBUF) & 1;
        const float sa_nxt = fetch_sa(kb + 1), sb_nxt = fetch_sb(kb + 1);
        // All 32 lanes wait together: one warp-wide instruction stream, uniform by construction
        // (every lane sees the same barrier phase, timer value and abort flag).
        if (!mbar_wait(&tfull_bar[b], aph, abort_flag, p.status, p.flags)) { alive = false; break; }
        tc_fence_after();
        if (active) {
          const uint32_t taddr =
              tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * BN + cgrp * EPI_COLS);
          float2 scale2 = make_float2(0.0f, 0.0f);
          // two 32-column loads in flight per wait; the buffer is released as soon as the last
          // pair has landed in registers, before its FMAs
#pragma unroll
          for (int c = 0; c < kChunks; c += 2) {
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(taddr + c * 32, r0);
            tmem_ld_32x32b_x32(taddr + (c + 1) * 32, r1);
            tmem_ld_wait(r0);
            reg_fence(r1);
            if (c + 2 == kChunks) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty_bar[b]);
            }
            if (c == 0) {
              const float scale = sa_cur * sb_cur;
              scale2 = make_float2(scale, scale);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              acc2[c * 16 + j] = __ffma2_rn(make_float2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1])),
                                            scale2, acc2[c * 16 + j]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              acc2[(c + 1) * 16 + j] = __ffma2_rn(make_float2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1])),
                                                  scale2, acc2[(c + 1) * 16 + j]);
            }
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[b]);
        }
        sa_cur = sa_nxt;
        sb_cur = sb_nxt;
      }
      if (!alive) break;
      if (kClusterCapable && (p.flags & kFlagClusterSplit)) {   // one unit per CTA: the reduction follows the loop
        have_partial = true;
        break;
      }
      // the tile description, back from shared memory
      Tile tile;
      tile.g = stash[0]; tile.m_blk = stash[1]; tile.n_blk = stash[2]; tile.rows = stash[6];
      tile.split = stash[3]; tile.out_idx = stash[4]; tile.a_row = stash[5]; tile.splits = stash[7];
      const int m_local = tile.m_blk * 128 + row_in_tile;   // row within the group
      const bool row_exists = row_in_tile < tile.rows;
      const int n_col0 = first_col(tile.n_blk);
      const bool col_exists = n_col0 < p.N;

      // ---------------- split-K: publish the partial, and let the last split reduce
      if (tile.splits > 1) {
        float* ws_tile = p.workspace + (size_t)tile.out_idx * tile.splits * (128 * BN);
        float* mine = ws_tile + (size_t)tile.split * (128 * BN);
        if (row_exists && col_exists) {
          // layout [column/4][row][4]: a warp's float4 stores are 512 contiguous bytes
#pragma unroll
          for (int j = 0; j < EPI_COLS; j += 4) {
            const int cq = (cgrp * EPI_COLS + j) / 4;
            __stcg(reinterpret_cast<float4*>(mine + ((size_t)cq * 128 + row_in_tile) * 4),
                   make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]));
          }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_arrive_bar);
        int ok = 1;
        if (warp == 0 && lane == 0) {
          ok = mbar_wait(epi_arrive_bar, sk_it & 1, abort_flag, p.status, p.flags);
          if (ok) {
            const int prev = atomicAdd(p.counters + tile.out_idx, 1);
            const int last = (prev == tile.splits - 1);
            if (last) p.counters[tile.out_idx] = 0;   // ready for the next call
            *last_flag = last;
            mbar_arrive(epi_release_bar);
          }
        }
        if (lane == 0 && ok) ok = mbar_wait(epi_release_bar, sk_it & 1, abort_flag, p.status, p.flags);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        ++sk_it;
        if (!ok) { alive = false; break; }
        if (*last_flag == 0) continue;
        __threadfence();
        if (row_exists && col_exists) {
          // total = partial_0 + partial_1 + ... in split order, whichever split arrived last
#pragma unroll
          for (int i = 0; i < EPI_COLS; ++i) acc[i] = 0.0f;
          for (int sp = 0; sp < tile.splits; ++sp) {
            const float* src = ws_tile + (size_t)sp * (128 * BN);
#pragma unroll
            for (int j = 0; j < EPI_COLS; j += 4) {
              const int cq = (cgrp * EPI_COLS + j) / 4;
              const float4 v = __ldcg(reinterpret_cast<const float4*>(src + ((size_t)cq * 128 + row_in_tile) * 4));
              acc[j] += v.x; acc[j + 1] += v.y; acc[j + 2] += v.z; acc[j + 3] += v.w;
            }
          }
        }
      }

      if constexpr (SWIGLU) {
        // Fused SwiGLU: warp cgrp 1 (up) hands its accumulators to warp cgrp 0 (gate) of the same
        // quadrant, 32 columns per round, through its own staging buffer; both warps hold the same
        // 32 rows. The hand-over is guarded by two mbarriers per quadrant (bounded waits). The gate
        // warp forms silu(gate)·up and stores those 32 columns of H.
        const unsigned row_mask = __ballot_sync(0xffffffffu, row_exists);
        if (row_mask == 0u) continue;                   // the same decision in both warps of the pair
        const bool all_rows = row_mask == 0xffffffffu;
        const uint32_t xchg = smem_u32(smem + Plan::kStagingOff + (quad + 4) * Plan::kStagingPerWarp);
        const int h_col0 = tile.n_blk * 128;           // the tile's first column of H
        constexpr int kColsPerBox = OUT_F32 ? 16 : 32;
        bool ok = true;
#pragma unroll
        for (int r = 0; r < 4; ++r) {   // unrolled: the accumulator indices stay compile-time constants
          const uint32_t xph = x_it & 1;
          ++x_it;
          if (cgrp == 1) {
            ok = mbar_wait(&xempty_bar[quad], xph ^ 1, abort_flag, p.status, p.flags);
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int c = r * 32 + j * 4;
              st_shared_v4(xchg + lane * 128 + (uint32_t)((j ^ (lane & 7)) * 16), __float_as_uint(acc[c]),
                           __float_as_uint(acc[c + 1]), __float_as_uint(acc[c + 2]), __float_as_uint(acc[c + 3]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&xfull_bar[quad]);
            continue;
          }
          ok = mbar_wait(&xfull_bar[quad], xph, abort_flag, p.status, p.flags);
          if (!ok) break;
          float h[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t u0, u1, u2, u3;
            ld_shared_v4(xchg + lane * 128 + (uint32_t)((j ^ (lane & 7)) * 16), u0, u1, u2, u3);
            const int c = r * 32 + j * 4;
            h[j * 4 + 0] = silu_f32(acc[c + 0]) * __uint_as_float(u0);
            h[j * 4 + 1] = silu_f32(acc[c + 1]) * __uint_as_float(u1);
            h[j * 4 + 2] = silu_f32(acc[c + 2]) * __uint_as_float(u2);
            h[j * 4 + 3] = silu_f32(acc[c + 3]) * __uint_as_float(u3);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&xempty_bar[quad]);   // the up warp may refill the buffer
          if constexpr (SWIGLU == kSwigluFp8) {
            // keep H in place of the gate values until the row's 128 columns are all formed
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[r * 32 + j] = h[j];
            continue;
          }
          if (all_rows) {
#pragma unroll
            for (int box = 0; box < 32 / kColsPerBox; ++box) {
              const uint32_t sel = store_count & 1;
              if (store_count >= 2) {
                if (lane == 0) tma_store_wait_read_1();
                __syncwarp();
              }
#pragma unroll
              for (int j = 0; j < 4; ++j) {   // four 16-byte pieces per 64-byte row
                uint32_t w0, w1, w2, w3;
                if constexpr (OUT_F32) {
                  const int c = box * 16 + j * 4;
                  w0 = __float_as_uint(h[c]); w1 = __float_as_uint(h[c + 1]);
                  w2 = __float_as_uint(h[c + 2]); w3 = __float_as_uint(h[c + 3]);
                } else {
                  const int c = j * 8;
                  w0 = pack_bf16x2(h[c], h[c + 1]); w1 = pack_bf16x2(h[c + 2], h[c + 3]);
                  w2 = pack_bf16x2(h[c + 4], h[c + 5]); w3 = pack_bf16x2(h[c + 6], h[c + 7]);
                }
                const uint32_t phys = (uint32_t)(j ^ ((lane >> 1) & 3));
                st_shared_v4(staging_addr + sel * Plan::kStagingBox + lane * 64 + phys * 16, w0, w1, w2, w3);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmD, staging + sel * Plan::kStagingBox, h_col0 + r * 32 + box * kColsPerBox,
                             tile.a_row + quad * 32);
                tma_store_commit();
              }
              ++store_count;
              __syncwarp();
            }
          } else if (row_exists) {
            // predicated plain stores: rows past masked_m stay untouched
            const size_t hrow = (size_t)(tile.a_row + row_in_tile) * p.swiglu_i + h_col0 + r * 32;
            if constexpr (OUT_F32) {
              float* dst = reinterpret_cast<float*>(p.D) + hrow;
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
            } else {
              uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + hrow;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint4 v;
                v.x = pack_bf16x2(h[j], h[j + 1]); v.y = pack_bf16x2(h[j + 2], h[j + 3]);
                v.z = pack_bf16x2(h[j + 4], h[j + 5]); v.w = pack_bf16x2(h[j + 6], h[j + 7]);
                *reinterpret_cast<uint4*>(dst + j) = v;
              }
            }
          }
        }
        if (!ok) { alive = false; break; }
        if (SWIGLU == kSwigluFp8 && cgrp == 0 && row_exists) {
          // the row's 128 columns of H are one 1x128 group: its scale, then its FP8 codes
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 128; ++j) amax = fmaxf(amax, fabsf(acc[j]));
          // one division per row for the factor and one for the scale; a product per element
          const float f = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
          const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
          uint8_t* qrow = reinterpret_cast<uint8_t*>(p.D) + (size_t)(tile.a_row + row_in_tile) * p.swiglu_i + h_col0;
#pragma unroll
          for (int j = 0; j < 128; j += 16) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c = j + q * 4;
              const uint32_t lo = e4m3x2_satfinite(__fmul_rn(acc[c], f), __fmul_rn(acc[c + 1], f));
              const uint32_t hi = e4m3x2_satfinite(__fmul_rn(acc[c + 2], f), __fmul_rn(acc[c + 3], f));
              w[q] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(qrow + j) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          p.h_scales[((size_t)tile.g * (p.swiglu_i / 128) + tile.n_blk) * p.ldsa + m_local] = sc;
        }
        continue;
      }

      // ---------------- output
      bool write_row;
      if constexpr (MODE == kDense || MODE == kKGrouped) {
        write_row = row_exists;
      } else if constexpr (MODE == kMasked) {
        write_row = row_exists;   // rows counts only the valid rows of the group
      } else {
        write_row = false;
        if (row_exists) {
          const int idx = __ldg(p.m_indices + m_local);
          write_row = (idx == tile.g);
          if (idx != tile.g && idx != -1) atomicOr(p.status, kStatusBadGroup);
        }
      }
      const int d_row = tile.a_row + row_in_tile;   // row in D's 2-D view
      if (!__any_sync(0xffffffffu, write_row)) continue;   // no row of this warp is stored
      const bool use_tma = (MODE == kDense) || __all_sync(0xffffffffu, write_row);
      if (!col_exists) continue;
      if (use_tma) {
        // 32-row x 64-byte boxes (32 BF16 or 16 FP32 columns) alternate between two staging
        // buffers: the TMA engine reads one while the warp fills the other.
        constexpr int kColsPerBox = OUT_F32 ? 16 : 32;
#pragma unroll
        for (int chunk = 0; chunk < EPI_COLS / kColsPerBox; ++chunk) {
          if (n_col0 + chunk * kColsPerBox >= p.N) break;
          const uint32_t sel = store_count & 1;
          if (store_count >= 2) {
            if (lane == 0) tma_store_wait_read_1();   // the box that used this buffer has been read
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {   // four 16-byte pieces per 64-byte row
            uint32_t w0, w1, w2, w3;
            if constexpr (OUT_F32) {
              const int c = chunk * 16 + j * 4;
              w0 = __float_as_uint(acc[c]); w1 = __float_as_uint(acc[c + 1]);
              w2 = __float_as_uint(acc[c + 2]); w3 = __float_as_uint(acc[c + 3]);
            } else {
              const int c = chunk * 32 + j * 8;
              w0 = pack_bf16x2(acc[c], acc[c + 1]); w1 = pack_bf16x2(acc[c + 2], acc[c + 3]);
              w2 = pack_bf16x2(acc[c + 4], acc[c + 5]); w3 = pack_bf16x2(acc[c + 6], acc[c + 7]);
            }
            // 64-byte swizzle: 16-byte piece j of row r sits at piece j ^ ((r >> 1) & 3)
            const uint32_t phys = (uint32_t)(j ^ ((lane >> 1) & 3));
            st_shared_v4(staging_addr + sel * Plan::kStagingBox + lane * 64 + phys * 16, w0, w1, w2, w3);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (OUT_F32 && (p.flags & kFlagAccumulate))
              tma_reduce_add_2d(&tmD, staging + sel * Plan::kStagingBox, n_col0 + chunk * kColsPerBox,
                                tile.a_row + quad * 32);
            else
              tma_store_2d(&tmD, staging + sel * Plan::kStagingBox, n_col0 + chunk * kColsPerBox,
                           tile.a_row + quad * 32);
            tma_store_commit();
          }
          ++store_count;
          __syncwarp();
        }
      } else if (write_row) {
        // Predicated plain stores: this warp's 32 rows include rows that must stay untouched.
        if constexpr (OUT_F32) {
          float* drow = reinterpret_cast<float*>(p.D) + (size_t)d_row * p.N;
#pragma unroll
          for (int j = 0; j < EPI_COLS; j += 4) {
            if (n_col0 + j < p.N) {
              float* dst = drow + n_col0 + j;
              if (p.flags & kFlagAccumulate) {
                atomicAdd(dst, acc[j]); atomicAdd(dst + 1, acc[j + 1]);
                atomicAdd(dst + 2, acc[j + 2]); atomicAdd(dst + 3, acc[j + 3]);
              } else {
                *reinterpret_cast<float4*>(dst) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
              }
            }
          }
        } else {
          uint16_t* drow = reinterpret_cast<uint16_t*>(p.D) + (size_t)d_row * p.N;
#pragma unroll
          for (int j = 0; j < EPI_COLS; j += 8) {
            if (n_col0 + j < p.N) {
              uint4 v;
              v.x = pack_bf16x2(acc[j], acc[j + 1]); v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
              v.z = pack_bf16x2(acc[j + 4], acc[j + 5]); v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
              *reinterpret_cast<uint4*>(drow + n_col0 + j) = v;
            }
          }
        }
      }
    }
    if constexpr (kClusterCapable) if (p.flags & kFlagClusterSplit) {
      // Split-K in a cluster. The S CTAs of the cluster computed the S K ranges of one tile (cluster
      // rank = split). Each writes its FP32 partial into its own stage buffers, idle once the K loop
      // is done. After a cluster barrier, each CTA sums the partials of an interleaved set of rows
      // (row r goes to rank r % S) in split order 0..S-1, reading its peers' shared memory, and
      // stores those rows of D. A second barrier keeps every CTA's shared memory in place until its
      // peers have read it. Every thread of the cluster reaches both barriers on every path.
      constexpr uint32_t kRowBytes = (BN + 4) * 4;   // +16 bytes a row: 32 rows cover all banks
      static_assert(128 * kRowBytes <= STAGES * Plan::kStageBytes, "partial tile exceeds the stage buffers");
      const uint32_t part = smem_u32(smem);
      if (have_partial) {
#pragma unroll
        for (int j = 0; j < EPI_COLS; j += 4)
          st_shared_v4(part + row_in_tile * kRowBytes + (cgrp * EPI_COLS + j) * 4, __float_as_uint(acc[j]),
                       __float_as_uint(acc[j + 1]), __float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3]));
      } else if (lane == 0) {
        *no_partial = 1;
      }
      cluster_sync_all();
      // Sum only if every CTA of the cluster holds its partial: a CTA that gave up (a wait timed out)
      // has none, and its stage buffers hold stale bytes that must not reach D.
      const bool complete = cluster_all_zero_u32(smem_u32(const_cast<int*>(no_partial))) && have_partial;
      if (complete) {
        const int S = stash[7], g = stash[0], n_blk = stash[2], a_row = stash[5], rows = stash[6];
        const int rank = (int)cluster_ctarank();
        constexpr int kVec = BN / 4;                       // float4 per row
        constexpr int kRowsPerPass = R::kEpiThreads / kVec;   // 4 (BN=256) or 8 (BN=128)
        const int c4 = threadIdx.x % kVec;
        const int n = n_blk * BN + c4 * 4;
        for (int r = rank + (threadIdx.x / kVec) * S; r < rows; r += kRowsPerPass * S) {
          float4 tot = cluster_sum_v4(part + r * kRowBytes + c4 * 16, S);
          if (n >= p.N) continue;
          const size_t d_row = (size_t)(a_row + r);
          if constexpr (MODE == kContiguous) {
            const int idx = __ldg(p.m_indices + a_row + r);
            if (idx != g) {
              if (idx != -1 && c4 == 0) atomicOr(p.status, kStatusBadGroup);
              continue;   // a padding row (or another group's): left untouched
            }
          }
          if constexpr (OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.D) + d_row * p.N + n);
            if (p.flags & kFlagAccumulate) {
              const float4 c = *dst;
              tot.x = c.x + tot.x; tot.y = c.y + tot.y; tot.z = c.z + tot.z; tot.w = c.w + tot.w;
            }
            *dst = tot;
          } else {
            *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.D) + d_row * p.N + n) =
                make_uint2(pack_bf16x2(tot.x, tot.y), pack_bf16x2(tot.z, tot.w));
          }
        }
      }
      cluster_sync_all();
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  // pair mode: neither CTA leaves while its peer may still copy into it or arrive on its barriers
  if (pair) cluster_sync_all();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace dg
