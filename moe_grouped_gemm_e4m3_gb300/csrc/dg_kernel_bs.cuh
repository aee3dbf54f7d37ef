// dg_kernel_bs.cuh — the FP8 (E4M3) GEMM with packed UE8M0 scales, on the block-scaled tensor core
// of GB300 (sm_103a).
//
// What it computes: the same D = A·Bᵀ with one scale per 1x128 K-group of each A row and one per
// 128x128 block of B, D[m,n] = Σ_kb sA[m,kb]·sB[n/128,kb]·P_kb[m,n], when every scale is a power of
// two given as a UE8M0 code, four codes packed into one 32-bit word (the DeepGEMM SM100 input
// form: "DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
// tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları"). Byte j of word q holds
// K-group 4q+j; A's words are MN-major [ceil(nkb/4)][ldsa], B's are [G][nnb][ceil(nkb/4)].
//
// Power-of-two scales let the tensor core apply them itself: tcgen05.mma.kind::mxf8f6f4 with
// block_scale multiplies each 32-deep slice of every A row and B row by a UE8M0 factor read from
// TMEM, so the whole K loop accumulates into one TMEM accumulator and there is no per-K-block
// promotion on CUDA cores. (With FP32 amax/448 scales that is not exact, which is why the other
// kernel promotes on CUDA cores.)
//
// Scale factors in TMEM (scale_vec::1X, measured on GB300): the MMA reads the scale of A row m at
// lane m, column sfa + m/32, and the scale of B row n at column sfb + n/32, lane n%32 of the lane
// quadrant of the output row it is computing — so B's factors are written to all four quadrants.
// The instruction descriptor's scale-factor IDs pick the byte of the 32-bit cell; a packed word
// therefore serves four consecutive K-blocks with IDs 0..3.
//
// Roles (16 warps, one persistent CTA per SM):
//   * warps 0-7, epilogue: warp w owns TMEM lanes 32*(w%4).. and columns 128*(w/4)..; at the end of
//     a tile it loads its 32x128 FP32 block of the accumulator, frees the accumulator for the next
//     tile at once, then stores BF16 (or FP32) through TMA, or runs the split-K exchange;
//   * warps 8-11, scale writers: warp 8+q writes the packed scale words of its 32 A rows and of the
//     tile's two B blocks into lane quadrant q of a ring of scale slots, one slot per 4 K-blocks;
//   * warp 12, producer: TMA loads of A (128x128 B) and B (256x128 B) into a 4-stage ring;
//   * warp 13, MMA issuer: per K-block, 4 block-scaled MMAs (K = 32 each) into the accumulator.
// Every wait is bounded (mbar_wait); on a timeout the kernel records DG_DEV_TIMEOUT, drains its own
// copies and MMAs, frees TMEM and returns.
#pragma once

#include "dg_kernel.cuh"

namespace dg {

struct BsRoles {
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kScaleWarp0 = 8;      // warps 8..11 write scale factors, quadrant = warp % 4
  static constexpr int kProducerWarp = 12;
  static constexpr int kMmaWarp = 13;        // warps 14 and 15 idle (whole warpgroups for setmaxnreg)
  static constexpr int kWarps = 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kLaunchRegs = 65536 / kThreads;   // 128
  static constexpr int kOtherRegs = 56;
  static constexpr int kEpiRegs = ((kLaunchRegs * kThreads - kOtherRegs * (kThreads - kEpiThreads)) / kEpiThreads) / 8 * 8;
  static_assert(kEpiRegs * kEpiThreads + kOtherRegs * (kThreads - kEpiThreads) <= kLaunchRegs * kThreads,
                "register split exceeds the launch budget");
  static_assert(kEpiRegs <= 256 && kEpiRegs >= 160, "epilogue register budget");
};

struct BsSmemPlan {
  static constexpr int kStages = 4;
  static constexpr int kSfSlots = 4;
  static constexpr uint32_t kABytes = 128 * 128;
  static constexpr uint32_t kBBytes = 256 * 128;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kStagingBox = 32 * 64;
  static constexpr uint32_t kStagingPerWarp = 2 * kStagingBox;
  static constexpr uint32_t kStagingOff = kStages * kStageBytes;
  static constexpr uint32_t kBarOff = kStagingOff + BsRoles::kEpiWarps * kStagingPerWarp;
  static constexpr int kDescSlots = 2;
  // full[S], empty[S], sf_full[SL], sf_empty[SL], desc_full[2], desc_empty[2], acc_full, acc_empty,
  // epi_arrive, epi_release, drain
  static constexpr uint32_t kNumBars = 2 * kStages + 2 * kSfSlots + 2 * kDescSlots + 5;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kDescOff = kMiscOff + 64;           // tile descriptions, 8 ints a slot
  static constexpr uint32_t kStashOff = kDescOff + kDescSlots * 32;   // per epilogue warp: its tile
  static constexpr uint32_t kBytes = kStashOff + BsRoles::kEpiWarps * 64;
  static constexpr uint32_t kDynamicBytes = kBytes + 1024;
  static_assert(kDynamicBytes <= 232448, "shared memory plan exceeds 227 KB");
};

// TMEM columns: the 128x256 FP32 accumulator at 0..255, then the scale-factor slots, 32 columns
// apart: A's four columns at +0..3, B's eight at +16..23.
constexpr uint32_t kBsTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;
constexpr uint32_t kSfSlotCols = 32;
constexpr uint32_t kSfbOff = 16;
static_assert(kSfCol0 + BsSmemPlan::kSfSlots * kSfSlotCols <= kBsTmemCols, "scale slots exceed TMEM");

// SWIGLU (masked form only): the tile's 256 B rows are 128 gate rows (block n of [0, I)) and the
// matching 128 up rows (block n of [I, 2I)), and the epilogue stores H = silu(gate)·up, 128
// columns of H per tile. The whole K loop accumulates in TMEM, so each epilogue warp loads both
// its gate and its up columns itself: no hand-over between warps.
template <Mode MODE, bool OUT_F32, bool SWIGLU = false>
__global__ void __launch_bounds__(BsRoles::kThreads, 1)
    fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using R = BsRoles;
  using Plan = BsSmemPlan;
  constexpr int BN = 256;
  constexpr int EPI_COLS = 128;
  constexpr int STAGES = Plan::kStages;
  constexpr int SLOTS = Plan::kSfSlots;
  // cluster split-K (kFlagClusterSplit) is compiled into the dense and contiguous forms only
  constexpr bool kClusterCapable = MODE == kDense || MODE == kContiguous;
  static_assert(!SWIGLU || MODE == kMasked, "fused SwiGLU: masked form only");
  constexpr uint32_t kIdesc = make_idesc_e4m3_bs(128, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Plan::kBarOff);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* sf_full_bar = empty_bar + STAGES;      // [slot]: the slot's scale factors are in TMEM
  uint64_t* sf_empty_bar = sf_full_bar + SLOTS;    // [slot]: the MMAs reading the slot are done
  uint64_t* desc_full_bar = sf_empty_bar + SLOTS;  // [slot]: a tile description (or the end) is posted
  uint64_t* desc_empty_bar = desc_full_bar + Plan::kDescSlots;  // [slot]: every epilogue warp took it
  uint64_t* acc_full_bar = desc_empty_bar + Plan::kDescSlots;   // the tile's accumulator is complete
  uint64_t* acc_empty_bar = acc_full_bar + 1;      // every epilogue warp has loaded it
  uint64_t* epi_arrive_bar = acc_empty_bar + 1;    // split-K: all epilogue warps published a partial
  uint64_t* epi_release_bar = epi_arrive_bar + 1;  // split-K: the arrival count has been taken
  uint64_t* drain_bar = epi_release_bar + 1;       // abandon path: the MMAs issued have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Plan::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 8);
  // cluster split-K: set when an epilogue warp of this CTA ends without its partial (a skipped tile,
  // or a wait that gave up); the cluster then leaves D untouched
  volatile int* no_partial = reinterpret_cast<volatile int*>(smem + Plan::kMiscOff + 12);
  volatile int* desc_ring = reinterpret_cast<volatile int*>(smem + Plan::kDescOff);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int j = 0; j < SLOTS; ++j) {
      mbar_init(&sf_full_bar[j], 4);
      mbar_init(&sf_empty_bar[j], 1);
    }
    for (int j = 0; j < Plan::kDescSlots; ++j) {
      mbar_init(&desc_full_bar[j], 1);
      mbar_init(&desc_empty_bar[j], R::kEpiWarps);
    }
    mbar_init(acc_full_bar, 1);
    mbar_init(acc_empty_bar, R::kEpiWarps);
    mbar_init(epi_arrive_bar, R::kEpiWarps);
    mbar_init(epi_release_bar, 1);
    mbar_init(drain_bar, 1);
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
    tmem_alloc(tmem_slot, kBsTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // Programmatic dependent launch: the setup above reads no global memory that the previous kernel
  // in the stream may still be writing; the roles below do.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= R::kEpiWarps) {
    // ================================================================== scale / producer / MMA
    setmaxnreg_dec<R::kOtherRegs>();
    int tiles = p.num_tiles;
    if constexpr (MODE == kMasked) {
      if (warp <= R::kMmaWarp) tiles = masked_total_tiles(p, lane, blockIdx.x == 0 && warp == R::kProducerWarp);
    }
    const Sched sc = make_sched<BN, true, 300>(p, tiles, (int)gridDim.x);
    const int total_tiles = sc.units;
    if (warp == R::kProducerWarp) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t it = 0;
      bool alive = true;
      int issued_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
      const uint64_t policy = l2_policy_evict_last();
      for (int t = blockIdx.x; alive && t < total_tiles; t += gridDim.x) {
        const Tile tile = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile.skip) continue;
        // (K-grouped: B [K_total, N] is shared by the groups, and A's M coordinate is the m-block's)
        const int b_row = (MODE == kKGrouped ? 0 : tile.g * p.N) + tile.n_blk * BN;
        const int a_m = MODE == kKGrouped ? tile.m_blk * 128 : tile.a_row;
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
              tma_load_2d(&tmA, sa, &full_bar[s], a_m, kb * 128, policy);
            else
              tma_load_2d(&tmA, sa, &full_bar[s], kb * 128, tile.a_row, policy);
            if constexpr (SWIGLU) {
              // gate rows 128·n .. and up rows I + 128·n .. (B's tensor map box is 128 rows)
              const int gate_row = tile.g * p.N + tile.n_blk * 128;
              tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], kb * 128, gate_row, policy);
              tma_load_2d(&tmB, sa + Plan::kABytes + 128 * 128, &full_bar[s], kb * 128, gate_row + p.swiglu_i, policy);
            } else if (p.flags & kFlagBMN) {  // B stored [K, N]: two boxes of 128 K-rows x 128 N-bytes, 16 KB apart
              tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], b_row, kb * 128, policy);
              tma_load_2d(&tmB, sa + Plan::kABytes + 128 * 128, &full_bar[s], b_row + 128, kb * 128, policy);
            } else {
              tma_load_2d(&tmB, sa + Plan::kABytes, &full_bar[s], kb * 128, b_row, policy);
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
    } else if (warp == R::kMmaWarp) {
      // ---------------------------------------------------------------- block-scaled MMA issuer
      uint32_t it = 0, sf_it = 0, tile_it = 0;
      bool alive = true, issued_any = false;
      // An operand stored MN-major (the NN/TN/TT layouts) is read with an MN-major descriptor: one
      // K=32 step is +32 rows of 128 bytes (+256 in the >>4 address field) instead of +32 bytes.
      const bool a_mn = (p.flags & kFlagAMN) != 0, b_mn = (p.flags & kFlagBMN) != 0;
      const uint32_t a_step = a_mn ? 256u : 2u, b_step = b_mn ? 256u : 2u;
      const uint32_t idesc_layout = kIdesc | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
      for (int t = blockIdx.x; alive && t < total_tiles; t += gridDim.x) {
        const Tile tile = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile.skip) continue;
        int ok = 1;
        if (lane == 0) {
          // the epilogue has loaded the previous tile's accumulator
          ok = mbar_wait(acc_empty_bar, (tile_it & 1) ^ 1, abort_flag, p.status, p.flags);
          tc_fence_after();
          int cur_quad = -1;
          uint32_t slot = 0;
          for (int kb = tile.kb0; ok && kb < tile.kb1; ++kb, ++it) {
            const int quad = kb >> 2;
            if (quad != cur_quad) {
              slot = sf_it % SLOTS;
              ok = mbar_wait(&sf_full_bar[slot], (sf_it / SLOTS) & 1, abort_flag, p.status, p.flags);
              if (!ok) break;
              cur_quad = quad;
            }
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            ok = mbar_wait(&full_bar[s], ph, abort_flag, p.status, p.flags);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * Plan::kStageBytes);
            const uint64_t adesc = a_mn ? make_sw128_mnmajor_desc(a_addr, 128 * 128) : make_sw128_kmajor_desc(a_addr);
            const uint64_t bdesc = b_mn ? make_sw128_mnmajor_desc(a_addr + Plan::kABytes, 128 * 128)
                                        : make_sw128_kmajor_desc(a_addr + Plan::kABytes);
            const uint32_t idesc = idesc_with_sf_id(idesc_layout, (uint32_t)(kb & 3));
            const uint32_t sfa = tmem_base + kSfCol0 + slot * kSfSlotCols;
            const uint32_t sfb = sfa + kSfbOff;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // K-major: +32 bytes along K inside the 128-byte swizzled row (+2 in the >>4 field)
              mma_e4m3_block_scaled(tmem_base, adesc + a_step * k, bdesc + b_step * k, idesc, sfa, sfb,
                                    (kb > tile.kb0 || k > 0) ? 1u : 0u);
            }
            issued_any = true;
            mma_commit(&empty_bar[s]);
            if ((kb & 3) == 3 || kb + 1 == tile.kb1) {
              mma_commit(&sf_empty_bar[slot]);   // the slot is free once these MMAs are done
              ++sf_it;
              cur_quad = -1;
            }
          }
          if (ok) mma_commit(acc_full_bar);
        }
        ++tile_it;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { alive = false; break; }
      }
      if (!alive && lane == 0 && issued_any) {
        // Abandoned: wait for the MMAs already issued before TMEM is freed.
        mma_commit(drain_bar);
        const uint32_t a = smem_u32(drain_bar);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    } else if (warp < R::kScaleWarp0 + 4) {
      // ---------------------------------------------------------------- scale-factor writer
      // Warp 8 also posts each tile's description (then an end mark) for the epilogue, which
      // thereby never decodes tiles itself.
      const int q = warp % 4;                  // TMEM lane quadrant of this warp
      const int nkq = (p.nkb + 3) / 4;         // packed scale words along K
      const uint32_t lane_base = (uint32_t)(q * 32) << 16;
      const bool poster = (warp == R::kScaleWarp0);
      uint32_t sf_it = 0, desc_it = 0;
      bool alive = true;
      auto post = [&](const Tile& tl, int end) -> bool {
        const uint32_t ds = desc_it % Plan::kDescSlots;
        if (!mbar_wait(&desc_empty_bar[ds], ((desc_it / Plan::kDescSlots) & 1) ^ 1, abort_flag, p.status, p.flags))
          return false;
        if (lane == 0) {
          volatile int* d = desc_ring + ds * 8;
          d[0] = tl.g; d[1] = tl.m_blk; d[2] = tl.n_blk; d[3] = tl.split | (tl.splits << 16);
          d[4] = tl.out_idx; d[5] = tl.a_row; d[6] = tl.rows; d[7] = end;
          mbar_arrive(&desc_full_bar[ds]);
        }
        __syncwarp();
        ++desc_it;
        return true;
      };
      for (int t = blockIdx.x; alive && t < total_tiles; t += gridDim.x) {
        const Tile tile = decode_tile<BN, MODE>(p, sc, t, lane);
        if (tile.skip) continue;
        // (an empty K range, possible in the K-grouped form, is posted as such: the epilogue stores
        // zeros, and no scale slot is written for it)
        if (poster && !post(tile, tile.kb1 <= tile.kb0 ? 2 : 0)) { alive = false; break; }
        if (tile.kb1 <= tile.kb0) continue;
        const int row_in_tile = q * 32 + lane;
        const bool row_exists = row_in_tile < tile.rows;
        const int m_local = tile.m_blk * 128 + row_in_tile;
        const uint32_t* sfa_ptr = reinterpret_cast<const uint32_t*>(p.sA) + (MODE == kMasked ? (size_t)tile.g * nkq * p.ldsa : 0) + m_local;
        // the tile's two 128-row scale blocks of B: 2n and 2n + 1, or (SwiGLU) gate block n and up
        // block I/128 + n
        const int nb0 = SWIGLU ? tile.n_blk : tile.n_blk * 2;
        const uint32_t* sfb_ptr =
            reinterpret_cast<const uint32_t*>(p.sB) + ((size_t)(MODE == kKGrouped ? 0 : tile.g) * p.nnb + nb0) * nkq;
        const uint32_t* sfb1_ptr = SWIGLU ? sfb_ptr + (size_t)(p.swiglu_i / 128) * nkq : sfb_ptr + nkq;
        const bool has_nb1 = SWIGLU || nb0 + 1 < p.nnb;
        const int q_end = (tile.kb1 - 1) >> 2;
        for (int quad = tile.kb0 >> 2; quad <= q_end; ++quad, ++sf_it) {
          const uint32_t a = row_exists ? __ldg(sfa_ptr + (size_t)quad * p.ldsa) : 0x7F7F7F7Fu;
          const uint32_t b0 = __ldg(sfb_ptr + quad);
          const uint32_t b1 = has_nb1 ? __ldg(sfb1_ptr + quad) : 0x7F7F7F7Fu;
          const uint32_t slot = sf_it % SLOTS;
          if (!mbar_wait(&sf_empty_bar[slot], ((sf_it / SLOTS) & 1) ^ 1, abort_flag, p.status, p.flags)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t col = tmem_base + kSfCol0 + slot * kSfSlotCols;
          tmem_st_32x32b_x1(col + lane_base + (uint32_t)q, a);
          tmem_st_32x32b_x8(col + lane_base + kSfbOff, b0, b0, b0, b0, b1, b1, b1, b1);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_full_bar[slot]);
        }
      }
      if (poster && alive) {
        Tile end_mark;
        end_mark.g = end_mark.m_blk = end_mark.n_blk = end_mark.split = end_mark.out_idx = 0;
        end_mark.splits = 1;
        end_mark.a_row = end_mark.rows = 0;
        post(end_mark, 1);
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
    setmaxnreg_inc<R::kEpiRegs>();
    const int quad = warp % 4;              // TMEM lanes 32*quad .. 32*quad+31
    const int cgrp = warp / 4;              // columns EPI_COLS*cgrp .. of the tile
    const int row_in_tile = quad * 32 + lane;
    uint8_t* staging = smem + Plan::kStagingOff + warp * Plan::kStagingPerWarp;
    const uint32_t staging_addr = smem_u32(staging);
    uint32_t tile_it = 0, sk_it = 0, desc_it = 0;
    bool alive = true;
    uint32_t store_count = 0;

    // The tile description is parked in shared memory while the accumulator is loaded, so that
    // the 128 accumulator registers and the description are not live together.
    volatile int* stash = reinterpret_cast<volatile int*>(smem + Plan::kStashOff + warp * 64);

    bool have_partial = false;   // cluster split: this CTA's partial tile is in its stage buffers
    constexpr uint32_t kRowBytes = (BN + 4) * 4;   // partial rows in shared memory, +16 bytes: all banks
    static_assert(128 * kRowBytes <= STAGES * Plan::kStageBytes, "partial tile exceeds the stage buffers");
    while (alive) {
      // the next tile's description, copied into this warp's stash before its slot is released
      bool active, empty_k = false;
      {
        const uint32_t ds = desc_it % Plan::kDescSlots;
        if (!mbar_wait(&desc_full_bar[ds], (desc_it / Plan::kDescSlots) & 1, abort_flag, p.status, p.flags)) {
          alive = false;
          break;
        }
        ++desc_it;
        const volatile int* d = desc_ring + ds * 8;
        const int end = d[7];   // 1: no more tiles; 2: a tile with an empty K range (zeros)
        const int n_blk0 = d[2], rows0 = d[6];
        if (lane < 7) stash[lane] = d[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&desc_empty_bar[ds]);
        if (end == 1) break;
        empty_k = end == 2;
        active = (SWIGLU || n_blk0 * BN + cgrp * EPI_COLS < p.N) && __any_sync(0xffffffffu, row_in_tile < rows0);
      }
      // this warp's 32x128 block of the accumulator (live only within one tile)
      uint32_t accu[EPI_COLS];
      float* const acc = reinterpret_cast<float*>(accu);

      if (!mbar_wait(acc_full_bar, tile_it & 1, abort_flag, p.status, p.flags)) { alive = false; break; }
      ++tile_it;
      tc_fence_after();
      if (active) {
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
#pragma unroll
        for (int c = 0; c < EPI_COLS / 32; c += 2) {
          uint32_t(&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&accu[c * 32]);
          uint32_t(&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&accu[(c + 1) * 32]);
          // SwiGLU: registers 0..63 take gate columns 64·cgrp.., registers 64..127 the matching up
          // columns 128 + 64·cgrp..; otherwise the warp's 128 columns in order
          const uint32_t col = SWIGLU ? (uint32_t)((c == 0 ? 0 : 128) + cgrp * 64) : (uint32_t)(cgrp * EPI_COLS + c * 32);
          tmem_ld_32x32b_x32(lane_addr + col, r0);
          tmem_ld_32x32b_x32(lane_addr + col + 32, r1);
          tmem_ld_wait(r0);
          reg_fence(r1);
        }
      }
      // the accumulator is in registers: the MMA may start the next tile
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty_bar);
      if (empty_k) {
        // an empty K range: nothing was accumulated (the tensor memory holds the previous tile)
#pragma unroll
        for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;
      }
      Tile tile;
      tile.g = stash[0]; tile.m_blk = stash[1]; tile.n_blk = stash[2];
      tile.split = stash[3] & 0xFFFF; tile.splits = stash[3] >> 16;   // (split, splits) packed in one int
      tile.out_idx = stash[4]; tile.a_row = stash[5]; tile.rows = stash[6];
      const int m_local = tile.m_blk * 128 + row_in_tile;
      const bool row_exists = row_in_tile < tile.rows;
      const int n_col0 = tile.n_blk * BN + cgrp * EPI_COLS;
      const bool col_exists = n_col0 < p.N;

      if (kClusterCapable && (p.flags & kFlagClusterSplit)) {
        // one unit per CTA: the partial goes to this CTA's stage buffers (idle once the MMA is
        // done) and the reduction follows the loop. Rows or columns outside the tile (a warp that
        // loaded nothing) are written but never read.
        const uint32_t part = smem_u32(smem);
#pragma unroll
        for (int j = 0; j < EPI_COLS; j += 4)
          st_shared_v4(part + row_in_tile * kRowBytes + (cgrp * EPI_COLS + j) * 4, accu[j], accu[j + 1], accu[j + 2],
                       accu[j + 3]);
        have_partial = true;
        break;
      }

      // ---------------- split-K: publish the partial, and let the last split reduce
      if (tile.splits > 1) {
        float* ws_tile = p.workspace + (size_t)tile.out_idx * tile.splits * (128 * BN);
        float* mine = ws_tile + (size_t)tile.split * (128 * BN);
        if (row_exists && col_exists) {
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

      // (fused SwiGLU: the split-K step above publishes and reduces each warp's 64 gate and 64 up
      // columns under its own 128 slots of the partial tile, so the last split holds both)
      if constexpr (SWIGLU) {
        // H = silu(gate)·up for this warp's 64 of the tile's 128 columns of H (row stride I)
        if (!active || !__any_sync(0xffffffffu, row_exists)) continue;
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = silu_f32(acc[j]) * acc[64 + j];
        const int h_col0 = tile.n_blk * 128 + cgrp * 64;
        if (__all_sync(0xffffffffu, row_exists)) {
          constexpr int kColsPerBox = OUT_F32 ? 16 : 32;
#pragma unroll
          for (int chunk = 0; chunk < 64 / kColsPerBox; ++chunk) {
            const uint32_t sel = store_count & 1;
            if (store_count >= 2) {
              if (lane == 0) tma_store_wait_read_1();
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w0, w1, w2, w3;
              if constexpr (OUT_F32) {
                const int c = chunk * 16 + j * 4;
                w0 = accu[c]; w1 = accu[c + 1]; w2 = accu[c + 2]; w3 = accu[c + 3];
              } else {
                const int c = chunk * 32 + j * 8;
                w0 = pack_bf16x2(acc[c], acc[c + 1]); w1 = pack_bf16x2(acc[c + 2], acc[c + 3]);
                w2 = pack_bf16x2(acc[c + 4], acc[c + 5]); w3 = pack_bf16x2(acc[c + 6], acc[c + 7]);
              }
              const uint32_t phys = (uint32_t)(j ^ ((lane >> 1) & 3));
              st_shared_v4(staging_addr + sel * Plan::kStagingBox + lane * 64 + phys * 16, w0, w1, w2, w3);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, staging + sel * Plan::kStagingBox, h_col0 + chunk * kColsPerBox, tile.a_row + quad * 32);
              tma_store_commit();
            }
            ++store_count;
            __syncwarp();
          }
        } else if (row_exists) {
          // predicated plain stores: rows past masked_m stay untouched
          const size_t hrow = (size_t)(tile.a_row + row_in_tile) * p.swiglu_i + h_col0;
          if constexpr (OUT_F32) {
            float* dst = reinterpret_cast<float*>(p.D) + hrow;
#pragma unroll
            for (int j = 0; j < 64; j += 4)
              *reinterpret_cast<float4*>(dst + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
          } else {
            uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + hrow;
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
              uint4 v;
              v.x = pack_bf16x2(acc[j], acc[j + 1]); v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
              v.z = pack_bf16x2(acc[j + 4], acc[j + 5]); v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
              *reinterpret_cast<uint4*>(dst + j) = v;
            }
          }
        }
        continue;
      }

      // ---------------- output
      bool write_row;
      if constexpr (MODE == kContiguous) {
        write_row = false;
        if (row_exists) {
          const int idx = __ldg(p.m_indices + m_local);
          write_row = (idx == tile.g);
          if (idx != tile.g && idx != -1) atomicOr(p.status, kStatusBadGroup);
        }
      } else {
        write_row = row_exists;
      }
      const int d_row = tile.a_row + row_in_tile;
      if (!__any_sync(0xffffffffu, write_row)) continue;   // no row of this warp is stored
      const bool use_tma = (MODE == kDense) || __all_sync(0xffffffffu, write_row);
      if (!col_exists) continue;
      if (use_tma) {
        constexpr int kColsPerBox = OUT_F32 ? 16 : 32;
#pragma unroll
        for (int chunk = 0; chunk < EPI_COLS / kColsPerBox; ++chunk) {
          if (n_col0 + chunk * kColsPerBox >= p.N) break;
          const uint32_t sel = store_count & 1;
          if (store_count >= 2) {
            if (lane == 0) tma_store_wait_read_1();
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w0, w1, w2, w3;
            if constexpr (OUT_F32) {
              const int c = chunk * 16 + j * 4;
              w0 = accu[c]; w1 = accu[c + 1]; w2 = accu[c + 2]; w3 = accu[c + 3];
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
      // Split-K in a cluster, as in the FP32-scale kernel: the S CTAs of the cluster hold the S K
      // ranges of one tile (rank = range); after a cluster barrier each sums the rows r with
      // r % S = rank in range order from its peers' shared memory and stores them; a second barrier
      // keeps every CTA's shared memory in place until its peers have read it. Every thread of the
      // cluster reaches both barriers on every path.
      const uint32_t part = smem_u32(smem);
      if (!have_partial && lane == 0) *no_partial = 1;
      cluster_sync_all();
      // Sum only if every CTA of the cluster holds its partial: a CTA that gave up (a wait timed out)
      // has none, and its stage buffers hold stale bytes that must not reach D.
      const bool complete = cluster_all_zero_u32(smem_u32(const_cast<int*>(no_partial))) && have_partial;
      if (complete) {
        const int S = stash[3] >> 16, g = stash[0], n_blk = stash[2], a_row = stash[5], rows = stash[6];
        const int rank = (int)cluster_ctarank();
        constexpr int kVec = BN / 4;                       // float4 per row
        constexpr int kRowsPerPass = R::kEpiThreads / kVec;
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
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kBsTmemCols);
  }
}

}  // namespace dg
