// dg_ptx.cuh — inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (cp.async.bulk.tensor) loads and stores, and the tcgen05 tensor-core / tensor-memory
// instructions. Everything here is a thin, documented wrapper around one PTX instruction.
#pragma once

#include <cstdint>

#include <cuda_fp8.h>

namespace dg {

// ---------------------------------------------------------------------------------------------
// Addresses and misc.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// ---------------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bound of the drain waits on an abandoned path (the copies and MMAs already in flight): they do
// not use the caller's limit below, so that in-flight work is always waited for.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kStatusTimeout = 0x4;
// The time limit of every pipeline wait travels in bits 8..31 of the kernel's flags word, in
// microseconds (the host sets it; default 2 s, up to about 16.7 s). No legitimate wait comes near
// the default; when a wait exceeds the limit, the kernel records DG_DEV_TIMEOUT, raises the CTA's
// abort flag and unwinds.
constexpr int kWaitLimitShift = 8;

// Waits until the phase with the given parity of `bar` has completed. Returns false (and sets
// *abort) if the CTA's abort flag is raised or the time limit in `flags` passes; the caller then
// unwinds. The limit is only read once the phase was not already complete.
//
// The loop polls with try_wait and no suspend-time hint: the hardware may park the thread for a
// short, system-defined time inside each poll, and the poll returns as soon as the phase
// completes. A thread parked with a long explicit hint resumes some hundreds of cycles after the
// phase completes; measured on GB300, that made up about a quarter of the per-K-block
// MMA -> epilogue -> MMA handshake of the FP32-scale kernel with the loads and promotion
// removed (908 -> 671 cycles), and about 3% of the full kernel.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                          int flags) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t limit_ns = (uint64_t)((uint32_t)flags >> kWaitLimitShift) * 1000ull;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    // (a limit of 0 gives up at once on a phase that is not already complete)
    if (limit_ns != 0) {
#pragma unroll 1
      for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(a, parity)) return true;
    }
    if (*abort) return false;
    if (global_timer_ns() - t0 >= limit_ns) {
      atomicOr(status, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Thread-block clusters

// Cluster-wide barrier: every thread of every CTA of the cluster arrives, then waits. Writes to
// shared memory before it are visible to the cluster's reads after it (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address, in the cluster's shared-memory window, of `addr` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Two FP32 values as E4M3 codes (round to nearest even, saturating to ±448), `first` in the low
// byte, through CUDA's conversion intrinsic.
__device__ __forceinline__ uint32_t e4m3x2_satfinite(float first, float second) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(first, second), __NV_SATFINITE, __NV_E4M3);
}

// Largest cluster the split-K exchange uses (the portable cluster size).
constexpr int kMaxClusterCtas = 8;

// True if the u32 at `addr` (an address in this CTA's shared memory) is 0 in every CTA of the
// cluster. All the loads are in flight together, so the check costs one round trip through
// distributed shared memory rather than one per CTA.
__device__ __forceinline__ bool cluster_all_zero_u32(uint32_t addr) {
  const uint32_t n = cluster_nctarank();
  uint32_t v[kMaxClusterCtas];
#pragma unroll
  for (int r = 0; r < kMaxClusterCtas; ++r) v[r] = (uint32_t)r < n ? ld_cluster_u32(cluster_map(addr, (uint32_t)r)) : 0u;
  uint32_t any = 0;
#pragma unroll
  for (int r = 0; r < kMaxClusterCtas; ++r) any |= v[r];
  return any == 0;
}

// The sum over cluster ranks 0..S-1 (S <= kMaxClusterCtas) of the float4 at `addr` in each CTA's
// shared memory, added in rank order starting from zero. The S loads are issued before the first
// add, so they overlap instead of each waiting for the previous one.
__device__ __forceinline__ float4 cluster_sum_v4(uint32_t addr, int S) {
  float4 v[kMaxClusterCtas];
#pragma unroll
  for (int s = 0; s < kMaxClusterCtas; ++s)
    if (s < S) v[s] = ld_cluster_v4(cluster_map(addr, (uint32_t)s));
  float4 tot = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
  for (int s = 0; s < kMaxClusterCtas; ++s) {
    if (s < S) {
      tot.x += v[s].x; tot.y += v[s].y; tot.z += v[s].z; tot.w += v[s].w;
    }
  }
  return tot;
}

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with programmatic stream serialization may start
// before the kernel ahead of it in the stream has finished; griddep_wait() then blocks until that
// kernel has completed and its memory operations are visible. Without the launch attribute both
// instructions do nothing.

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream (if launched for it) begin its own launch while this one runs.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// TMA (tensor maps are __grid_constant__ kernel parameters)

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = outer) into shared memory; completion
// is signalled as transaction bytes on `bar`. Out-of-bounds elements are zero-filled.
__device__ __forceinline__ void tma_load_2d(const void* tmap, void* smem_dst, uint64_t* bar, int x, int y,
                                            uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(cache_policy)
      : "memory");
}

// As tma_load_2d, but the box is written to the same shared-memory offset in every CTA of the
// cluster named in `cta_mask`, and each of those CTAs' barrier at `bar`'s offset receives the
// transaction bytes (this GPU's own memory only).
__device__ __forceinline__ void tma_load_2d_multicast(const void* tmap, void* smem_dst, uint64_t* bar, int x, int y,
                                                      uint16_t cta_mask, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(cta_mask), "l"(cache_policy)
      : "memory");
}

// 2-D tiled store of a shared-memory box to global memory at (x, y); elements outside the
// tensor's bounds are not written.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}

// 2-D tiled reduce-add of a shared-memory box into global memory at (x, y): every element of the
// box is added to the tensor element it lands on (the tensor map's type, here FP32); elements
// outside the tensor's bounds are skipped.
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, const void* smem_src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until every committed store group has finished reading its shared-memory source.
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until at most one committed store group is still reading its shared-memory source.
__device__ __forceinline__ void tma_store_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until every committed store group is complete (written to global memory).
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core

// Allocates `ncols` TMEM columns (power of two, >= 32) for this CTA; the TMEM address is written
// to shared memory at `slot`. Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte swizzle:
// rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart (stride byte offset), tile base
// 1024-byte aligned. Fields: start address >> 4 [0,14), leading byte offset >> 4 [16,30) (unused
// for swizzled K-major, set to 1), stride byte offset >> 4 [32,46), descriptor version 1 at bit
// 46, base offset 0 [49,52), swizzle mode [61,64) = 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t make_sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Shared-memory matrix descriptor of an MN-major operand tile stored with the 128-byte swizzle, as a
// TMA box of 128 K-rows x 128 bytes (M or N) writes it: 8-row swizzle atoms along K 1024 bytes apart
// (stride byte offset) and `atom_stride` bytes between 128-byte-wide atoms along M/N (leading byte
// offset; unused when the tile is one atom wide). One K=32 step advances the start by 32 rows = 4096
// bytes. (Layout measured on GB300 against exact integer products.)
__device__ __forceinline__ uint64_t make_sw128_mnmajor_desc(uint32_t smem_addr, uint32_t atom_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((atom_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B, FP32 accumulator, both K-major,
// shape M x N: D format [4,6) = 1 (F32), A format [7,10) = 0 (E4M3), B format [10,13) = 0 (E4M3),
// A/B major bits 15/16 = 0 (K-major), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t make_idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D(tmem) (+)= A(smem) · B(smem)ᵀ for one K=32 step of E4M3 operands. Issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// As mma_commit, but the arrival goes to the barrier at `bar`'s offset in every CTA of the cluster
// named in `cta_mask`.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(cta_mask)
               : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 A and B (formats [7,10) and
// [10,13) = 0), both K-major, FP32 accumulator, N >> 3 at [17,23), scale-factor type UE8M0 at bit
// 23, M >> 7 at [27,29). The scale-factor IDs (which byte of the 32-bit TMEM cell the MMA reads:
// B at [4,6), A at [29,31)) are added per K-block.
__host__ __device__ constexpr uint32_t make_idesc_e4m3_bs(uint32_t M, uint32_t N) {
  return ((N >> 3) << 17) | (1u << 23) | ((M >> 7) << 27);
}

__host__ __device__ constexpr uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t sf_id) {
  return idesc | (sf_id << 29) | (sf_id << 4);
}

// D(tmem) (+)= (A·sfA)(smem) · (B·sfB)(smem)ᵀ for one K=32 step of E4M3 operands, each row of A and
// of B multiplied by its UE8M0 scale factor read from TMEM (one scale per 32 K-elements:
// scale_vec::1X). Issued by one thread.
__device__ __forceinline__ void mma_e4m3_block_scaled(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                      uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Stores one 32-bit column of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Stores eight consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3,
                                                  uint32_t v4, uint32_t v5, uint32_t v6, uint32_t v7) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(v0),
               "r"(v1), "r"(v2), "r"(v3), "r"(v4), "r"(v5), "r"(v6), "r"(v7)
               : "memory");
}

// Waits until this thread's tcgen05.st have completed.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Loads 32 consecutive FP32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld. The 32 destination registers of the load are
// tied to the wait as read-write operands so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Ties 32 registers to this point of the instruction stream (no instruction is emitted): no use
// of them can be scheduled before an earlier volatile asm such as tmem_ld_wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ---------------------------------------------------------------------------------------------
// Packed FP32x2 arithmetic (sm_100+): one instruction, two lanes of FP32 fused multiply-add.

// Two FP32 values packed in one 64-bit register pair (low = first).
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo, uint32_t hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(lo), "r"(hi));
  return v;
}

__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// acc += a * s on both lanes of packed FP32 pairs (one fma.rn.f32x2; IEEE fused, round to nearest).
__device__ __forceinline__ void ffma2_acc(uint64_t& acc, uint64_t a, uint64_t s) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(s));
}

__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float s) {
  uint64_t acc, av, sv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(d0), "f"(d1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(av), "l"(sv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(acc));
}

}  // namespace dg
