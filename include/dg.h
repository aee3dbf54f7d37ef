/*
 * dg.h — C ABI of libdg: FP8 (E4M3) GEMM D = A·Bᵀ with DeepSeek-V3 fine-grained scaling on
 * GB300 (sm_103a), in its dense form and the two MoE grouped forms.
 *
 * What the calls compute (sources are the DeepGEMM pages; the scale granularity is from the
 * DeepSeek-V3 Technical Report, § 3.3.2 "Fine-Grained Quantization"):
 *
 *   D[m,n] = Σ_kb  sA[m,kb] · sB[n/128,kb] · Σ_{k in kb} A[m,k]·B[n,k]        kb = k/128
 *
 * - "NT" naming and layout: fp8_gemm_nt computes D = C + A @ B.T, A row-major, B col-major
 *   ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
 *   tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları"). C is absent: D is
 *   overwritten.
 * - The per-128-K partial is promoted into an FP32 accumulator after the scales are applied
 *   (two-level accumulation on CUDA cores: "DeepGEMM" first-release summary,
 *   tr.news.hada.io/topic?id=19444, feature list).
 * - The LHS scaling factor is TMA-aligned and transposed (same page as the NT naming, same
 *   section), i.e. MN-major.
 *
 * Common conventions for every GEMM entry point:
 * - Pointers: all tensor pointers are DEVICE memory owned by the caller. libdg keeps no pointer
 *   after the call returns. Calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and never synchronise.
 * - A: E4M3 bytes, row-major [rows, K] (K contiguous). B: E4M3 bytes, [G, N, K] (K contiguous;
 *   dense G = 1). E4M3 is the OCP FP8 format (bias 7, 0x7F/0xFF NaN, max 448).
 * - sA: FP32, MN-major: sA[kb * ldsa + m] with ldsa = dg_get_tma_aligned_size(rows, 4)
 *   (rows rounded up to a multiple of 4), kb in [0, ceil(K/128)).
 * - sB: FP32, sB[(g * ceil(N/128) + nb) * ceil(K/128) + kb], one scale per 128x128 block.
 * - D: row-major [rows, N]; BF16 bit patterns (uint16_t) rounded to nearest-even, or FP32 for
 *   the *_f32 variants. The *_f32 variants run the same kernel with the same tile
 *   configuration and accumulation order and store the FP32 accumulator instead of rounding it:
 *   D_bf16 == RNE(D_f32) element by element.
 * - Alignment (TMA: 16-byte global strides and addresses): K % 16 == 0, N % 8 == 0 (BF16 D) or
 *   N % 4 == 0 (FP32 D); A, B and D 16-byte aligned; sA, sB 4-byte aligned.
 *   Violations return DG_ERR_ALIGNMENT or DG_ERR_INVALID_ARG and launch nothing.
 * - Empty problems (a zero M/N/G) return DG_OK and launch nothing.
 * - Errors found on the device (a group index out of range, masked_m outside [0, M_max], a
 *   pipeline wait that timed out) never trap: the kernel skips the affected rows or tiles, sets
 *   bits of a device status word and returns. Read it with dg_get_device_status().
 * - Split-K: for small problems the library may split K across CTAs and reduce the FP32
 *   partials in a fixed order (deterministic). Where the ranges of every tile fit on the GPU at
 *   once as thread-block clusters, they reduce through distributed shared memory and use no
 *   workspace (dg_set_cluster_split). Otherwise, and for the tail split (dg_set_tail_splits), the
 *   partials go to a library-owned buffer per device. It is allocated on the first call that needs
 *   it and grown when a larger one is needed; that call allocates, so make it before any CUDA-graph
 *   capture. Calls that use the workspace and overlap on the GPU (different streams of one device)
 *   race on it. The first call that considers clusters for a kernel also queries, once per device,
 *   how many of its clusters fit (cudaOccupancyMaxActiveClusters; no launch, no allocation).
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad G */
  DG_ERR_ALIGNMENT = 2,      /* K % 16, N % 8 (N % 4 for FP32 D), or pointer alignment */
  DG_ERR_UNSUPPORTED = 3,    /* no GB300-class device, or a size beyond a documented limit */
  DG_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed; see dg_last_error_string() */
  DG_ERR_DEVICE_STATUS = 5   /* dg_get_device_status() found a non-zero device status word */
} dg_status;

/* Bits of the device status word. */
#define DG_DEV_BAD_GROUP_INDEX 0x1  /* contiguous: m_indices[m] >= G or < -1, or two groups in one 128-row block */
#define DG_DEV_BAD_MASKED_M 0x2     /* masked: masked_m[g] < 0 or > M_max (clamped) */
#define DG_DEV_TIMEOUT 0x4          /* a pipeline wait exceeded its time limit; the kernel abandoned the work */
#define DG_DEV_BAD_SCALE 0x8        /* dg_transform_sf_into_ue8m0_*: a scale was not a power of two in [2^-127, 2^127] */

typedef void* dg_stream_t; /* cudaStream_t */

/*
 * Dense GEMM: D[M,N] = A[M,K]·B[N,K]ᵀ with fine-grained scales.
 * Source: fp8_gemm_nt ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
 * tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları" and § "Dense ve Grouped
 * GEMM").
 *   A  [M,K] E4M3          sA [ceil(K/128)][align4(M)] FP32 (MN-major)
 *   B  [N,K] E4M3          sB [ceil(N/128)][ceil(K/128)] FP32
 *   D  [M,N] BF16 bits
 */
dg_status dg_fp8_gemm_nt(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                         uint16_t* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_nt_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                             float* D, int M, int N, int K, dg_stream_t stream);

/*
 * Contiguous-layout grouped GEMM: grouped along M only; N and K are shared by the G groups
 * (experts). The experts' token rows are concatenated into one A, and each expert's segment is
 * aligned to the GEMM M block, dg_get_mk_alignment_for_contiguous_layout() = 128 rows.
 * Source: tr.news.hada.io/topic?id=19459, § "Dense ve Grouped GEMM"; first-release summary
 * tr.news.hada.io/topic?id=19444, § "MoE modelleri için gruplanmış GEMM performansı".
 *   A  [M_total,K] E4M3     sA [ceil(K/128)][align4(M_total)]
 *   B  [G,N,K] E4M3         sB [G][ceil(N/128)][ceil(K/128)]
 *   m_indices [M_total] int32 on the device: the group of each row, or -1 for a padding row.
 *             Every 128-row block must hold one group (plus -1 rows). Padding rows of D are
 *             left untouched; an all-padding block is skipped without reading B. An index
 *             >= G or < -1 sets DG_DEV_BAD_GROUP_INDEX and leaves that row (or block) untouched.
 *   D  [M_total,N] BF16 bits
 */
dg_status dg_fp8_grouped_contiguous(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                    const int32_t* m_indices, uint16_t* D, int M_total, int N, int K,
                                    int G, dg_stream_t stream);
dg_status dg_fp8_grouped_contiguous_f32(const uint8_t* A, const float* sA, const uint8_t* B,
                                        const float* sB, const int32_t* m_indices, float* D,
                                        int M_total, int N, int K, int G, dg_stream_t stream);

/*
 * Masked-layout grouped GEMM (MoE decode under CUDA graphs: the CPU does not know how many
 * tokens each expert received, so the counts are read on the device and only the valid rows are
 * computed). Source: tr.news.hada.io/topic?id=19459, § "Dense ve Grouped GEMM"
 * (m_grouped_fp8_gemm_nt_masked); tr.news.hada.io/topic?id=19444, § "MoE modelleri için
 * gruplanmış GEMM performansı".
 *   A  [G,M_max,K] E4M3     sA [G][ceil(K/128)][align4(M_max)]
 *   B  [G,N,K] E4M3         sB [G][ceil(N/128)][ceil(K/128)]
 *   masked_m [G] int32 on the device: valid rows of each group. Rows m >= masked_m[g] of D are
 *             never written; a group with masked_m[g] == 0 reads neither A nor B. Values outside
 *             [0, M_max] are clamped and set DG_DEV_BAD_MASKED_M.
 *   D  [G,M_max,N] BF16 bits
 * The host never reads masked_m, so the call can be captured in a CUDA graph.
 */
dg_status dg_fp8_grouped_masked(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                const int32_t* masked_m, uint16_t* D, int G, int M_max, int N, int K,
                                dg_stream_t stream);
dg_status dg_fp8_grouped_masked_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                    const int32_t* masked_m, float* D, int G, int M_max, int N, int K,
                                    dg_stream_t stream);

/*
 * Packed-UE8M0 variants: the same three GEMMs when every scale is a power of two, given as UE8M0
 * codes (OCP MX E8M0: value 2^(e-127); 0xFF is NaN) packed four to a 32-bit word, the scale form
 * the DeepGEMM SM100 kernels take ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM
 * çekirdekleri", tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları": the
 * SM100 implementation wants packed UE8M0, four UE8M0 values in one torch.int). The granularity is
 * unchanged: one scale per 1x128 K-group of each A row and one per 128x128 block of B.
 *   Packing: byte j (bits 8j..8j+7) of word q holds K-group 4q+j; unused bytes past ceil(K/128)
 *   are ignored.
 *   sA: int32, MN-major: sA[(g * ceil(nkb/4) + q) * ldsa + m], ldsa = dg_get_tma_aligned_size(rows, 4)
 *       (dense and contiguous: g = 0), nkb = ceil(K/128).
 *   sB: int32, sB[(g * ceil(N/128) + nb) * ceil(nkb/4) + q].
 * Because such scales are powers of two, the tensor core applies them itself (block-scaled MMA,
 * tcgen05.mma kind::mxf8f6f4 with scale_vec::1X) and the K loop accumulates in one FP32 TMEM
 * accumulator: there is no per-128-K promotion on CUDA cores, so the FP32 result can differ from
 * the FP32-scale calls' in its rounding, not in its value. Every other convention (layouts,
 * alignment, errors, device status, split-K workspace, the *_f32 variants) is that of the
 * corresponding FP32-scale call. The tile width is always 256 columns.
 */
dg_status dg_fp8_gemm_nt_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                               uint16_t* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_nt_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                   float* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_grouped_contiguous_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                          const int32_t* sB, const int32_t* m_indices, uint16_t* D,
                                          int M_total, int N, int K, int G, dg_stream_t stream);
dg_status dg_fp8_grouped_contiguous_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                              const int32_t* sB, const int32_t* m_indices, float* D,
                                              int M_total, int N, int K, int G, dg_stream_t stream);
dg_status dg_fp8_grouped_masked_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                      const int32_t* masked_m, uint16_t* D, int G, int M_max, int N, int K,
                                      dg_stream_t stream);
dg_status dg_fp8_grouped_masked_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                          const int32_t* sB, const int32_t* masked_m, float* D, int G, int M_max,
                                          int N, int K, dg_stream_t stream);

/*
 * Dense GEMM in the other layouts. The SM100 implementation supports the NT, TN, NN and TT layouts
 * (fp8_gemm_{nt, nn, tn, tt}: "DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM
 * çekirdekleri", tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları" and
 * § "Dense ve Grouped GEMM"). The product is always D[M,N] = A·Bᵀ of the logical A[M,K] and B[N,K];
 * the letters say how A and B are stored:
 *   nt (dg_fp8_gemm_nt): A [M,K], B [N,K]  (both K-contiguous)
 *   nn:                  A [M,K], B [K,N]  (B N-contiguous)
 *   tn:                  A [K,M], B [K,N]  (both M/N-contiguous: e.g. weight gradients over tokens)
 *   tt:                  A [K,M], B [N,K]
 * The scales keep the logical granularity and layouts of dg_fp8_gemm_nt: sA [ceil(K/128)][align4(M)]
 * (one per 1x128 K-group of each logical row of A), sB [ceil(N/128)][ceil(K/128)]. A stored [K,M]
 * needs M % 16 == 0; B stored [K,N] needs N % 16 == 0 (16-byte TMA strides). The tensor core reads
 * the M/N-contiguous tiles directly (no transposition pass). Other conventions as dg_fp8_gemm_nt.
 */
dg_status dg_fp8_gemm_nn(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D,
                         int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_nn_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D,
                             int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tn(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D,
                         int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tn_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D,
                             int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tt(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, uint16_t* D,
                         int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tt_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, float* D,
                             int M, int N, int K, dg_stream_t stream);

/* The NN, TN and TT layouts with power-of-two scales packed as UE8M0 (the block-scaled kernel):
   the storage of A and B as for dg_fp8_gemm_nn / _tn / _tt, the packed scale layouts of
   dg_fp8_gemm_nt_ue8m0 (sA [ceil(ceil(K/128)/4)][align4(M)], sB [ceil(N/128)][ceil(ceil(K/128)/4)]).
   Each gives the NT call's result bit for bit. The pages list the four layouts for the SM100
   implementation, which takes packed UE8M0 scales (same page, § "GEMM arayüzü ve yerleşim
   kısıtları"). */
dg_status dg_fp8_gemm_nn_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                               uint16_t* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_nn_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                   float* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tn_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                               uint16_t* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tn_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                   float* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tt_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                               uint16_t* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_tt_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B, const int32_t* sB,
                                   float* D, int M, int N, int K, dg_stream_t stream);

/*
 * K-grouped contiguous GEMM (MoE weight backward): grouped along K, with M and N shared by the groups
 * (k_grouped_fp8_gemm_tn_contiguous, tr.news.hada.io/topic?id=19459, § "Dense ve Grouped GEMM").
 * The experts' token segments are concatenated along K; segment g is k in [k_offsets[g],
 * k_offsets[g+1]), and D[g] = Σ over it of A[k,:]ᵀ·B[k,:] with the scales of those K-blocks:
 *   A  [K_total, M] E4M3 (M contiguous)    sA [K_total/128][align4(M)] FP32 (1x128 K-groups of each m)
 *   B  [K_total, N] E4M3 (N contiguous)    sB [ceil(N/128)][K_total/128] FP32 (128x128 blocks)
 *   k_offsets [G+1] int32 on the device: non-decreasing multiples of 128, k_offsets[G] <= K_total
 *   D  [G, M, N] BF16 bits (or FP32 for _f32). An empty segment gives D[g] = 0.
 * M and N must be multiples of 16 and K_total of 128. Offsets that break these rules set
 * DG_DEV_BAD_GROUP_INDEX and leave D[g] of that group untouched. The host never reads k_offsets.
 */
dg_status dg_fp8_k_grouped_gemm_tn_contiguous(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                              const int32_t* k_offsets, uint16_t* D, int G, int M, int N,
                                              int K_total, dg_stream_t stream);
dg_status dg_fp8_k_grouped_gemm_tn_contiguous_f32(const uint8_t* A, const float* sA, const uint8_t* B,
                                                  const float* sB, const int32_t* k_offsets, float* D, int G, int M,
                                                  int N, int K_total, dg_stream_t stream);
/* The K-grouped form with power-of-two scales packed as UE8M0, on the block-scaled kernel: A, B,
   k_offsets and D as above; sA [ceil(K_total/512)][align4(M)] and sB [ceil(N/128)][ceil(K_total/512)]
   int32, four 128-deep K-blocks per word along the whole K_total axis (a group whose offset is not a
   multiple of 512 starts inside a word; the kernel picks each K-block's byte). An empty group stores
   zeros. */
dg_status dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                    const int32_t* sB, const int32_t* k_offsets, uint16_t* D, int G,
                                                    int M, int N, int K_total, dg_stream_t stream);
dg_status dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                        const int32_t* sB, const int32_t* k_offsets, float* D, int G,
                                                        int M, int N, int K_total, dg_stream_t stream);

/*
 * Masked grouped GEMM fused with SwiGLU (MoE decode): the up/gate projection of each expert and the
 * SwiGLU after it in one kernel, so the 2I-wide intermediate never reaches memory. It is the first
 * fusion of the pages' Mega MoE, which fuses linear 1, SwiGLU and linear 2 of the experts
 * (tr.news.hada.io/topic?id=19459, § "Mega MoE"); here on one GPU with FP8 weights and FP32 scales.
 *   A  [G,M_max,K] E4M3     sA [G][ceil(K/128)][align4(M_max)]      (as dg_fp8_grouped_masked)
 *   B  [G,N,K] E4M3 with N = 2I: rows [0, I) are the gate projection, rows [I, 2I) the up projection
 *      (I a multiple of 128)                                        sB [G][N/128][ceil(K/128)]
 *   masked_m [G] int32 on the device (as dg_fp8_grouped_masked)
 *   H  [G,M_max,I] BF16 bits (or FP32 for the _f32 variant):
 *      H[g,m,j] = silu(D[g,m,j]) · D[g,m,I+j],  D = the masked GEMM,  silu(x) = x / (1 + e^-x)
 *      (SwiGLU as defined by Shazeer, "GLU Variants Improve Transformer", 2020)
 *   Rows m >= masked_m[g] of H are never written. The FP32-scale kernel computes D in FP32 and H in FP32
 *   (silu with the fast exponential and division, relative error ~1e-6), then rounds H to BF16 once:
 *   H_bf16 == RNE(H_f32). Like the masked GEMM it may cut the tiles of a last, partial wave along K
 *   (dg_set_tail_splits), using the library's workspace.
 */
dg_status dg_fp8_grouped_masked_swiglu(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                       const int32_t* masked_m, uint16_t* H, int G, int M_max, int N, int K,
                                       dg_stream_t stream);
dg_status dg_fp8_grouped_masked_swiglu_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                           const int32_t* masked_m, float* H, int G, int M_max, int N, int K,
                                           dg_stream_t stream);
/* The fused SwiGLU with H cast to FP8 for the down projection. The Mega MoE kernel runs linear 1,
   the SwiGLU and linear 2 back to back, and linear 2 takes FP8 activations ("DeepGEMM: İnce
   ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri", tr.news.hada.io/topic?id=19459,
   § "Mega MoE"); the cast between them is this call. Arguments as dg_fp8_grouped_masked_swiglu,
   except the output: for each valid row m < masked_m[g] and each 1x128 group j of H's I columns,
   with amax the largest |H| over that row's 128 values of H = silu(gate)·up (the FP32 values
   dg_fp8_grouped_masked_swiglu_f32 produces), Hq[g][m][128j + c] = e4m3_rne(clamp(H · (448/amax),
   ±448)) (the factor 448/amax an IEEE FP32 division, the product rounded to nearest even in FP32,
   then to the nearest E4M3 value, ties to even) and sH[g][j][m] = amax/448 (IEEE FP32 division),
   the scale that dequantises the codes; an all-zero group has codes 0 and sH = 1. Hq is [G][M_max][I] bytes, sH is [G][I/128][align4(M_max)] FP32: exactly the A and sA
   layouts dg_fp8_grouped_masked takes, so the down projection consumes them as they are. Rows
   past masked_m are untouched in both. Hq must be 16-byte aligned, sH 4-byte aligned. */
dg_status dg_fp8_grouped_masked_swiglu_fp8(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                           const int32_t* masked_m, uint8_t* Hq, float* sH, int G, int M_max, int N,
                                           int K, dg_stream_t stream);
/* The fused SwiGLU with power-of-two scales packed as UE8M0, on the block-scaled kernel: the layouts
   of A, B, masked_m and H as for dg_fp8_grouped_masked_swiglu, the packed scale layouts of
   dg_fp8_grouped_masked_ue8m0 (sA [G][ceil(ceil(K/128)/4)][align4(M_max)], sB [G][N/128][ceil(ceil(K/128)/4)],
   N = 2I). The accumulator of a tile stays in tensor memory for the whole K loop, so each epilogue
   warp reads both its gate and its up columns from it; silu as in the FP32-scale form. */
dg_status dg_fp8_grouped_masked_swiglu_ue8m0(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                             const int32_t* sB, const int32_t* masked_m, uint16_t* H, int G,
                                             int M_max, int N, int K, dg_stream_t stream);
dg_status dg_fp8_grouped_masked_swiglu_ue8m0_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                                 const int32_t* sB, const int32_t* masked_m, float* H, int G,
                                                 int M_max, int N, int K, dg_stream_t stream);

/*
 * Accumulating dense GEMM: D = C + A·Bᵀ, the full definition of fp8_gemm_nt ("DeepGEMM: İnce
 * ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri", tr.news.hada.io/topic?id=19459,
 * § "GEMM arayüzü ve yerleşim kısıtları": the kernels are named after D = C + A @ B, and
 * fp8_gemm_nt computes D = C + A @ B.T). C and D are FP32 [M,N] row-major. C may be D itself (in-place
 * accumulation, e.g. of weight gradients); otherwise C is copied into D on `stream` first, and C and D
 * must not overlap. Each element of D receives the product exactly once (a TMA reduce-add onto D),
 * so D = fl32(C + fl32(A·Bᵀ)) and the result is deterministic. The other arguments, layouts and
 * errors are those of dg_fp8_gemm_nt_f32 (or dg_fp8_gemm_nt_ue8m0_f32 for packed UE8M0 scales).
 */
dg_status dg_fp8_gemm_nt_acc_f32(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                 const float* C, float* D, int M, int N, int K, dg_stream_t stream);
dg_status dg_fp8_gemm_nt_ue8m0_acc_f32(const uint8_t* A, const int32_t* sA, const uint8_t* B,
                                       const int32_t* sB, const float* C, float* D, int M, int N, int K,
                                       dg_stream_t stream);

/*
 * Allocation-free dense GEMM: the same computation, arguments and result as dg_fp8_gemm_nt (the
 * same validation, kernel, tile configuration, schedule and accumulation order: both entry points
 * run one code path, which differs only in where split-K scratch comes from), for callers that
 * cannot let a library call cudaMalloc — for example a framework whose caching allocator already
 * owns the device memory, or a serving loop that must not block on the device synchronisation
 * cudaMalloc/cudaFree may do.
 * The DeepGEMM pages have no counterpart to this call; it is an addition of this library.
 *   - It allocates nothing. The split-K partials and arrival counters it may need live in one fixed
 *     array inside libdg (20 MiB of FP32 partials + 4096 counters, about 20.02 MiB), which every
 *     device that loads the library holds until the process exits.
 *   - The first call on each device looks up that array's device address (cudaGetSymbolAddress,
 *     with the device current) and caches it; make that first call before any stream capture.
 *   - A shape whose split-K scratch would exceed the array returns DG_ERR_UNSUPPORTED with a message
 *     naming the sizes (dg_fp8_gemm_nt has no such limit). Shapes that need no split-K use no scratch,
 *     nor do shapes whose split-K runs inside thread-block clusters (dg_set_cluster_split); a tail
 *     split (dg_set_tail_splits) needs at most one wave of partials, which the array holds.
 *   - Every call on a device shares the array and the array keeps the last call's contents; the call
 *     clears the counters it uses (an asynchronous memset on `stream`) before its kernel. Calls that
 *     overlap on the GPU (e.g. on two streams of one device) race on the array and give wrong results.
 */
dg_status dg_fp8_gemm_nt_noalloc(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                 uint16_t* D, int M, int N, int K, dg_stream_t stream);

/* x rounded up so that x * elem_bytes is a multiple of 16 bytes (the TMA alignment).
   Source: get_tma_aligned_size, tr.news.hada.io/topic?id=19459, § "Yardımcı fonksiyonlar ve
   ortam değişkenleri". Returns -1 for x < 0 or elem_bytes not in {1, 2, 4, 8, 16}. */
int dg_get_tma_aligned_size(int x, int elem_bytes);

/* Row alignment of each group's segment in the contiguous layout (128, the M block).
   Source: get_mk_alignment_for_contiguous_layout, same page and section. */
int dg_get_mk_alignment_for_contiguous_layout(void);

/* Cap on the SMs the kernels use (0 restores the device's SM count; the environment variable
   DG_NUM_SMS sets the initial cap). Source: set_num_sms / get_num_sms, same page and section.
   dg_get_num_sms() returns the cap in force for the current device. */
void dg_set_num_sms(int n);
int dg_get_num_sms(void);

/* Time limit, in microseconds, of every pipeline wait inside the kernels (a wait on a copy, an MMA or
   a hand-over between warps). No wait of a working launch comes near the default of 2 s. A wait that
   exceeds the limit sets DG_DEV_TIMEOUT in the device status word; the kernel then stops issuing work,
   waits (with a fixed 2 s bound) for its copies and MMAs already in flight, frees its tensor memory and
   returns, leaving the output undefined where it gave up; dg_get_device_status reports the bit and
   clears the split-K counters, and the next call works normally. The limit applies to launches made
   after the call. us < 0 restores the default; values above 16777215 (about 16.8 s) are clamped;
   0 makes every wait that is not already satisfied give up at once (a way to exercise the recovery
   path without a fault). The environment variable DG_WAIT_LIMIT_US sets the initial value. Returns
   the previous value. The pages have no counterpart: this is part of this library's failure
   detection. */
long long dg_set_wait_limit_us(long long us);

/* Tail split of the dense, contiguous and masked forms (dg_fp8_gemm_nt_noalloc and the fused
   SwiGLU included), with either scale form (not the K-grouped form; calls whose configuration
   already splits K are unaffected). The fused SwiGLU reduces the gate and up partials before it
   forms H. When the output tiles of a launch
   leave a last, partial wave of at most half the grid, the kernel may cut each of those tiles into
   up to n K ranges, computed by otherwise idle SMs and summed in range order (deterministic) by the
   last range to finish, exactly as split-K does. The kernel takes the split only when its cost model
   says the K-blocks saved outweigh the exchange. n = 1 switches the tail split off; n <= 0 restores
   the default (4); values above 16 are clamped. The environment variable DG_TAIL_SPLITS sets the
   initial value. Returns the previous value. This is a scheduling choice: results stay within the
   accuracy bar either way, but the tail tiles' FP32 rounding differs between the two settings.
   Source: it extends the unified (persistent) block scheduler of the feature list on
   biggo.id/news/202502260712_DeepGEMM_FFMA_Optimization, § "Fitur Utama dan Persyaratan DeepGEMM".
   The pages do not describe splitting K; the tail rule is this implementation's choice for GB300's
   152 SMs. */
int dg_set_tail_splits(int n);

/* Pairs of CTAs sharing B tiles (dense and contiguous calls with FP32 scales and K-major operands,
   BN = 256, no split-K, at least 256 rows). The CTAs run as clusters of two over pairs of 128-row
   blocks that use the same B tile: each CTA loads its own A tile and half of the B tile, which TMA
   multicasts into both CTAs' shared memory, so each SM pulls a third less operand data from L2 per
   K-block. A contiguous pair whose two blocks belong to different groups loads each group's B tile
   separately. Results are bit-identical with pairing on or off; only the schedule changes, and a
   paired launch has no tail split. dg_query_config reports a paired configuration as block_m 256.
   Pairing is off by default: on = 1 switches it on, on = 0 off; the environment variable
   DG_PAIR_B=1 sets it on initially. Returns the previous setting. Measured on GB300, pairing does
   not shorten the kernel's period per K-block: that is set by the hand-off MMA -> promotion -> MMA
   through the tensor memory, and each SM still receives the whole B tile. Pairing also loses the
   tail split (4096x7168x16384: 397 us single, 419 us paired; under a sustained load the paired
   launch draws less power and runs about 4% higher in clock, but needs about 8% more cycles).
   The pages say only that the design moves its operands with TMA ("DeepSeek AI libera DeepGEMM…",
   7minutos.es, § "Detalles y beneficios técnicos"); sharing them through multicast is this
   implementation's choice. */
int dg_set_pair_b(int on);

/* Scale factors into the packed UE8M0 layout of the block-scaled (_ue8m0) calls, on the GPU: the
   counterpart of the library's helper that brings scaling factors into the layout its SM100 kernels
   require ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
   tr.news.hada.io/topic?id=19459, § "Yardımcı fonksiyonlar ve ortam değişkenleri" and § "GEMM
   arayüzü ve yerleşim kısıtları": four UE8M0 codes per int32).
     _a: sA [G][ceil(K/128)][align4(M)] FP32 (A's MN-major layout; G = 1 for the dense and contiguous
         calls, M = M_max for the masked ones) -> sA_packed [G][ceil(ceil(K/128)/4)][align4(M)] int32.
     _b: sB [G][ceil(N/128)][ceil(K/128)] FP32 -> sB_packed [G][ceil(N/128)][ceil(ceil(K/128)/4)] int32.
   Byte j of each word is the code of K-block 4q + j (bytes past the last K-block: 127). A scale
   2^e with e in [-127, 127] becomes the code e + 127, so the packed call computes exactly what the
   FP32-scale call computes with these scales. A zero scale (the padding rows m >= M of A's layout)
   packs as 127. Any other value sets DG_DEV_BAD_SCALE in the device status word and packs as the
   smallest power of two at or above its magnitude (clamped to [2^-127, 2^127]; NaN as 1): the
   block-scaled MMA cannot apply it exactly. Device pointers, 4-byte aligned, launched on `stream`;
   the output must not overlap the input. */
dg_status dg_transform_sf_into_ue8m0_a(const float* sA, int32_t* sA_packed, int G, int M, int K, dg_stream_t stream);
/* A's FP32 scales from the row-major layout a per-token quantiser writes, sA_rows [G][M][ceil(K/128)]
   (row m's scales contiguous), into the MN-major layout every call takes, sA [G][ceil(K/128)][align4(M)],
   rows m >= M set to 0: the other conversion of the library's transform_sf_into_required_layout (same
   section as above). Device pointers, 4-byte aligned, launched on `stream`; no overlap. */
dg_status dg_transform_sf_a_into_mn_major(const float* sA_rows, float* sA, int G, int M, int K, dg_stream_t stream);
dg_status dg_transform_sf_into_ue8m0_b(const float* sB, int32_t* sB_packed, int G, int N, int K, dg_stream_t stream);

/* Programmatic dependent launch for every GEMM call. With on != 0, each kernel is launched with
   programmatic stream serialization: it may start while the kernel ahead of it in the stream is
   still running, set up its shared memory, barriers and tensor memory, and then wait
   (griddepcontrol.wait) until that kernel has completed and its writes are visible, before it
   reads any input. Each kernel also signals, once its own setup is done, that the next kernel may
   start (griddepcontrol.launch_dependents). Back-to-back calls on one stream then hide part of
   each launch's setup. A kernel that follows one of these in the stream starts early only if it
   was itself launched for it. Results are the same bits either way. on = 0 (the default; the
   environment variable DG_PDL=1 sets the initial value to on) launches in plain stream order.
   Returns the previous value (0 or 1). The pages name a PDL switch among the library's utilities,
   set_pdl / get_pdl ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
   tr.news.hada.io/topic?id=19459, § "Yardımcı fonksiyonlar ve ortam değişkenleri"). */
int dg_set_pdl(int on);
/* The current setting of dg_set_pdl (0 or 1). */
int dg_get_pdl(void);

/* Split-K inside thread-block clusters (dense and contiguous forms, either scale form). When a call
   splits K (few output tiles) into at most 8 ranges and every tile's ranges fit on the GPU at once
   as one cluster of CTAs, the ranges reduce through distributed shared memory: partials in each
   CTA's shared memory, cluster barriers, sums in range order. Otherwise they go through a global
   workspace with an arrival counter per tile. Both orders are the same, so the results are bitwise
   equal. on = 0 forces the global workspace; on != 0 (the default) allows clusters. The environment
   variable DG_CLUSTER_SPLIT=0 sets the initial value to off. Returns the previous value (0 or 1).
   This is an addition of this implementation; the pages do not describe split-K. */
int dg_set_cluster_split(int on);

/* Reads and clears the device status word of the current device after synchronising `stream`.
   *code receives the DG_DEV_* bits. Returns DG_ERR_DEVICE_STATUS when a bit was set. */
dg_status dg_get_device_status(int* code, dg_stream_t stream);

/* Message describing the last error returned by a call on this thread ("" if none). */
const char* dg_last_error_string(void);

/* The tile configuration a GEMM call with these arguments would launch, for logging and tests.
   mode: 0 dense, 1 contiguous, 2 masked; out_f32: 0 or 1. Writes 6 ints to cfg:
   {block_m, block_n, stages, splits, grid, num_tiles_upper_bound}. Setting the environment
   variable DG_PRINT_CONFIGS=1 prints the same per call on stderr. */
dg_status dg_query_config(int mode, int M, int N, int K, int G, int out_f32, int* cfg);
/* The same for the packed-UE8M0 calls. */
dg_status dg_query_config_ue8m0(int mode, int M, int N, int K, int G, int out_f32, int* cfg);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
