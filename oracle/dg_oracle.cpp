// dg_oracle.cpp — plain, slow, obviously correct CPU oracle of the FP8 (E4M3) fine-grained-scaled
// GEMM D = A·Bᵀ and its two MoE grouped forms.
//
// TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the benchmark's CPU
// baseline may load this library. It shares no code, header, table or helper with the CUDA path,
// and the CUDA path never calls it.
//
// What it computes, and where that is defined:
//   * "FP8 GEMM with the fine-grained scaling proposed in DeepSeek-V3" and the NT convention
//     fp8_gemm_nt: D = C + A @ B.T with A row-major and B col-major, i.e. B stored [N,K] with K
//     contiguous ("DeepGEMM: İnce ölçeklendirmeyle temiz ve verimli FP8 GEMM çekirdekleri",
//     tr.news.hada.io/topic?id=19459, § "GEMM arayüzü ve yerleşim kısıtları"). C is absent here:
//     D is overwritten.
//   * Scale granularity: one FP32 scale per 1x128 K-group of each A row and one per 128x128 block
//     of B (DeepSeek-V3 Technical Report, § 3.3.2 "Fine-Grained Quantization"). A's scales are
//     MN-major, "TMA-aligned and transposed" (same page and section): sA[kb * ldsa + m].
//     B's scales are row-major sB[nb * nkb + kb] per group.
//   * Two-level accumulation ("promotion"): the FP8 tensor-core partial of each 128-deep K-slice
//     is scaled and added into a higher-precision accumulator on CUDA cores ("DeepGEMM" first
//     release summary, tr.news.hada.io/topic?id=19444, feature list; "DeepSeek AI libera
//     DeepGEMM", 7minutos.es, § "Detalles y beneficios técnicos"). The oracle follows the same two
//     levels in FP64: P_kb = Σ_{k in kb} a·b exactly, then acc += (sA·sB)·P_kb.
//   * Contiguous layout: grouped along M only, N and K shared, experts' token rows concatenated,
//     each segment aligned to the M block (tr.news.hada.io/topic?id=19459, § "Dense ve Grouped
//     GEMM"). Row m uses group m_indices[m]; -1 marks a padding row, which is left untouched.
//   * Masked layout: the kernel computes only the valid region given by a mask tensor, read on
//     the device because the CPU does not know the per-expert token count under CUDA graphs (same
//     page and section; tr.news.hada.io/topic?id=19444, § "MoE modelleri için gruplanmış GEMM
//     performansı"). Rows m < masked_m[g] of group g are written; the other rows are untouched.
//   * E4M3: the OCP 8-bit floating point format (1 sign, 4 exponent bits with bias 7, 3 mantissa
//     bits; exponent field 15 with mantissa 7 is NaN; no infinities; largest finite value 448).
//   * BF16 output rounding: IEEE round-to-nearest-even, taken directly from the FP64 value (no
//     intermediate FP32 rounding).
//   * Masked GEMM fused with SwiGLU: the pages' Mega MoE fuses linear 1, SwiGLU and linear 2 of the
//     experts into one kernel (tr.news.hada.io/topic?id=19459, § "Mega MoE"); this is its first
//     fusion, on one GPU and with FP8 weights. SwiGLU is taken from its definition (Shazeer, "GLU
//     Variants Improve Transformer", 2020): silu(gate)·up with silu(x) = x / (1 + e^-x). B holds 2I
//     rows per group, gate rows [0, I) then up rows [I, 2I) (a reading: the pages give no layout);
//     H[g,m,j] = silu(D[g,m,j]) · D[g,m,I+j] for the valid rows m < masked_m[g]; other rows untouched.
//   * K-grouped contiguous GEMM (MoE weight backward: k_grouped_fp8_gemm_tn_contiguous, grouped
//     along K with M and N fixed, same page, § "Dense ve Grouped GEMM"): the experts' token
//     segments are concatenated along K, each a multiple of 128 long; group g covers
//     k in [off[g], off[g+1]) and D[g] = Σ over that range, with the scales of those K-blocks.
//     An empty segment gives D[g] = 0.
//   * Accumulating form D = C + A @ B.T (the kernel naming D = C + A @ B and fp8_gemm_nt's
//     definition, same page and section): C is an FP32 [M,N] matrix added to the FP64 GEMM value.
//   * Packed UE8M0 scales (the Blackwell input form): the SM100 implementation takes its scaling
//     factors as UE8M0 values, four of them packed into one 32-bit integer (same page, § "GEMM
//     arayüzü ve yerleşim kısıtları"). UE8M0 is the OCP Microscaling (MX) v1.0 E8M0 format
//     (§ 5.4.1): eight exponent bits with bias 127, no sign, no mantissa, 0xFF is NaN; the value of
//     code e is 2^(e-127). Byte j (bits 8j..8j+7) of packed word q holds K-group 4q+j. Such scales
//     are powers of two, so unpacking them into FP32 is exact and the GEMM is the one above.
//
// Exactness: every product of two E4M3 values has at most 8 significant bits and lies in
// [2^-18, 448^2]; 128 of them sum exactly in FP64 (53 bits). (sA·sB) of two FP32 values is exact
// in FP64; only the product with P_kb and the running sum round, once each, in FP64.
//
// Compiled with -ffp-contract=off so that no multiply-add is fused on any host.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// OCP E4M3 decode, written from the format definition.
double e4m3_value(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 15 && m == 7) return std::nan("");
  double mag;
  if (e == 0) {
    mag = std::ldexp((double)m, -9);                 // subnormal: m/8 · 2^(1-7)
  } else {
    mag = std::ldexp(1.0 + (double)m / 8.0, e - 7);  // normal: (1 + m/8) · 2^(e-7)
  }
  return s ? -mag : mag;
}

// IEEE binary32 bit pattern of a float.
uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// Round an FP64 value to BF16 (8 significant bits, FP32 exponent range) with ties to even.
uint16_t bf16_rne(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0x0000;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e2;
  std::frexp(a, &e2);                 // a in [2^(e2-1), 2^e2)
  int e = e2 - 1;
  if (e < -126) e = -126;             // BF16 subnormals share the quantum of the smallest binade
  const int q_exp = e - 7;            // value of one unit in the last place
  const double q = std::nearbyint(std::ldexp(a, -q_exp));  // default rounding mode: ties to even
  const double v = std::ldexp(q, q_exp);                   // representable in BF16, or 2^128
  const float vf = (float)v;                               // exact; 2^128 becomes +inf
  return (uint16_t)(sign | (uint16_t)(f32_bits(vf) >> 16));
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// OCP MX E8M0 decode, written from the format definition.
double ue8m0_value(uint8_t code) {
  if (code == 0xFF) return std::nan("");
  return std::ldexp(1.0, (int)code - 127);
}

// One output element: Σ_kb sA[m,kb]·sB[n/128,kb]·P_kb with P_kb the exact FP64 partial.
//   a_row : the K bytes of row m of A          sA_m : pointer to sA[0][m], stride ldsa per kb
//   b_row : the K bytes of row n of B          sB_n : pointer to sB[n/128][0] (stride 1 per kb)
double element(const uint8_t* a_row, const float* sA_m, int64_t ldsa,
               const uint8_t* b_row, const float* sB_n, int K) {
  const int nkb = ceil_div(K, 128);
  double acc = 0.0;
  for (int kb = 0; kb < nkb; ++kb) {
    const int k0 = kb * 128;
    const int k1 = (k0 + 128 < K) ? k0 + 128 : K;
    double P = 0.0;
    for (int k = k0; k < k1; ++k) P += e4m3_value(a_row[k]) * e4m3_value(b_row[k]);
    const double scale = (double)sA_m[(int64_t)kb * ldsa] * (double)sB_n[kb];
    acc += scale * P;
  }
  return acc;
}

// As element(), over the K-blocks [kb0, kb1) only (the rows are indexed from k = 0).
double element_range(const uint8_t* a_row, const float* sA_m, int64_t ldsa, const uint8_t* b_row,
                     const float* sB_n, int K, int kb0, int kb1) {
  double acc = 0.0;
  for (int kb = kb0; kb < kb1; ++kb) {
    const int k0 = kb * 128;
    const int k1 = (k0 + 128 < K) ? k0 + 128 : K;
    double P = 0.0;
    for (int k = k0; k < k1; ++k) P += e4m3_value(a_row[k]) * e4m3_value(b_row[k]);
    acc += (double)sA_m[(int64_t)kb * ldsa] * (double)sB_n[kb] * P;
  }
  return acc;
}

template <class F>
void parallel_rows(int rows, int threads, F&& body) {
  if (threads < 1) threads = 1;
  if (threads > rows) threads = rows > 0 ? rows : 1;
  std::vector<std::thread> pool;
  const int chunk = ceil_div(rows > 0 ? rows : 1, threads);
  for (int t = 0; t < threads; ++t) {
    const int lo = t * chunk, hi = (lo + chunk < rows) ? lo + chunk : rows;
    if (lo >= hi) break;
    pool.emplace_back([&body, lo, hi] { for (int r = lo; r < hi; ++r) body(r); });
  }
  for (auto& th : pool) th.join();
}

// Dense rows [0, M): D[m, n] for one group whose B and sB start at the given pointers.
void dense_rows(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B, const float* sB,
                int M, int N, int K, double* ref64, uint16_t* D, int threads) {
  const int nkb = ceil_div(K, 128);
  parallel_rows(M, threads, [&](int m) {
    for (int n = 0; n < N; ++n) {
      const double v = element(A + (int64_t)m * K, sA + m, ldsa, B + (int64_t)n * K,
                               sB + (int64_t)(n / 128) * nkb, K);
      if (ref64) ref64[(int64_t)m * N + n] = v;
      if (D) D[(int64_t)m * N + n] = bf16_rne(v);
    }
  });
}

}  // namespace

extern "C" {

double dgo_e4m3_decode(uint8_t code) { return e4m3_value(code); }

uint16_t dgo_bf16_from_f64(double x) { return bf16_rne(x); }

void dgo_bf16_from_f64_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_rne(x[i]);
}

// Dense D[M,N] = A[M,K]·B[N,K]ᵀ with sA[nkb][ldsa] (MN-major) and sB[nnb][nkb].
// ref64 (FP64, [M,N]) and D (BF16 bits, [M,N]) are each optional (nullptr skips).
void dgo_gemm_nt(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B, const float* sB,
                 int M, int N, int K, double* ref64, uint16_t* D, int threads) {
  dense_rows(A, sA, ldsa, B, sB, M, N, K, ref64, D, threads);
}

// Dense accumulating D = C + A[M,K]·B[N,K]ᵀ: ref64[m,n] = C[m,n] + (the dense value above), in
// FP64 (C, FP32, is exact in FP64).
void dgo_gemm_nt_acc(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B, const float* sB,
                     const float* C, int M, int N, int K, double* ref64, int threads) {
  const int nkb = ceil_div(K, 128);
  parallel_rows(M, threads, [&](int m) {
    for (int n = 0; n < N; ++n) {
      const double v = element(A + (int64_t)m * K, sA + m, ldsa, B + (int64_t)n * K,
                               sB + (int64_t)(n / 128) * nkb, K);
      ref64[(int64_t)m * N + n] = (double)C[(int64_t)m * N + n] + v;
    }
  });
}

// Contiguous grouped: A[M_total,K], sA[nkb][ldsa], B[G,N,K], sB[G][nnb][nkb], m_indices[M_total].
// Rows whose index is -1 are padding; rows whose index is < -1 or >= G are invalid. Both are left
// untouched in ref64/D. Returns the number of invalid rows.
int dgo_grouped_contiguous(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B,
                           const float* sB, const int32_t* m_indices, int M_total, int N, int K, int G,
                           double* ref64, uint16_t* D, int threads) {
  const int nkb = ceil_div(K, 128), nnb = ceil_div(N, 128);
  int bad = 0;
  for (int m = 0; m < M_total; ++m) if (m_indices[m] < -1 || m_indices[m] >= G) ++bad;
  parallel_rows(M_total, threads, [&](int m) {
    const int g = m_indices[m];
    if (g < 0 || g >= G) return;
    const uint8_t* Bg = B + (int64_t)g * N * K;
    const float* sBg = sB + (int64_t)g * nnb * nkb;
    for (int n = 0; n < N; ++n) {
      const double v = element(A + (int64_t)m * K, sA + m, ldsa, Bg + (int64_t)n * K,
                               sBg + (int64_t)(n / 128) * nkb, K);
      if (ref64) ref64[(int64_t)m * N + n] = v;
      if (D) D[(int64_t)m * N + n] = bf16_rne(v);
    }
  });
  return bad;
}

// Masked grouped: A[G,M_max,K], sA[G][nkb][ldsa], B[G,N,K], sB[G][nnb][nkb], masked_m[G],
// D/ref64 [G,M_max,N]. Rows m >= masked_m[g] are untouched. masked_m outside [0, M_max] is
// clamped; returns the number of clamped groups.
int dgo_grouped_masked(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B,
                       const float* sB, const int32_t* masked_m, int G, int M_max, int N, int K,
                       double* ref64, uint16_t* D, int threads) {
  const int nkb = ceil_div(K, 128), nnb = ceil_div(N, 128);
  int bad = 0;
  for (int g = 0; g < G; ++g) {
    int valid = masked_m[g];
    if (valid < 0) { valid = 0; ++bad; }
    if (valid > M_max) { valid = M_max; ++bad; }
    dense_rows(A + (int64_t)g * M_max * K, sA + (int64_t)g * nkb * ldsa, ldsa,
               B + (int64_t)g * N * K, sB + (int64_t)g * nnb * nkb, valid, N, K,
               ref64 ? ref64 + (int64_t)g * M_max * N : nullptr,
               D ? D + (int64_t)g * M_max * N : nullptr, threads);
  }
  return bad;
}

// Masked grouped GEMM fused with SwiGLU: A[G,M_max,K], sA[G][nkb][ldsa], B[G,2I,K], sB[G][2I/128][nkb],
// masked_m[G]; ref64/H [G,M_max,I]. Rows m >= masked_m[g] (clamped to [0, M_max]) are untouched.
int dgo_grouped_masked_swiglu(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B,
                              const float* sB, const int32_t* masked_m, int G, int M_max, int I, int K,
                              double* ref64, uint16_t* H, int threads) {
  const int nkb = ceil_div(K, 128), N2 = 2 * I, nnb = ceil_div(N2, 128);
  int bad = 0;
  for (int g = 0; g < G; ++g) {
    int valid = masked_m[g];
    if (valid < 0) { valid = 0; ++bad; }
    if (valid > M_max) { valid = M_max; ++bad; }
    const uint8_t* Ag = A + (int64_t)g * M_max * K;
    const float* sAg = sA + (int64_t)g * nkb * ldsa;
    const uint8_t* Bg = B + (int64_t)g * N2 * K;
    const float* sBg = sB + (int64_t)g * nnb * nkb;
    parallel_rows(valid, threads, [&](int m) {
      for (int j = 0; j < I; ++j) {
        const double gate = element(Ag + (int64_t)m * K, sAg + m, ldsa, Bg + (int64_t)j * K,
                                    sBg + (int64_t)(j / 128) * nkb, K);
        const int u = I + j;
        const double up = element(Ag + (int64_t)m * K, sAg + m, ldsa, Bg + (int64_t)u * K,
                                  sBg + (int64_t)(u / 128) * nkb, K);
        const double h = gate / (1.0 + std::exp(-gate)) * up;
        const int64_t o = ((int64_t)g * M_max + m) * I + j;
        if (ref64) ref64[o] = h;
        if (H) H[o] = bf16_rne(h);
      }
    });
  }
  return bad;
}

double dgo_silu(double x) { return x / (1.0 + std::exp(-x)); }

// K-grouped: logical A[M,K_total] and B[N,K_total] (K contiguous), sA[nkb][ldsa], sB[nnb][nkb] over the
// whole K_total, off[G+1] K offsets (multiples of 128, non-decreasing); ref64 [G,M,N]. Returns the
// number of invalid offsets (not a multiple of 128, decreasing, or beyond K_total); then computes nothing.
int dgo_k_grouped(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B, const float* sB,
                  const int32_t* off, int G, int M, int N, int K_total, double* ref64, int threads) {
  int bad = 0;
  for (int g = 0; g <= G; ++g)
    if (off[g] % 128 != 0 || off[g] < 0 || off[g] > K_total || (g > 0 && off[g] < off[g - 1])) ++bad;
  if (bad) return bad;
  const int nkb = ceil_div(K_total, 128);
  for (int g = 0; g < G; ++g) {
    const int kb0 = off[g] / 128, kb1 = off[g + 1] / 128;
    parallel_rows(M, threads, [&](int m) {
      for (int n = 0; n < N; ++n)
        ref64[((int64_t)g * M + m) * N + n] =
            element_range(A + (int64_t)m * K_total, sA + m, ldsa, B + (int64_t)n * K_total,
                          sB + (int64_t)(n / 128) * nkb, K_total, kb0, kb1);
    });
  }
  return 0;
}

// Selected elements (ms[i], ns[i]) of a dense problem, in FP64. For a grouped problem the caller
// passes the group's A/sA/B/sB base pointers.
void dgo_gemm_nt_sampled(const uint8_t* A, const float* sA, int64_t ldsa, const uint8_t* B,
                         const float* sB, int M, int N, int K, int64_t count, const int64_t* ms,
                         const int64_t* ns, double* out, int threads) {
  (void)M; (void)N;
  const int nkb = ceil_div(K, 128);
  const int rows = (int)count;
  parallel_rows(rows, threads, [&](int i) {
    const int64_t m = ms[i], n = ns[i];
    out[i] = element(A + m * K, sA + m, ldsa, B + n * K, sB + (n / 128) * nkb, K);
  });
}

double dgo_ue8m0_decode(uint8_t code) { return ue8m0_value(code); }

// Unpacks UE8M0 scales, four per 32-bit word, into FP32 (exact: every value is a power of two in
// [2^-127, 2^127], or NaN). Item i's scale of K-group kb is byte (kb % 4) of
// packed[(kb / 4) * stride_quad + i * stride_item]; it is written to out[i * out_item + kb * out_kb].
//   A's MN-major scales [ceil(nkb/4)][ldsa]:  stride_item = 1,    stride_quad = ldsa
//   B's scales [nnb][ceil(nkb/4)] per group:  stride_item = nkq,  stride_quad = 1
void dgo_ue8m0_unpack(const int32_t* packed, int64_t n_items, int nkb, int64_t stride_item,
                      int64_t stride_quad, float* out, int64_t out_item, int64_t out_kb) {
  for (int64_t i = 0; i < n_items; ++i) {
    for (int kb = 0; kb < nkb; ++kb) {
      const uint32_t word = (uint32_t)packed[(int64_t)(kb / 4) * stride_quad + i * stride_item];
      const uint8_t code = (uint8_t)((word >> (8 * (kb % 4))) & 0xFFu);
      out[i * out_item + (int64_t)kb * out_kb] = (float)ue8m0_value(code);
    }
  }
}

// Number of hardware threads of this host (the oracle's default parallelism).
int dgo_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

}  // extern "C"
