/*
 * dg_inputs.c — seeded synthetic operands for the FP8 (E4M3) fine-grained-scaled GEMM.
 *
 * This module is input preparation only. It draws values, quantises them to E4M3 bytes plus
 * FP32 scales, and hands the SAME bytes and scales to both the CUDA path and the CPU oracle.
 * It holds none of the GEMM's arithmetic (no E4M3 decode, no products, no accumulation, no
 * BF16 rounding), so it cannot make the two sides agree by sharing a mistake.
 *
 * Random numbers: a counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014). Value i of a (seed, stream, sub) triple is
 * mix(key + (i+1)*gamma), so every value is independent of the thread that computes it and of
 * the order in which values are drawn. Normals come from Box-Muller, Student-t(nu=3) from
 * z0 / sqrt((z1^2+z2^2+z3^2)/3) with four independent normal streams.
 *
 * Quantiser: the DeepSeek-V3 fine-grained scheme the DeepGEMM pages name ("DeepGEMM: clean
 * and efficient FP8 GEMM kernels with fine-grained scaling", first section): one FP32 scale per
 * 1x128 K-group of each A row and one per 128x128 block of B, s = amax/448 (448 is the largest
 * finite E4M3 value), q = E4M3(x/s) rounded to nearest-even with saturation. amax == 0 gives
 * s = 1. Partial groups and blocks at the M/N/K tails take amax over the elements present.
 * For the packed-UE8M0 input form (the DeepGEMM SM100 kernels take UE8M0 scales) the scale is
 * instead the smallest power of two >= amax/448, so that it is exactly an E8M0 value.
 *
 * A scales are written MN-major ("the LHS scaling factor must be TMA-aligned and transposed",
 * DeepGEMM README summary, section "GEMM arayuzu ve yerlesim kisitlari"): sA[kb][m] with a row
 * stride ldsa = M rounded up to a multiple of 4 (16 bytes). B scales are row-major
 * sB[g][nb][kb].
 *
 * Built with -ffp-contract=off so that x86-64 and aarch64 hosts produce identical bytes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DGI_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t dgi_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of the (seed, stream, sub) sequence. */
uint64_t dgi_key(uint64_t seed, uint64_t stream, uint64_t sub) {
  uint64_t k = dgi_mix(seed * DGI_GAMMA + 1ULL);
  k = dgi_mix(k ^ (stream * DGI_GAMMA + 2ULL));
  k = dgi_mix(k ^ (sub * DGI_GAMMA + 3ULL));
  return k;
}

/* i-th 64-bit output of SplitMix64 started from state `key`. */
static inline uint64_t dgi_bits(uint64_t key, uint64_t i) { return dgi_mix(key + (i + 1ULL) * DGI_GAMMA); }

/* Uniform in the open interval (0, 1). */
static inline double dgi_uniform(uint64_t key, uint64_t i) {
  return ((double)(dgi_bits(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of the sequence (Box-Muller on the pair i/2). */
static inline double dgi_normal(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = dgi_uniform(key, 2 * j), u2 = dgi_uniform(key, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* dist: 0 = N(0,1), 1 = Student-t with 3 degrees of freedom. */
static inline float dgi_draw(const uint64_t keys[4], int dist, uint64_t i) {
  double z0 = dgi_normal(keys[0], i);
  if (dist == 0) return (float)z0;
  double z1 = dgi_normal(keys[1], i), z2 = dgi_normal(keys[2], i), z3 = dgi_normal(keys[3], i);
  return (float)(z0 / sqrt((z1 * z1 + z2 * z2 + z3 * z3) / 3.0));
}

/* E4M3 (OCP FP8, 1-4-3, bias 7, no infinities, 0x7F/0xFF NaN) nearest-even encode with
   saturation to +-448. Input preparation only. */
uint8_t dgi_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < 0.015625) { /* below 2^-6: subnormal quantum 2^-9; q == 8 is the smallest normal 0x08 */
    double q = nearbyint(a * 512.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  frexp(a, &e2);
  int E = e2 - 1; /* a in [2^E, 2^(E+1)), E in [-6, 8] */
  double q = nearbyint((ldexp(a, -E) - 1.0) * 8.0);
  int be = E + 7, m = (int)q;
  if (m == 8) { m = 0; be += 1; }
  int code = (be << 3) | m;
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

void dgi_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = dgi_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* Parallel-for over [0, n) in contiguous chunks.                                             */

typedef void (*dgi_body)(void* ctx, int64_t lo, int64_t hi);
typedef struct { dgi_body f; void* ctx; int64_t lo, hi; } dgi_task;

static void* dgi_run(void* p) {
  dgi_task* t = (dgi_task*)p;
  if (t->hi > t->lo) t->f(t->ctx, t->lo, t->hi);
  return NULL;
}

static void dgi_parallel(dgi_body f, void* ctx, int64_t n, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < threads) threads = (int)(n > 0 ? n : 1);
  pthread_t tid[256];
  dgi_task task[256];
  int64_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    task[t].f = f; task[t].ctx = ctx;
    task[t].lo = (int64_t)t * chunk;
    task[t].hi = task[t].lo + chunk < n ? task[t].lo + chunk : n;
    if (t == 0) continue;
    if (pthread_create(&tid[t], NULL, dgi_run, &task[t]) != 0) { dgi_run(&task[t]); tid[t] = 0; }
  }
  dgi_run(&task[0]);
  for (int t = 1; t < threads; ++t) if (tid[t]) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------------------------ */
/* Raw values.                                                                                */

typedef struct { uint64_t keys[4]; int dist; float* out; int64_t base; } dgi_fill_ctx;

static void dgi_fill_body(void* p, int64_t lo, int64_t hi) {
  dgi_fill_ctx* c = (dgi_fill_ctx*)p;
  for (int64_t i = lo; i < hi; ++i) c->out[i] = dgi_draw(c->keys, c->dist, (uint64_t)(c->base + i));
}

/* Values [base, base+n) of the (seed, stream) sequence as float32. */
void dgi_fill(uint64_t seed, uint64_t stream, int dist, int64_t base, int64_t n, float* out, int threads) {
  dgi_fill_ctx c;
  for (int s = 0; s < 4; ++s) c.keys[s] = dgi_key(seed, stream, (uint64_t)s);
  c.dist = dist; c.out = out; c.base = base;
  dgi_parallel(dgi_fill_body, &c, n, threads);
}

/* round(frac*K) distinct K-channels from a seeded Fisher-Yates shuffle of 0..K-1 (stream 2). */
int dgi_outlier_channels(uint64_t seed, int K, double frac, int32_t* out) {
  int n_out = (int)floor(frac * (double)K + 0.5);
  if (n_out <= 0 || K <= 0) return 0;
  if (n_out > K) n_out = K;
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  if (!perm) return -1;
  for (int i = 0; i < K; ++i) perm[i] = i;
  uint64_t key = dgi_key(seed, 2, 0);
  for (int i = K - 1; i >= 1; --i) {
    int j = (int)floor(dgi_uniform(key, (uint64_t)i) * (double)(i + 1));
    if (j > i) j = i;
    int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
  }
  memcpy(out, perm, sizeof(int32_t) * (size_t)n_out);
  free(perm);
  return n_out;
}

/* ------------------------------------------------------------------------------------------ */
/* Scale of a group with absolute maximum amax. scale_fmt 0: s = amax/448 (FP32, the DeepSeek-V3
   rule). scale_fmt 1: the smallest power of two >= amax/448, kept in [2^-127, 2^127] so that it
   is a UE8M0 (OCP MX E8M0) value; the block then never saturates. amax == 0 gives s = 1.      */
static float dgi_scale(float amax, int scale_fmt) {
  if (!(amax > 0.0f)) return 1.0f;
  float t = amax / 448.0f;
  if (scale_fmt == 0) return t;
  int e;
  float f = frexpf(t, &e);            /* t = f * 2^e, f in [0.5, 1) */
  int p = (f == 0.5f) ? e - 1 : e;    /* 2^p is the smallest power of two >= t */
  if (p < -127) p = -127;
  if (p > 127) p = 127;
  return ldexpf(1.0f, p);
}

/* ------------------------------------------------------------------------------------------ */
/* A: rows of x drawn (or given), quantised per 1x128 K-group, scales MN-major.               */

typedef struct {
  uint64_t keys[4]; int dist; int64_t base_row;      /* draw mode */
  const float* x;                                    /* given mode (row-major [M,K]) */
  const uint8_t* is_outlier; float outlier_scale;
  int M, K, nkb; int64_t ldsa; int scale_fmt;
  uint8_t* A; float* sA;
} dgi_qa_ctx;

static void dgi_qa_body(void* p, int64_t lo, int64_t hi) {
  dgi_qa_ctx* c = (dgi_qa_ctx*)p;
  float* row = (float*)malloc(sizeof(float) * (size_t)c->K);
  if (!row) return;
  for (int64_t m = lo; m < hi; ++m) {
    if (c->x) {
      memcpy(row, c->x + m * (int64_t)c->K, sizeof(float) * (size_t)c->K);
    } else {
      int64_t off = (c->base_row + m) * (int64_t)c->K;
      for (int k = 0; k < c->K; ++k) row[k] = dgi_draw(c->keys, c->dist, (uint64_t)(off + k));
    }
    if (c->is_outlier)
      for (int k = 0; k < c->K; ++k) if (c->is_outlier[k]) row[k] *= c->outlier_scale;
    for (int kb = 0; kb < c->nkb; ++kb) {
      int k0 = kb * 128, k1 = k0 + 128 < c->K ? k0 + 128 : c->K;
      float amax = 0.0f;
      for (int k = k0; k < k1; ++k) { float v = fabsf(row[k]); if (v > amax) amax = v; }
      float s = dgi_scale(amax, c->scale_fmt);
      c->sA[(int64_t)kb * c->ldsa + m] = s;
      for (int k = k0; k < k1; ++k) c->A[m * (int64_t)c->K + k] = dgi_e4m3_encode(row[k] / s);
    }
  }
  free(row);
}

/* Draws A[M,K] as rows [base_row, base_row+M) of the (seed, stream) sequence (row-major element
   counter), applies the optional channel outliers, and quantises. sA must hold nkb*ldsa floats
   and is fully written (padding columns m >= M are set to 0). */
void dgi_make_a(uint64_t seed, uint64_t stream, int dist, int64_t base_row, int M, int K,
                const int32_t* outlier_ch, int n_outlier, float outlier_scale,
                uint8_t* A, float* sA, int64_t ldsa, int scale_fmt, int threads) {
  dgi_qa_ctx c;
  memset(&c, 0, sizeof(c));
  for (int s = 0; s < 4; ++s) c.keys[s] = dgi_key(seed, stream, (uint64_t)s);
  c.dist = dist; c.base_row = base_row; c.M = M; c.K = K; c.nkb = (K + 127) / 128; c.ldsa = ldsa;
  c.scale_fmt = scale_fmt;
  c.A = A; c.sA = sA; c.outlier_scale = outlier_scale;
  uint8_t* flag = NULL;
  if (n_outlier > 0) {
    flag = (uint8_t*)calloc((size_t)K, 1);
    for (int i = 0; i < n_outlier; ++i) flag[outlier_ch[i]] = 1;
    c.is_outlier = flag;
  }
  for (int kb = 0; kb < c.nkb; ++kb)
    for (int64_t m = M; m < ldsa; ++m) sA[(int64_t)kb * ldsa + m] = 0.0f;
  dgi_parallel(dgi_qa_body, &c, M, threads);
  free(flag);
}

/* Quantises a given row-major float32 x[M,K] the same way. */
void dgi_quantize_a(const float* x, int M, int K, uint8_t* A, float* sA, int64_t ldsa, int scale_fmt,
                    int threads) {
  dgi_qa_ctx c;
  memset(&c, 0, sizeof(c));
  c.x = x; c.M = M; c.K = K; c.nkb = (K + 127) / 128; c.ldsa = ldsa; c.A = A; c.sA = sA;
  c.scale_fmt = scale_fmt;
  for (int kb = 0; kb < c.nkb; ++kb)
    for (int64_t m = M; m < ldsa; ++m) sA[(int64_t)kb * ldsa + m] = 0.0f;
  dgi_parallel(dgi_qa_body, &c, M, threads);
}

/* ------------------------------------------------------------------------------------------ */
/* B: [G,N,K] drawn (or given), quantised per 128x128 block, scales sB[g][nb][kb].            */

typedef struct {
  uint64_t keys[4]; int dist;
  const float* x;
  int G, N, K, nnb, nkb, scale_fmt;
  uint8_t* B; float* sB;
} dgi_qb_ctx;

static void dgi_qb_body(void* p, int64_t lo, int64_t hi) {
  dgi_qb_ctx* c = (dgi_qb_ctx*)p;
  float* strip = (float*)malloc(sizeof(float) * 128 * (size_t)c->K);
  if (!strip) return;
  for (int64_t t = lo; t < hi; ++t) { /* t = g*nnb + nb */
    int64_t g = t / c->nnb, nb = t % c->nnb;
    int n0 = (int)nb * 128, n1 = n0 + 128 < c->N ? n0 + 128 : c->N, rows = n1 - n0;
    int64_t row0 = g * (int64_t)c->N + n0;
    for (int r = 0; r < rows; ++r) {
      if (c->x) {
        memcpy(strip + (int64_t)r * c->K, c->x + (row0 + r) * (int64_t)c->K, sizeof(float) * (size_t)c->K);
      } else {
        int64_t off = (row0 + r) * (int64_t)c->K;
        for (int k = 0; k < c->K; ++k) strip[(int64_t)r * c->K + k] = dgi_draw(c->keys, c->dist, (uint64_t)(off + k));
      }
    }
    for (int kb = 0; kb < c->nkb; ++kb) {
      int k0 = kb * 128, k1 = k0 + 128 < c->K ? k0 + 128 : c->K;
      float amax = 0.0f;
      for (int r = 0; r < rows; ++r)
        for (int k = k0; k < k1; ++k) { float v = fabsf(strip[(int64_t)r * c->K + k]); if (v > amax) amax = v; }
      float s = dgi_scale(amax, c->scale_fmt);
      c->sB[(g * c->nnb + nb) * c->nkb + kb] = s;
      for (int r = 0; r < rows; ++r)
        for (int k = k0; k < k1; ++k)
          c->B[(row0 + r) * (int64_t)c->K + k] = dgi_e4m3_encode(strip[(int64_t)r * c->K + k] / s);
    }
  }
  free(strip);
}

/* Draws B[G,N,K] (row-major element counter over the whole tensor) and quantises it. */
void dgi_make_b(uint64_t seed, uint64_t stream, int dist, int G, int N, int K,
                uint8_t* B, float* sB, int scale_fmt, int threads) {
  dgi_qb_ctx c;
  memset(&c, 0, sizeof(c));
  for (int s = 0; s < 4; ++s) c.keys[s] = dgi_key(seed, stream, (uint64_t)s);
  c.dist = dist; c.G = G; c.N = N; c.K = K; c.nnb = (N + 127) / 128; c.nkb = (K + 127) / 128;
  c.scale_fmt = scale_fmt;
  c.B = B; c.sB = sB;
  dgi_parallel(dgi_qb_body, &c, (int64_t)G * c.nnb, threads);
}

/* Quantises a given row-major float32 x[G,N,K] the same way. */
void dgi_quantize_b(const float* x, int G, int N, int K, uint8_t* B, float* sB, int scale_fmt,
                    int threads) {
  dgi_qb_ctx c;
  memset(&c, 0, sizeof(c));
  c.x = x; c.G = G; c.N = N; c.K = K; c.nnb = (N + 127) / 128; c.nkb = (K + 127) / 128;
  c.scale_fmt = scale_fmt;
  c.B = B; c.sB = sB;
  dgi_parallel(dgi_qb_body, &c, (int64_t)G * c.nnb, threads);
}

/* masked_m[g] uniform in [0, M_max] (stream 3); then masked_m[0] = 0 and masked_m[G-1] = M_max
   so that both the empty and the full group are always present. */
void dgi_make_masked_m(uint64_t seed, int G, int M_max, int force_ends, int32_t* out) {
  uint64_t key = dgi_key(seed, 3, 0);
  for (int g = 0; g < G; ++g) {
    int v = (int)floor(dgi_uniform(key, (uint64_t)g) * (double)(M_max + 1));
    if (v > M_max) v = M_max;
    out[g] = v;
  }
  if (force_ends && G >= 1) { out[0] = 0; out[G - 1] = M_max; }
}
