/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the W4A16 + paged
 * GQA single-token decode path.  TEST INFRASTRUCTURE ONLY: nothing in the
 * product library links, includes or calls this file.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it.
 *
 * It shares no code with the CUDA path: its own fp16 codec, its own int4
 * unpack, its own loops.  Arithmetic is fp64; values are rounded to fp16 only
 * at the operator boundaries listed below, once each.
 *
 * Sources (web pages on the "annotated-llm-runtime" project):
 *   [RU] aikraft.ru, "How to build your own LLM runtime from scratch",
 *        sections "Ключевые метрики производительности" and
 *        "Архитектурные решения и оптимизации" (model shape: 28 layers,
 *        hidden 3584, 28 heads with 7:1 GQA; symmetric group-wise INT4 with
 *        group 128; RMSNorm and lm_head in FP16; 16-token KV pages).
 *   [EN] explore.n1n.ai, "Building a Custom LLM Inference Runtime on H100",
 *        sections "2. The KV Cache and PagedAttention" and
 *        "Bug 1: The KV Cache Indexing 'Off-By-One'" (logical token position
 *        -> physical page mapping).
 * The pages never spell out RoPE, the SiLU-gated MLP, the q/k/v bias, the
 * residual adds, the embedding or the argmax; those follow the plain meaning
 * of a "Qwen2.5-7B-shaped" decoder and are marked "not on the pages" below.
 *
 * Readings taken where the pages are silent (each one is restated here so a
 * reader can check the code against it):
 *   - int4 storage: weight k of row n is nibble (k % 8) of word
 *     qweight[n][k / 8], lowest nibble first, stored offset-binary u = q + 8,
 *     so q = u - 8 lies in [-8, 7].  One fp16 scale per 128 consecutive k:
 *     scales[n][k / 128].  Dequantised weight = q * scale (no zero point:
 *     "symmetric").
 *   - rounding to fp16 happens at: RMSNorm output, each GEMV output (after
 *     bias and residual), q and k after RoPE, attention output, SiLU-mul
 *     output, lm_head logits (the argmax uses the unrounded fp64 logits).
 *   - RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma, eps inside the root,
 *     gamma applied before the single rounding.
 *   - RoPE: rotate-half pairs (i, i + D/2); inverse frequency
 *     theta^(-2i/D) rounded to fp32; angle = fp32 product of the position and
 *     that inverse frequency; cos/sin and the rotation in fp64.
 *   - context_lens counts tokens AFTER the current token is appended; the new
 *     token sits at position len - 1, in page block_table[b][(len-1) / 16],
 *     slot (len-1) % 16; attention covers positions [0, len).
 *   - GQA: query head h reads kv head h / (Hq / Hkv).
 *   - attention scale 1/sqrt(D); no mask besides the length.
 *   - argmax: lowest index wins ties.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (OpenMP only splits independent
 * output rows; every reduction is a sequential fp64 loop).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_PAGE_TOKENS 16
#define ORC_GROUP 128

/* ------------------------------------------------------------------------ */
/* fp16 codec, written from the IEEE 754 binary16 definition:               */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have */
/* exponent field 0 and value fraction * 2^-24.                             */
/* ------------------------------------------------------------------------ */

double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24);
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25);
  }
  return sign ? -v : v;
}

/* Round-to-nearest-even conversion of a double to binary16. */
uint16_t orc_double_to_half(double d) {
  if (isnan(d)) return 0x7e00;
  uint16_t sign = signbit(d) ? 0x8000 : 0;
  double a = fabs(d);
  /* 65504 is the largest finite half; halfway to the next binade step
   * (65520) and above rounds to infinity. */
  if (a >= 65520.0) return sign | 0x7c00;
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: integer multiple of 2^-24, ties to even */
    double q = nearbyint(ldexp(a, 24));
    return sign | (uint16_t)q; /* q == 1024 encodes the smallest normal */
  }
  int e;
  (void)frexp(a, &e);         /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;              /* a = m * 2^E, m in [1, 2) */
  double m = nearbyint(ldexp(a, 10 - E)); /* in [1024, 2048] */
  if (m == 2048.0) {
    m = 1024.0;
    E += 1;
  }
  if (E > 15) return sign | 0x7c00;
  return sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* Every binary16 value decoded once by orc_half_to_double (65536 entries,
 * filled when the library loads); h2d is a lookup into it. */
static double g_h2d[65536];
__attribute__((constructor)) static void orc_fill_h2d(void) {
  for (uint32_t h = 0; h < 65536u; ++h) g_h2d[h] = orc_half_to_double((uint16_t)h);
}
static inline double h2d(uint16_t h) { return g_h2d[h]; }
static inline uint16_t d2h(double d) { return orc_double_to_half(d); }

void orc_half_to_double_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = h2d(h[i]);
}

void orc_double_to_half_array(const double* d, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = d2h(d[i]);
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads later parallel loops use (timing on one core or on all of them). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* INT4 format ([RU] "symmetric group-wise INT4 (group 128)").              */
/* ------------------------------------------------------------------------ */

/* Signed code of nibble i (0..7) of a packed word. */
int orc_unpack_code(uint32_t word, int i) {
  int u = (int)((word >> (4 * i)) & 0xFu);
  return u - 8;
}

/* q[n][k] in [-8, 7] -> qweight[n][k/8]. */
void orc_pack_int4(const int8_t* q, int64_t N, int64_t K, uint32_t* qw) {
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t w = 0; w < K / 8; ++w) {
      uint32_t word = 0;
      for (int i = 0; i < 8; ++i) {
        int code = q[n * K + w * 8 + i];
        uint32_t u = (uint32_t)(code + 8) & 0xFu;
        word |= u << (4 * i);
      }
      qw[n * (K / 8) + w] = word;
    }
  }
}

void orc_unpack_int4(const uint32_t* qw, int64_t N, int64_t K, int8_t* q) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      q[n * K + k] = (int8_t)orc_unpack_code(qw[n * (K / 8) + k / 8], (int)(k % 8));
}

/* w[n][k] = q[n][k] * scale[n][k/128] (exact in fp64). */
void orc_dequant(const uint32_t* qw, const uint16_t* scales, int64_t N, int64_t K, double* w) {
  int64_t G = K / ORC_GROUP;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w[n * K + k] = (double)orc_unpack_code(qw[n * (K / 8) + k / 8], (int)(k % 8)) *
                     h2d(scales[n * G + k / ORC_GROUP]);
}

/* Test-only quantiser: per 128-group scale = fp16(amax / 7),
 * q = clamp(round-half-even(w / scale), -8, 7).  Not on the decode path. */
void orc_quantize(const double* w, int64_t N, int64_t K, uint32_t* qw, uint16_t* scales) {
  int64_t G = K / ORC_GROUP;
  int8_t* q = (int8_t*)malloc((size_t)(N * K));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < G; ++g) {
      double amax = 0.0;
      for (int64_t j = 0; j < ORC_GROUP; ++j) {
        double a = fabs(w[n * K + g * ORC_GROUP + j]);
        if (a > amax) amax = a;
      }
      uint16_t sh = d2h(amax / 7.0);
      double s = h2d(sh);
      scales[n * G + g] = sh;
      for (int64_t j = 0; j < ORC_GROUP; ++j) {
        double r = (s > 0.0) ? nearbyint(w[n * K + g * ORC_GROUP + j] / s) : 0.0;
        if (r < -8.0) r = -8.0;
        if (r > 7.0) r = 7.0;
        q[n * K + g * ORC_GROUP + j] = (int8_t)r;
      }
    }
  }
  orc_pack_int4(q, N, K, qw);
  free(q);
}

/* ------------------------------------------------------------------------ */
/* W4A16 GEMV ([RU] "Архитектурные решения и оптимизации"):                  */
/* y[m][n] = fp16( sum_k x[m][k] * q[n][k] * s[n][k/128]                    */
/*                 + bias[n] + residual[m][n] )                             */
/* bias and residual are optional (NULL).                                   */
/* ------------------------------------------------------------------------ */
void orc_w4a16_gemv(const uint16_t* x, int M, int K, const uint32_t* qw, const uint16_t* scales,
                    int N, const uint16_t* bias, const uint16_t* residual, uint16_t* y) {
  int G = K / ORC_GROUP;
  for (int m = 0; m < M; ++m) {
    const uint16_t* xm = x + (int64_t)m * K;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        int code = orc_unpack_code(qw[(int64_t)n * (K / 8) + k / 8], k % 8);
        double wv = (double)code * h2d(scales[(int64_t)n * G + k / ORC_GROUP]);
        acc += h2d(xm[k]) * wv;
      }
      if (bias) acc += h2d(bias[n]);
      if (residual) acc += h2d(residual[(int64_t)m * N + n]);
      y[(int64_t)m * N + n] = d2h(acc);
    }
  }
}

/* Dense fp16-weight GEMV returning fp64 results (lm_head, kept in FP16 per
 * [RU] "Архитектурные решения и оптимизации"). w is [N][K]. */
void orc_fp16_gemv(const uint16_t* x, int K, const uint16_t* w, int N, double* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += h2d(x[k]) * h2d(w[(int64_t)n * K + k]);
    out[n] = acc;
  }
}

/* Index of the largest value, lowest index on ties. */
int64_t orc_argmax(const double* v, int64_t n) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm ([RU]: RMSNorm kept in FP16).                                     */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, int M, int H, double eps, uint16_t* y) {
  for (int m = 0; m < M; ++m) {
    double ss = 0.0;
    for (int i = 0; i < H; ++i) {
      double v = h2d(x[(int64_t)m * H + i]);
      ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)H + eps);
    for (int i = 0; i < H; ++i)
      y[(int64_t)m * H + i] = d2h(h2d(x[(int64_t)m * H + i]) * r * h2d(gamma[i]));
  }
}

/* ------------------------------------------------------------------------ */
/* RoPE, rotate-half form (not on the pages; plain Qwen2 reading).           */
/* ------------------------------------------------------------------------ */

/* Inverse frequency of pair i, rounded to fp32. */
float orc_rope_inv_freq(int i, int D, double theta) {
  return (float)pow(theta, -2.0 * (double)i / (double)D);
}

/* Angle of pair i at position pos: the fp32 product pos * inv_freq. */
float orc_rope_angle(int pos, int i, int D, double theta) {
  float inv = orc_rope_inv_freq(i, D, theta);
  volatile float prod = (float)pos * inv; /* one fp32 rounding */
  return prod;
}

/* Rotate nheads heads of length D at position pos, in place, fp16 out. */
void orc_rope(uint16_t* x, int nheads, int D, int pos, double theta) {
  int half = D / 2;
  for (int h = 0; h < nheads; ++h) {
    uint16_t* v = x + (int64_t)h * D;
    for (int i = 0; i < half; ++i) {
      double a = (double)orc_rope_angle(pos, i, D, theta);
      double c = cos(a), s = sin(a);
      double x0 = h2d(v[i]), x1 = h2d(v[i + half]);
      v[i] = d2h(x0 * c - x1 * s);
      v[i + half] = d2h(x1 * c + x0 * s);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Paged KV cache ([EN] "2. The KV Cache and PagedAttention", "Bug 1";      */
/* [RU] 16-token pages, each (page, kv head) slice 16*128*2 B = 4 KiB).      */
/* Pool layout: [num_pages][Hkv][16][D] fp16.  Token t of sequence b lives  */
/* in page block_table[b*max_blocks + t/16], slot t%16.                      */
/* ------------------------------------------------------------------------ */

static inline int64_t orc_slot_offset(int32_t page, int h, int slot, int Hkv, int D) {
  return (((int64_t)page * Hkv + h) * ORC_PAGE_TOKENS + slot) * D;
}

/* Write k[b][h][:] and v[b][h][:] at position context_lens[b]-1. */
void orc_kv_append(const uint16_t* k, const uint16_t* v, uint16_t* k_pool, uint16_t* v_pool,
                   const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                   int B, int Hkv, int D) {
  for (int b = 0; b < B; ++b) {
    int pos = context_lens[b] - 1;
    int32_t page = block_table[(int64_t)b * max_blocks + pos / ORC_PAGE_TOKENS];
    int slot = pos % ORC_PAGE_TOKENS;
    for (int h = 0; h < Hkv; ++h) {
      int64_t off = orc_slot_offset(page, h, slot, Hkv, D);
      for (int d = 0; d < D; ++d) {
        k_pool[off + d] = k[((int64_t)b * Hkv + h) * D + d];
        v_pool[off + d] = v[((int64_t)b * Hkv + h) * D + d];
      }
    }
  }
}

/* Gather the first L tokens of one sequence into contiguous [L][Hkv][D]. */
void orc_gather_kv(const uint16_t* pool, const int32_t* block_table_row, int L, int Hkv, int D,
                   uint16_t* out) {
  for (int t = 0; t < L; ++t) {
    int32_t page = block_table_row[t / ORC_PAGE_TOKENS];
    int slot = t % ORC_PAGE_TOKENS;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = orc_slot_offset(page, h, slot, Hkv, D);
      memcpy(out + ((int64_t)t * Hkv + h) * D, pool + src, sizeof(uint16_t) * (size_t)D);
    }
  }
}

/* Contiguous GQA attention for one sequence (textbook softmax attention):
 * q [Hq][D], k/v [L][Hkv][D] -> out [Hq][D] (fp16), scale applied to q.k. */
void orc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int Hq, int Hkv,
                   int D, int L, double scale, uint16_t* out) {
  int group = Hq / Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  for (int h = 0; h < Hq; ++h) {
    int kh = h / group;
    double mx = -INFINITY;
    for (int t = 0; t < L; ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += h2d(q[(int64_t)h * D + d]) * h2d(k[((int64_t)t * Hkv + kh) * D + d]);
      s[t] = dot * scale;
      if (s[t] > mx) mx = s[t];
    }
    double den = 0.0;
    for (int t = 0; t < L; ++t) {
      s[t] = exp(s[t] - mx);
      den += s[t];
    }
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int t = 0; t < L; ++t) acc += s[t] * h2d(v[((int64_t)t * Hkv + kh) * D + d]);
      out[(int64_t)h * D + d] = d2h(L > 0 ? acc / den : 0.0);
    }
  }
  free(s);
}

/* Softmax probabilities of one head (used by the oracle's own tests). */
void orc_attention_probs(const uint16_t* q, const uint16_t* k, int Hq, int Hkv, int D, int L,
                         double scale, int h, double* p) {
  int kh = h / (Hq / Hkv);
  double mx = -INFINITY;
  for (int t = 0; t < L; ++t) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += h2d(q[(int64_t)h * D + d]) * h2d(k[((int64_t)t * Hkv + kh) * D + d]);
    p[t] = dot * scale;
    if (p[t] > mx) mx = p[t];
  }
  double den = 0.0;
  for (int t = 0; t < L; ++t) {
    p[t] = exp(p[t] - mx);
    den += p[t];
  }
  for (int t = 0; t < L; ++t) p[t] /= den;
}

/* Paged attention = gather through the block table, then the contiguous
 * definition.  q [B][Hq][D], out [B][Hq][D]. */
void orc_paged_attention(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                         const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                         int B, int Hq, int Hkv, int D, double scale, uint16_t* out) {
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    int L = context_lens[b];
    uint16_t* kc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(L > 0 ? L : 1) * Hkv * D);
    uint16_t* vc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(L > 0 ? L : 1) * Hkv * D);
    const int32_t* row = block_table + (int64_t)b * max_blocks;
    orc_gather_kv(k_pool, row, L, Hkv, D, kc);
    orc_gather_kv(v_pool, row, L, Hkv, D, vc);
    orc_attention(q + (int64_t)b * Hq * D, kc, vc, Hq, Hkv, D, L, scale,
                  out + (int64_t)b * Hq * D);
    free(kc);
    free(vc);
  }
}

/* ------------------------------------------------------------------------ */
/* FP8 KV pages.  [EN] "1. Weight Packing and FP8 Utilization" (twin: [ZH]   */
/* "1. 权重打包（Weight Packing）与 FP8 利用"): FP8 values need scaling        */
/* factors; E4M3 is one of the two FP8 formats it names.  Reading taken     */
/* here (the page gives no granularity): one fp32 scale per (page, kv head, */
/* token) row, chosen so the row's largest magnitude maps to 448 (the       */
/* largest finite E4M3 value); the pools hold the codes, [pages][Hkv][16][D] */
/* uint8, beside fp32 scales [pages][Hkv][16].                              */
/*                                                                          */
/* E4M3 ("fn" variant, no infinities): 1 sign bit, 4 exponent bits (bias   */
/* 7), 3 fraction bits; exponent field 0 is subnormal, fraction * 2^-9;     */
/* S.1111.111 is NaN; the largest finite value is 1.75 * 2^8 = 448.         */
/* ------------------------------------------------------------------------ */

double orc_e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int expo = (c >> 3) & 0xf;
  int frac = c & 0x7;
  double v;
  if (expo == 15 && frac == 7) return NAN;
  if (expo == 0) {
    v = ldexp((double)frac, -9);
  } else {
    v = ldexp((double)(8 + frac), expo - 10);
  }
  return sign ? -v : v;
}

/* Round-to-nearest-even encoding of an fp32 value; magnitudes past 448
 * saturate to 448 (no NaN for a finite input). */
uint8_t orc_float_to_e4m3(float f) {
  if (isnan(f)) return 0x7f;
  uint8_t sign = signbit(f) ? 0x80 : 0;
  double a = fabs((double)f);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: integer multiple of 2^-9, ties to even; 8 is the
     * smallest normal (exponent field 1, fraction 0) */
    double q = nearbyint(ldexp(a, 9));
    return sign | (uint8_t)q;
  }
  int e;
  (void)frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;                /* a = m * 2^E, m in [1, 2) */
  double m = nearbyint(ldexp(a, 3 - E)); /* in [8, 16] */
  if (m == 16.0) {
    m = 8.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && m > 14.0)) return sign | 0x7e; /* 448 */
  return sign | (uint8_t)((E + 7) << 3) | (uint8_t)((int)m - 8);
}

/* Quantise one row of D fp16 values: amax = max |x|, inv = 448 / amax and
 * scale = amax / 448 in fp32, code_i = E4M3(x_i * inv) with the product in
 * fp32 (an all-zero row gets scale 0 and zero codes).  Dequantised value:
 * code * scale. */
void orc_fp8_quantize_row(const uint16_t* x, int D, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int d = 0; d < D; ++d) {
    float a = (float)fabs(h2d(x[d]));
    if (a > amax) amax = a;
  }
  float inv = amax > 0.0f ? 448.0f / amax : 0.0f;
  for (int d = 0; d < D; ++d) {
    float y = (float)h2d(x[d]) * inv;
    codes[d] = orc_float_to_e4m3(y);
  }
  *scale = amax / 448.0f;
}

/* Append k[b][h][:] and v[b][h][:] (fp16, k already rotated) at position
 * context_lens[b]-1 of FP8 pools. */
void orc_kv_append_fp8(const uint16_t* k, const uint16_t* v, uint8_t* k_pool, uint8_t* v_pool,
                       float* k_scale, float* v_scale, const int32_t* block_table, int max_blocks,
                       const int32_t* context_lens, int B, int Hkv, int D) {
  for (int b = 0; b < B; ++b) {
    int pos = context_lens[b] - 1;
    int32_t page = block_table[(int64_t)b * max_blocks + pos / ORC_PAGE_TOKENS];
    int slot = pos % ORC_PAGE_TOKENS;
    for (int h = 0; h < Hkv; ++h) {
      int64_t row = ((int64_t)page * Hkv + h) * ORC_PAGE_TOKENS + slot;
      orc_fp8_quantize_row(k + ((int64_t)b * Hkv + h) * D, D, k_pool + row * D, &k_scale[row]);
      orc_fp8_quantize_row(v + ((int64_t)b * Hkv + h) * D, D, v_pool + row * D, &v_scale[row]);
    }
  }
}

/* Paged attention over FP8 pools: each gathered row dequantised (code *
 * scale, in fp64), then the same softmax attention as orc_attention. */
void orc_paged_attention_fp8(const uint16_t* q, const uint8_t* k_pool, const uint8_t* v_pool,
                             const float* k_scale, const float* v_scale, const int32_t* block_table,
                             int max_blocks, const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                             double scale, uint16_t* out) {
  int group = Hq / Hkv;
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    int L = context_lens[b];
    size_t n = (size_t)(L > 0 ? L : 1) * Hkv * D;
    double* kd = (double*)malloc(sizeof(double) * n);
    double* vd = (double*)malloc(sizeof(double) * n);
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    const int32_t* bt = block_table + (int64_t)b * max_blocks;
    for (int t = 0; t < L; ++t) {
      int32_t page = bt[t / ORC_PAGE_TOKENS];
      for (int h = 0; h < Hkv; ++h) {
        int64_t row = ((int64_t)page * Hkv + h) * ORC_PAGE_TOKENS + t % ORC_PAGE_TOKENS;
        for (int d = 0; d < D; ++d) {
          kd[((int64_t)t * Hkv + h) * D + d] = orc_e4m3_to_double(k_pool[row * D + d]) * (double)k_scale[row];
          vd[((int64_t)t * Hkv + h) * D + d] = orc_e4m3_to_double(v_pool[row * D + d]) * (double)v_scale[row];
        }
      }
    }
    for (int h = 0; h < Hq; ++h) {
      int kh = h / group;
      const uint16_t* qh = q + ((int64_t)b * Hq + h) * D;
      double mx = -INFINITY;
      for (int t = 0; t < L; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += h2d(qh[d]) * kd[((int64_t)t * Hkv + kh) * D + d];
        s[t] = dot * scale;
        if (s[t] > mx) mx = s[t];
      }
      double den = 0.0;
      for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - mx);
        den += s[t];
      }
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int t = 0; t < L; ++t) acc += s[t] * vd[((int64_t)t * Hkv + kh) * D + d];
        out[((int64_t)b * Hq + h) * D + d] = d2h(L > 0 ? acc / den : 0.0);
      }
    }
    free(kd);
    free(vd);
    free(s);
  }
}

/* Split-K (flash-decoding) form of one head's attention, kept in fp64:
 * the tokens are cut into partitions of `part` tokens; partition j keeps
 * m_j = max score, l_j = sum exp(s - m_j), o_j = sum exp(s - m_j) v.
 * The combine takes M = max m_j, l = sum l_j e^(m_j - M),
 * o = sum o_j e^(m_j - M) / l.  Returns out[D] in fp64.  Not on the pages;
 * it is the long-context form the decode path uses. */
void orc_attention_split_combine(const uint16_t* q, const uint16_t* k, const uint16_t* v, int Hq,
                                 int Hkv, int D, int L, double scale, int h, int part,
                                 double* out) {
  int kh = h / (Hq / Hkv);
  int P = (L + part - 1) / part;
  double* m = (double*)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
  double* l = (double*)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
  double* o = (double*)calloc((size_t)(P > 0 ? P : 1) * D, sizeof(double));
  for (int j = 0; j < P; ++j) {
    int t0 = j * part, t1 = t0 + part < L ? t0 + part : L;
    m[j] = -INFINITY;
    for (int t = t0; t < t1; ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += h2d(q[(int64_t)h * D + d]) * h2d(k[((int64_t)t * Hkv + kh) * D + d]);
      if (dot * scale > m[j]) m[j] = dot * scale;
    }
    l[j] = 0.0;
    for (int t = t0; t < t1; ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += h2d(q[(int64_t)h * D + d]) * h2d(k[((int64_t)t * Hkv + kh) * D + d]);
      double e = exp(dot * scale - m[j]);
      l[j] += e;
      for (int d = 0; d < D; ++d) o[(int64_t)j * D + d] += e * h2d(v[((int64_t)t * Hkv + kh) * D + d]);
    }
  }
  double M = -INFINITY;
  for (int j = 0; j < P; ++j)
    if (m[j] > M) M = m[j];
  double den = 0.0;
  for (int j = 0; j < P; ++j) den += l[j] * exp(m[j] - M);
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int j = 0; j < P; ++j) acc += o[(int64_t)j * D + d] * exp(m[j] - M);
    out[d] = acc / den;
  }
  free(m);
  free(l);
  free(o);
}

/* ------------------------------------------------------------------------ */
/* MLP gate (not on the pages; Qwen2 SwiGLU): m = fp16(silu(g) * u),        */
/* silu(g) = g / (1 + e^-g), g and u already rounded to fp16.               */
/* ------------------------------------------------------------------------ */
void orc_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* m) {
  for (int64_t i = 0; i < n; ++i) {
    double gv = h2d(g[i]);
    m[i] = d2h(gv / (1.0 + exp(-gv)) * h2d(u[i]));
  }
}

/* ------------------------------------------------------------------------ */
/* One Qwen2-shaped decoder layer and the whole decode step.                 */
/* ------------------------------------------------------------------------ */
typedef struct {
  int hidden, n_q_heads, n_kv_heads, head_dim, inter, n_layers, vocab;
  double eps, theta;
} orc_config;

typedef struct {
  const uint16_t *ln1, *ln2;                           /* [H] */
  const uint32_t *wq, *wk, *wv, *wo, *wg, *wu, *wd;    /* packed int4 */
  const uint16_t *sq, *sk, *sv, *so, *sg, *su, *sd;    /* group scales */
  const uint16_t *bq, *bk, *bv;                        /* nullable */
  uint16_t *k_pool, *v_pool;                           /* [pages][Hkv][16][D] */
  /* FP8 (E4M3) pools instead of k_pool / v_pool when k8 is set: codes
   * [pages][Hkv][16][D] and fp32 row scales [pages][Hkv][16] */
  uint8_t *k8, *v8;
  float *k_scale, *v_scale;
} orc_layer;

/* x [B][H] is replaced by the layer output.  context_lens are post-append. */
void orc_decoder_layer(const orc_config* c, const orc_layer* w, uint16_t* x,
                       const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                       int B) {
  int H = c->hidden, Hq = c->n_q_heads, Hkv = c->n_kv_heads, D = c->head_dim, I = c->inter;
  size_t szH = (size_t)B * H, szQ = (size_t)B * Hq * D, szK = (size_t)B * Hkv * D,
         szI = (size_t)B * I;
  uint16_t* xn = (uint16_t*)malloc(2 * szH);
  uint16_t* q = (uint16_t*)malloc(2 * szQ);
  uint16_t* k = (uint16_t*)malloc(2 * szK);
  uint16_t* v = (uint16_t*)malloc(2 * szK);
  uint16_t* att = (uint16_t*)malloc(2 * szQ);
  uint16_t* h = (uint16_t*)malloc(2 * szH);
  uint16_t* gt = (uint16_t*)malloc(2 * szI);
  uint16_t* up = (uint16_t*)malloc(2 * szI);
  uint16_t* mm = (uint16_t*)malloc(2 * szI);

  orc_rmsnorm(x, w->ln1, B, H, c->eps, xn);
  orc_w4a16_gemv(xn, B, H, w->wq, w->sq, Hq * D, w->bq, NULL, q);
  orc_w4a16_gemv(xn, B, H, w->wk, w->sk, Hkv * D, w->bk, NULL, k);
  orc_w4a16_gemv(xn, B, H, w->wv, w->sv, Hkv * D, w->bv, NULL, v);
  for (int b = 0; b < B; ++b) {
    int pos = context_lens[b] - 1;
    orc_rope(q + (size_t)b * Hq * D, Hq, D, pos, c->theta);
    orc_rope(k + (size_t)b * Hkv * D, Hkv, D, pos, c->theta);
  }
  if (w->k8) {
    /* the KV cache in FP8 pages: the new rows quantised, every row read back
     * as code * scale ([EN] "1. Weight Packing and FP8 Utilization") */
    orc_kv_append_fp8(k, v, w->k8, w->v8, w->k_scale, w->v_scale, block_table, max_blocks, context_lens, B,
                      Hkv, D);
    orc_paged_attention_fp8(q, w->k8, w->v8, w->k_scale, w->v_scale, block_table, max_blocks, context_lens,
                            B, Hq, Hkv, D, 1.0 / sqrt((double)D), att);
  } else {
    orc_kv_append(k, v, w->k_pool, w->v_pool, block_table, max_blocks, context_lens, B, Hkv, D);
    orc_paged_attention(q, w->k_pool, w->v_pool, block_table, max_blocks, context_lens, B, Hq, Hkv,
                        D, 1.0 / sqrt((double)D), att);
  }
  orc_w4a16_gemv(att, B, Hq * D, w->wo, w->so, H, NULL, x, h);
  orc_rmsnorm(h, w->ln2, B, H, c->eps, xn);
  orc_w4a16_gemv(xn, B, H, w->wg, w->sg, I, NULL, NULL, gt);
  orc_w4a16_gemv(xn, B, H, w->wu, w->su, I, NULL, NULL, up);
  orc_silu_mul(gt, up, (int64_t)szI, mm);
  orc_w4a16_gemv(mm, B, I, w->wd, w->sd, H, NULL, h, x);

  free(xn); free(q); free(k); free(v); free(att); free(h); free(gt); free(up); free(mm);
}

/* Whole decode step: embedding row gather -> layers -> final RMSNorm ->
 * fp16 lm_head -> argmax.  tokens_out [B]; logits_out [B][vocab] fp16 is
 * optional (NULL).  context_lens are post-append (every layer appends the
 * new token at len - 1).  n_layers_run lets a test stop early (<= n_layers). */
void orc_decode_step(const orc_config* c, const orc_layer* layers, int n_layers_run,
                     const uint16_t* embed, const uint16_t* final_norm, const uint16_t* lm_head,
                     const int32_t* tokens_in, const int32_t* block_table, int max_blocks,
                     const int32_t* context_lens, int B, int32_t* tokens_out,
                     uint16_t* logits_out, uint16_t* hidden_out) {
  int H = c->hidden, V = c->vocab;
  uint16_t* x = (uint16_t*)malloc(2 * (size_t)B * H);
  uint16_t* xn = (uint16_t*)malloc(2 * (size_t)B * H);
  double* logits = (double*)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; ++b)
    memcpy(x + (size_t)b * H, embed + (size_t)tokens_in[b] * H, 2 * (size_t)H);
  for (int l = 0; l < n_layers_run; ++l)
    orc_decoder_layer(c, &layers[l], x, block_table, max_blocks, context_lens, B);
  if (hidden_out) memcpy(hidden_out, x, 2 * (size_t)B * H);
  orc_rmsnorm(x, final_norm, B, H, c->eps, xn);
  for (int b = 0; b < B; ++b) {
    orc_fp16_gemv(xn + (size_t)b * H, H, lm_head, V, logits);
    tokens_out[b] = (int32_t)orc_argmax(logits, V);
    if (logits_out)
      for (int n = 0; n < V; ++n) logits_out[(size_t)b * V + n] = d2h(logits[n]);
  }
  free(x);
  free(xn);
  free(logits);
}
