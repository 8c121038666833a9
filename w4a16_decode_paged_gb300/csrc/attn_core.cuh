// attn_core.cuh -- the per-page tensor-core step of the paged GQA decode
// attention, shared by the stand-alone attention kernel and the persistent
// decode kernel.
//
// Token t of a sequence lives in slot t % 16 of page block_table[t / 16]
// ("Building a Custom LLM Inference Runtime on H100", explore.n1n.ai,
// "2. The KV Cache and PagedAttention"); a (page, kv head) slice of the pool
// is 16 rows of 128 fp16.  In shared memory the rows sit 272 bytes apart (16
// bytes of padding), so the eight rows of an 8x8 ldmatrix tile fall on eight
// different bank groups.  The G query heads that share a kv head are the M
// rows (padded to 16) of warp-level mma.sync m16n8k16 products: the scores
// S = Q K^T, an fp32 online softmax in registers (exp2, scale folded in), and
// O += P V with the probabilities rounded to fp16 as the A operand.
#pragma once

#include <math.h>

#include "common.cuh"

namespace w4 {

constexpr int ATT_D = 128;
constexpr int ATT_PAGE = 16;
constexpr int ATT_SLICE = ATT_PAGE * ATT_D;        // halves per (page, kv head) slice in the pool
constexpr int ATT_PITCH = ATT_D + 8;               // halves per row in shared memory
constexpr int ATT_SSLICE = ATT_PAGE * ATT_PITCH;   // halves per slice in shared memory
constexpr unsigned long long ATT_TIMEOUT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// d += A (16 x 16, fp16, rows 8-15 zero) x B (16 x 8, fp16), fp32 accumulate.
// a0: A[g][2t..2t+1], a2: A[g][8+2t..8+2t+1]; b0, b1: B[2t..2t+1][g], B[8+2t..][g].
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// A fragments of the (rotated) query rows: lane (g = lane / 4, t4 = lane % 4)
// holds head g, dims 16 s + 2 t4 + {0, 1} and 16 s + 8 + 2 t4 + {0, 1} for the
// eight 16-dim k steps; heads g >= G are zero.
__device__ __forceinline__ void attn_q_frags(const float (*s_q)[ATT_D], int G, int g, int t4, uint32_t (&qa)[8][2]) {
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (g < G) {
      const float* qrow = s_q[g] + 16 * st + 2 * t4;
      const __half2 lo = __floats2half2_rn(qrow[0], qrow[1]);
      const __half2 hi = __floats2half2_rn(qrow[8], qrow[9]);
      qa[st][0] = *reinterpret_cast<const uint32_t*>(&lo);
      qa[st][1] = *reinterpret_cast<const uint32_t*>(&hi);
    } else {
      qa[st][0] = qa[st][1] = 0u;
    }
  }
}

// ldmatrix row addresses (bytes within a slice): lane l feeds row l % 8 of
// tile l / 8; K tiles are tokens x dims, V tiles (read transposed) tokens x dims.
__device__ __forceinline__ uint32_t attn_k_off(int lane) {
  const int lt = lane >> 3, lr8 = lane & 7;
  return (uint32_t)((((lt >> 1) * 8 + lr8) * ATT_PITCH + (lt & 1) * 8) * 2);
}
__device__ __forceinline__ uint32_t attn_v_off(int lane) {
  const int lt = lane >> 3, lr8 = lane & 7;
  return (uint32_t)((((lt & 1) * 8 + lr8) * ATT_PITCH + (lt >> 1) * 8) * 2);
}

// One page (nv >= 1 valid tokens, K rows at Ks and V rows at Vs in the padded
// layout) against the warp's query fragments: scores, online-softmax update
// of this lane's head (m_run in the log2 domain, l_run the running sum) and
// O = O * c + P V.  Warp-wide.
__device__ __forceinline__ void attn_page(const __half* Ks, const __half* Vs, int nv, const uint32_t (&qa)[8][2],
                                          float scale_log2, uint32_t k_off, uint32_t v_off, int t4, float& m_run,
                                          float& l_run, float (&o)[16][4]) {
  // ---- scores S[head][token], tokens 0-7 (n-block 0) and 8-15 (1) -------
  float sc[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
  const uint32_t kbase = smem_u32(Ks) + k_off;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    uint32_t b0, b1, b2, b3;  // (tokens 0-7: dims lo, hi), (tokens 8-15: dims lo, hi)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(kbase + st * 32));
    mma_16816(sc[0], qa[st][0], qa[st][1], b0, b1);
    mma_16816(sc[1], qa[st][0], qa[st][1], b2, b3);
  }
  // ---- online softmax over this page (row g; four lanes share a row) ----
  float s00 = sc[0][0] * scale_log2, s01 = sc[0][1] * scale_log2;
  float s10 = sc[1][0] * scale_log2, s11 = sc[1][1] * scale_log2;
  if (2 * t4 >= nv) s00 = -INFINITY;
  if (2 * t4 + 1 >= nv) s01 = -INFINITY;
  if (8 + 2 * t4 >= nv) s10 = -INFINITY;
  if (8 + 2 * t4 + 1 >= nv) s11 = -INFINITY;
  float mx = fmaxf(fmaxf(s00, s01), fmaxf(s10, s11));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(m_run, mx);  // finite: token 0 of the page is valid
  const float c = exp2f(m_run - m_new);  // 0 while m_run is -inf
  const float p00 = exp2f(s00 - m_new), p01 = exp2f(s01 - m_new);
  const float p10 = exp2f(s10 - m_new), p11 = exp2f(s11 - m_new);
  float sum = (p00 + p01) + (p10 + p11);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  l_run = l_run * c + sum;
  m_run = m_new;
  const __half2 pa = __floats2half2_rn(p00, p01), pb = __floats2half2_rn(p10, p11);
  const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&pa), a2 = *reinterpret_cast<const uint32_t*>(&pb);
  // ---- O = O * c + P V ----------------------------------------------------
  const uint32_t vbase = smem_u32(Vs) + v_off;
#pragma unroll
  for (int nb = 0; nb < 16; nb += 2) {
    uint32_t b0, b1, b2, b3;  // (dims 8nb: tokens 0-7, 8-15), (dims 8nb+8: tokens 0-7, 8-15)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(vbase + nb * 16));
    o[nb][0] *= c;
    o[nb][1] *= c;
    o[nb + 1][0] *= c;
    o[nb + 1][1] *= c;
    mma_16816(o[nb], a0, a2, b0, b1);
    mma_16816(o[nb + 1], a0, a2, b2, b3);
  }
}

// The same page step for half of the head dimensions: P V only for dims
// [64 dh, 64 dh + 64) (o holds those 8 n-blocks).  Two warps that share a page,
// one per half, keep identical softmax states and half the accumulators each.
__device__ __forceinline__ void attn_page_half(const __half* Ks, const __half* Vs, int nv, const uint32_t (&qa)[8][2],
                                               float scale_log2, uint32_t k_off, uint32_t v_off, int t4, int dh,
                                               float& m_run, float& l_run, float (&o)[8][4]) {
  float sc[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
  const uint32_t kbase = smem_u32(Ks) + k_off;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    uint32_t b0, b1, b2, b3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(kbase + st * 32));
    mma_16816(sc[0], qa[st][0], qa[st][1], b0, b1);
    mma_16816(sc[1], qa[st][0], qa[st][1], b2, b3);
  }
  float s00 = sc[0][0] * scale_log2, s01 = sc[0][1] * scale_log2;
  float s10 = sc[1][0] * scale_log2, s11 = sc[1][1] * scale_log2;
  if (2 * t4 >= nv) s00 = -INFINITY;
  if (2 * t4 + 1 >= nv) s01 = -INFINITY;
  if (8 + 2 * t4 >= nv) s10 = -INFINITY;
  if (8 + 2 * t4 + 1 >= nv) s11 = -INFINITY;
  float mx = fmaxf(fmaxf(s00, s01), fmaxf(s10, s11));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float c = exp2f(m_run - m_new);
  const float p00 = exp2f(s00 - m_new), p01 = exp2f(s01 - m_new);
  const float p10 = exp2f(s10 - m_new), p11 = exp2f(s11 - m_new);
  float sum = (p00 + p01) + (p10 + p11);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  l_run = l_run * c + sum;
  m_run = m_new;
  const __half2 pa = __floats2half2_rn(p00, p01), pb = __floats2half2_rn(p10, p11);
  const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&pa), a2 = *reinterpret_cast<const uint32_t*>(&pb);
  const uint32_t vbase = smem_u32(Vs) + v_off + (uint32_t)(dh * 128);
#pragma unroll
  for (int nb = 0; nb < 8; nb += 2) {
    uint32_t b0, b1, b2, b3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(vbase + nb * 16));
    o[nb][0] *= c;
    o[nb][1] *= c;
    o[nb + 1][0] *= c;
    o[nb + 1][1] *= c;
    mma_16816(o[nb], a0, a2, b0, b1);
    mma_16816(o[nb + 1], a0, a2, b2, b3);
  }
}

// d += A (16 x 16, fp16, all rows) x B (16 x 8, fp16), fp32 accumulate.
// a0: A[g][2t..], a1: A[8+g][2t..], a2: A[g][8+2t..], a3: A[8+g][8+2t..].
__device__ __forceinline__ void mma_16816_full(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One page against two query tokens at once (causal prompt attention): the
// MMA's rows 0-7 are the heads of token A, rows 8-15 those of token B
// (qa[st][0..3] = a0..a3 of k step st).  Keys at positions past a row's own
// position (page tokens tok0 + n > pos) are masked.  Per lane: the states of
// row g (token A) and row 8 + g (token B); o[nb][0..1] row g, o[nb][2..3]
// row 8 + g.  Warp-wide.
__device__ __forceinline__ void attn_page_pair(const __half* Ks, const __half* Vs, int tok0, int posA, int posB,
                                               const uint32_t (&qa)[8][4], float scale_log2, uint32_t k_off,
                                               uint32_t v_off, int t4, float (&m_run)[2], float (&l_run)[2],
                                               float (&o)[16][4]) {
  float sc[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
  const uint32_t kbase = smem_u32(Ks) + k_off;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    uint32_t b0, b1, b2, b3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(kbase + st * 32));
    mma_16816_full(sc[0], qa[st][0], qa[st][1], qa[st][2], qa[st][3], b0, b1);
    mma_16816_full(sc[1], qa[st][0], qa[st][1], qa[st][2], qa[st][3], b2, b3);
  }
  // s[r][j]: row r (0: token A, 1: token B), page token n = 8 (j >> 1) + 2 t4 + (j & 1)
  float s[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int pos = r ? posB : posA;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = 8 * (j >> 1) + 2 * t4 + (j & 1);
      const float v = sc[j >> 1][2 * r + (j & 1)] * scale_log2;
      s[r][j] = (tok0 + n <= pos) ? v : -INFINITY;
    }
  }
  float c[2], p[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float mx = fmaxf(fmaxf(s[r][0], s[r][1]), fmaxf(s[r][2], s[r][3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run[r], mx);
    // a row with no valid key yet keeps m = -inf: nothing to rescale, no weight
    const bool none = m_new == -INFINITY;
    c[r] = none ? 1.f : exp2f(m_run[r] - m_new);
#pragma unroll
    for (int j = 0; j < 4; ++j) p[r][j] = none ? 0.f : exp2f(s[r][j] - m_new);
    float sum = (p[r][0] + p[r][1]) + (p[r][2] + p[r][3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    l_run[r] = l_run[r] * c[r] + sum;
    m_run[r] = m_new;
  }
  const __half2 h0 = __floats2half2_rn(p[0][0], p[0][1]), h1 = __floats2half2_rn(p[1][0], p[1][1]);
  const __half2 h2 = __floats2half2_rn(p[0][2], p[0][3]), h3 = __floats2half2_rn(p[1][2], p[1][3]);
  const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&h0), a1 = *reinterpret_cast<const uint32_t*>(&h1);
  const uint32_t a2 = *reinterpret_cast<const uint32_t*>(&h2), a3 = *reinterpret_cast<const uint32_t*>(&h3);
  const uint32_t vbase = smem_u32(Vs) + v_off;
#pragma unroll
  for (int nb = 0; nb < 16; nb += 2) {
    uint32_t b0, b1, b2, b3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(vbase + nb * 16));
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      o[nb + e][0] *= c[0];
      o[nb + e][1] *= c[0];
      o[nb + e][2] *= c[1];
      o[nb + e][3] *= c[1];
    }
    mma_16816_full(o[nb], a0, a1, a2, a3, b0, b1);
    mma_16816_full(o[nb + 1], a0, a1, a2, a3, b2, b3);
  }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) pages: a (page, kv head) slice holds 16 rows of 128 one-byte
// codes per K and V plus one fp32 scale per row (value = code * scale).  In
// shared memory the code rows sit 144 bytes apart (16 bytes of padding: the
// 16-bit fragment loads of eight rows fall on eight bank groups), followed
// by the 16 K and 16 V scales.
// ---------------------------------------------------------------------------
constexpr int ATT8_PITCH = ATT_D + 16;                         // bytes per code row in shared memory
constexpr int ATT8_CODES = ATT_PAGE * ATT8_PITCH;              // bytes of one slice's K (or V) codes
constexpr int ATT8_SLOT = 2 * ATT8_CODES + 2 * ATT_PAGE * 4;   // K codes | V codes | K scales | V scales
static_assert(ATT8_SLOT % 16 == 0, "slots stay 16-byte aligned");

// two E4M3 codes (low byte first) -> half2 (exact: every E4M3 value is an fp16)
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
  uint32_t d;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(d) : "r"(two));
  return d;
}
// E4M3 codes of two fp32 values, round to nearest even, saturating at 448:
// lo in the low byte, hi in the high byte
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint32_t d;
  asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tcvt.u32.u16 %0, c;\n\t}"
      : "=r"(d)
      : "f"(hi), "f"(lo));
  return d;
}

// Four E4M3 codes (bytes 0..3 of w) -> half2 of bytes (0, 1) and of (2, 3).
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// FP8 pages are read with 16-byte loads by permuting the two contractions'
// index order (a sum does not depend on the order of its terms):
//  * Q K^T: the MMA step st, lane quad t4 multiplies (logical k) pairs
//    2 t4 + {0,1} and 8 + 2 t4 + {0,1}; they are taken as the physical dims
//    p0 + {0,1} and p0 + {2,3} with p0 = 64 (st / 4) + 16 t4 + 4 (st % 4), so
//    a lane's K codes for steps 0-3 (4-7) are the 16 bytes at 16 t4 (64 +
//    16 t4) of the token's row.  The query fragments use the same order.
//  * P V: n-block nb, column n is output dim 16 n + nb (not 8 nb + n), so the
//    16 V codes a lane needs from a token row are the 16 bytes at 16 g.  The
//    accumulator column 2 t4 + e of n-block nb is then dim 32 t4 + 16 e + nb.
__device__ __forceinline__ int attn8_qdim(int st, int t4) { return 64 * (st >> 2) + 16 * t4 + 4 * (st & 3); }
__device__ __forceinline__ int attn8_odim(int nb, int t4, int e) { return 32 * t4 + 16 * e + nb; }

// Query fragments in the FP8 pages' dim order (see above); heads g >= G are zero.
__device__ __forceinline__ void attn_q_frags_fp8(const float (*s_q)[ATT_D], int G, int g, int t4,
                                                 uint32_t (&qa)[8][2]) {
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (g < G) {
      const float4 q4 = *reinterpret_cast<const float4*>(s_q[g] + attn8_qdim(st, t4));
      const __half2 lo = __floats2half2_rn(q4.x, q4.y);
      const __half2 hi = __floats2half2_rn(q4.z, q4.w);
      qa[st][0] = *reinterpret_cast<const uint32_t*>(&lo);
      qa[st][1] = *reinterpret_cast<const uint32_t*>(&hi);
    } else {
      qa[st][0] = qa[st][1] = 0u;
    }
  }
}

// One FP8 page against the warp's query fragments (built by attn_q_frags_fp8):
// scores scaled by the K row scales, probabilities by the V row scales before
// P V (the softmax sum keeps the unscaled probabilities); o in the FP8 output
// dim order (attn8_odim).
__device__ __forceinline__ void attn_page_fp8(const unsigned char* slot, int nv, const uint32_t (&qa)[8][2],
                                              float scale_log2, int g, int t4, float& m_run, float& l_run,
                                              float (&o)[16][4]) {
  const unsigned char* Kc = slot;
  const unsigned char* Vc = slot + ATT8_CODES;
  const float* ks = reinterpret_cast<const float*>(slot + 2 * ATT8_CODES);
  const float* vs = ks + ATT_PAGE;
  // K codes: tokens g (n-block 0) and 8 + g (n-block 1), dims [16 t4, +16) and [64 + 16 t4, +16)
  uint4 kw[2][2];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      kw[r][h] = *reinterpret_cast<const uint4*>(Kc + (g + 8 * r) * ATT8_PITCH + 64 * h + 16 * t4);
  // V codes (used after the softmax, loaded now): tokens 2 t4, 2 t4 + 1, 8 + 2 t4, 9 + 2 t4,
  // dims [16 g, +16) (dim 16 g + nb of n-block nb)
  uint4 vw[4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
    vw[r] = *reinterpret_cast<const uint4*>(Vc + (2 * t4 + (r & 1) + 8 * (r >> 1)) * ATT8_PITCH + 16 * g);
  // the 8 k steps of each n-block alternate between two accumulators
  float sc[2][4], sd[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nb][e] = sd[nb][e] = 0.f;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    uint32_t b0, b1, b2, b3;
    e4m3x4_to_h2x2((&kw[0][st >> 2].x)[st & 3], b0, b1);
    e4m3x4_to_h2x2((&kw[1][st >> 2].x)[st & 3], b2, b3);
    float (&acc)[2][4] = (st & 1) ? sd : sc;
    mma_16816(acc[0], qa[st][0], qa[st][1], b0, b1);
    mma_16816(acc[1], qa[st][0], qa[st][1], b2, b3);
  }
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nb][e] += sd[nb][e];
  float s00 = sc[0][0] * ks[2 * t4] * scale_log2, s01 = sc[0][1] * ks[2 * t4 + 1] * scale_log2;
  float s10 = sc[1][0] * ks[8 + 2 * t4] * scale_log2, s11 = sc[1][1] * ks[9 + 2 * t4] * scale_log2;
  if (2 * t4 >= nv) s00 = -INFINITY;
  if (2 * t4 + 1 >= nv) s01 = -INFINITY;
  if (8 + 2 * t4 >= nv) s10 = -INFINITY;
  if (8 + 2 * t4 + 1 >= nv) s11 = -INFINITY;
  float mx = fmaxf(fmaxf(s00, s01), fmaxf(s10, s11));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float c = exp2f(m_run - m_new);
  const float p00 = exp2f(s00 - m_new), p01 = exp2f(s01 - m_new);
  const float p10 = exp2f(s10 - m_new), p11 = exp2f(s11 - m_new);
  float sum = (p00 + p01) + (p10 + p11);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  l_run = l_run * c + sum;
  m_run = m_new;
  const __half2 pa = __floats2half2_rn(p00 * vs[2 * t4], p01 * vs[2 * t4 + 1]);
  const __half2 pb = __floats2half2_rn(p10 * vs[8 + 2 * t4], p11 * vs[9 + 2 * t4]);
  const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&pa), a2 = *reinterpret_cast<const uint32_t*>(&pb);
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    const uint32_t sel = (uint32_t)(nb & 3) | ((uint32_t)(4 + (nb & 3)) << 4);
    uint32_t pair0, pair1;  // (token 2 t4, 2 t4 + 1) and (8 + 2 t4, 9 + 2 t4) of dim 16 g + nb
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pair0) : "r"((&vw[0].x)[nb >> 2]), "r"((&vw[1].x)[nb >> 2]), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pair1) : "r"((&vw[2].x)[nb >> 2]), "r"((&vw[3].x)[nb >> 2]), "r"(sel));
    const uint32_t b0 = e4m3x2_to_h2(pair0);
    const uint32_t b1 = e4m3x2_to_h2(pair1);
    o[nb][0] *= c;
    o[nb][1] *= c;
    mma_16816(o[nb], a0, a2, b0, b1);
  }
}

// attn_page_pair over an FP8 page (codes and row scales as attn_page_fp8
// reads them): two query tokens at once, query fragments qa[st][0..3] in the
// FP8 dim order (attn8_qdim), o in the FP8 output dim order (attn8_odim).
__device__ __forceinline__ void attn_page_pair_fp8(const unsigned char* slot, int tok0, int posA, int posB,
                                                   const uint32_t (&qa)[8][4], float scale_log2, int g, int t4,
                                                   float (&m_run)[2], float (&l_run)[2], float (&o)[16][4]) {
  const unsigned char* Kc = slot;
  const unsigned char* Vc = slot + ATT8_CODES;
  const float* ks = reinterpret_cast<const float*>(slot + 2 * ATT8_CODES);
  const float* vs = ks + ATT_PAGE;
  float sc[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
  uint4 kw[2][2];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      kw[r][h] = *reinterpret_cast<const uint4*>(Kc + (g + 8 * r) * ATT8_PITCH + 64 * h + 16 * t4);
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    uint32_t b0, b1, b2, b3;
    e4m3x4_to_h2x2((&kw[0][st >> 2].x)[st & 3], b0, b1);
    e4m3x4_to_h2x2((&kw[1][st >> 2].x)[st & 3], b2, b3);
    mma_16816_full(sc[0], qa[st][0], qa[st][1], qa[st][2], qa[st][3], b0, b1);
    mma_16816_full(sc[1], qa[st][0], qa[st][1], qa[st][2], qa[st][3], b2, b3);
  }
  float s[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int pos = r ? posB : posA;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = 8 * (j >> 1) + 2 * t4 + (j & 1);
      const float v = sc[j >> 1][2 * r + (j & 1)] * ks[n] * scale_log2;
      s[r][j] = (tok0 + n <= pos) ? v : -INFINITY;
    }
  }
  float c[2], p[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float mx = fmaxf(fmaxf(s[r][0], s[r][1]), fmaxf(s[r][2], s[r][3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run[r], mx);
    const bool none = m_new == -INFINITY;
    c[r] = none ? 1.f : exp2f(m_run[r] - m_new);
#pragma unroll
    for (int j = 0; j < 4; ++j) p[r][j] = none ? 0.f : exp2f(s[r][j] - m_new);
    float sum = (p[r][0] + p[r][1]) + (p[r][2] + p[r][3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    l_run[r] = l_run[r] * c[r] + sum;
    m_run[r] = m_new;
  }
  // P times the V row scales (token n = 8 (j >> 1) + 2 t4 + (j & 1)) as the A operand
  const float v0 = vs[2 * t4], v1 = vs[2 * t4 + 1], v8 = vs[8 + 2 * t4], v9 = vs[9 + 2 * t4];
  const __half2 h0 = __floats2half2_rn(p[0][0] * v0, p[0][1] * v1), h1 = __floats2half2_rn(p[1][0] * v0, p[1][1] * v1);
  const __half2 h2 = __floats2half2_rn(p[0][2] * v8, p[0][3] * v9), h3 = __floats2half2_rn(p[1][2] * v8, p[1][3] * v9);
  const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&h0), a1 = *reinterpret_cast<const uint32_t*>(&h1);
  const uint32_t a2 = *reinterpret_cast<const uint32_t*>(&h2), a3 = *reinterpret_cast<const uint32_t*>(&h3);
  uint4 vw[4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
    vw[r] = *reinterpret_cast<const uint4*>(Vc + (2 * t4 + (r & 1) + 8 * (r >> 1)) * ATT8_PITCH + 16 * g);
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    const uint32_t sel = (uint32_t)(nb & 3) | ((uint32_t)(4 + (nb & 3)) << 4);
    uint32_t pair0, pair1;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pair0) : "r"((&vw[0].x)[nb >> 2]), "r"((&vw[1].x)[nb >> 2]), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pair1) : "r"((&vw[2].x)[nb >> 2]), "r"((&vw[3].x)[nb >> 2]), "r"(sel));
    o[nb][0] *= c[0];
    o[nb][1] *= c[0];
    o[nb][2] *= c[1];
    o[nb][3] *= c[1];
    mma_16816_full(o[nb], a0, a1, a2, a3, e4m3x2_to_h2(pair0), e4m3x2_to_h2(pair1));
  }
}

}  // namespace w4
