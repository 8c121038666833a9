// int4_dot.cuh -- the INT4 x fp16 chunk product shared by the CUDA-core
// GEMV kernels (the stand-alone GEMVs and the persistent decode kernel).
//
// Per packed word w (nibbles u0..u7, u = q + 8), nibbles i and i + 4 sit 16
// bits apart, so one LOP3 drops a pair into the two halves of a half2 whose
// exponent field is that of 1024: (w & 0x000F000F) | 0x64006400 is
// half2{1024 + u0, 1024 + u4}, (w & 0x00F000F0) | 0x64006400 is
// half2{1024 + 16 u1, 1024 + 16 u5}, and the same on w >> 8 for u2/u6 and
// u3/u7.  Activations staged in the matching order ({x0,x4}, {x1,x5},
// {x2,x6}, {x3,x7} per word) meet them in mixed-precision fp16 x fp16 -> fp32
// FMAs (exact products, fp32 sums); over a 32-weight chunk
//   sum_i q_i x_i = A + B/16 - (1032 sum_{i even} x_i + 72 sum_{i odd} x_i)
// with A, B the sums over the even / odd nibble positions and the bracket
// staged once per chunk beside x.
#pragma once

#include "common.cuh"

namespace w4 {

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

constexpr uint32_t MAGIC_H2 = 0x64006400u;  // half2{1024, 1024}

constexpr int gcd_c(int x, int y) { return y == 0 ? x : gcd_c(y, x % y); }
constexpr int lcm_c(int x, int y) { return x / gcd_c(x, y) * y; }

// w >> 8 as the high word of an integer multiply, so it issues on the FMA
// pipe and leaves the half-rate ALU pipe to the LOP3s.
__device__ __forceinline__ uint32_t shr8_fma(uint32_t w) {
  uint32_t d;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(1u << 24));
  return d;
}

// Partial sums over the 8 nibbles of word w (nibble i = element i, offset
// binary u = q + 8) against x in staged order {x0,x4},{x1,x5},{x2,x6},{x3,x7}:
// a nibble ORed into the low mantissa bits of fp16 1024 is exactly 1024 + u,
// one placed four bits higher 1024 + 16 u, so
//   p[0] + p[1] = sum over i even of x_i (1024 + u_i),
//   p[2] + p[3] = sum over i odd  of x_i (1024 + 16 u_i),
// each product exact (fma.rn.f32.f16), and
//   sum_i x_i q_i = p0 + p1 + (p2 + p3) / 16 - 1032 sum_even x - 72 sum_odd x.
// One shift and four LOP3s per eight weights.
__device__ __forceinline__ void word_dot(float (&p)[4], uint32_t w, const uint4 xv) {
  const uint32_t w8 = shr8_fma(w);
  fma2_f16_f32_split(p[0], p[1], and_or(w, 0x000F000Fu, MAGIC_H2), xv.x);
  fma2_f16_f32_split(p[2], p[3], and_or(w, 0x00F000F0u, MAGIC_H2), xv.y);
  fma2_f16_f32_split(p[0], p[1], and_or(w8, 0x000F000Fu, MAGIC_H2), xv.z);
  fma2_f16_f32_split(p[2], p[3], and_or(w8, 0x00F000F0u, MAGIC_H2), xv.w);
}

// sum over a 32-weight chunk of x q from its partial sums and the chunk's
// activation constant c = 1032 sum_even x + 72 sum_odd x
__device__ __forceinline__ float chunk_sum(const float (&p)[4], float c) {
  return fmaf(0.0625f, p[2] + p[3], (p[0] + p[1]) - c);
}

// Stage x (optionally RMS-normalised, rounded to fp16) in shared memory in
// nibble order: for 32-weight chunk j and word w of the chunk, one uint4 holds
// {x0, x4}, {x1, x5}, {x2, x6}, {x3, x7} of k = 32 j + 8 w + i.
// Layout [MT][4][K/32] uint4, so consecutive chunks are consecutive 16 bytes.
// Beside it, per chunk, cs = 1032 sum_{i even} x + 72 sum_{i odd} x.
// Work unit: one 8-element group (16 bytes) per thread and step; the four
// groups of a chunk sit on four neighbouring lanes, which add their parts of
// cs with two shuffles.  With the RMSNorm the groups stay in registers
// between the sum of squares and the scaling (x and gamma are read once).
constexpr int STAGE_GMAX = 2;  // 8-element groups per thread held for the fused RMSNorm (K <= 4096 at 256 threads)

__device__ __forceinline__ void stage_group(uint4* xs, float* cs, int NCH, int m, int g, const __half (&h)[8],
                                            bool active) {
  float part = 0.f;
  if (active) {
    uint4 o;
    o.x = pack_h2(h[0], h[4]);
    o.y = pack_h2(h[1], h[5]);
    o.z = pack_h2(h[2], h[6]);
    o.w = pack_h2(h[3], h[7]);
    xs[(size_t)(m * 4 + (g & 3)) * NCH + (g >> 2)] = o;
    const float se = (__half2float(h[0]) + __half2float(h[2])) + (__half2float(h[4]) + __half2float(h[6]));
    const float so = (__half2float(h[1]) + __half2float(h[3])) + (__half2float(h[5]) + __half2float(h[7]));
    part = 1032.0f * se + 72.0f * so;
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  if (active && (g & 3) == 0) cs[(size_t)m * NCH + (g >> 2)] = part;
}

}  // namespace w4
