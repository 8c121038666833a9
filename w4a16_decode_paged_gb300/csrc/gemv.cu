// gemv.cu -- W4A16 GEMV for decode (M <= 4 activation rows), CUDA cores.
//
// Computes y[m][n] = sum_k x[m][k] * q[n][k] * s[n][k/128] (+bias, +residual)
// for symmetric group-wise INT4 weights (group 128) with fp16 activations,
// as the aikraft.ru article "How to build your own LLM runtime from scratch"
// describes in "Архитектурные решения и оптимизации".  That section notes a
// byte-permute unpack beat the dp4a/INT8-activation path on Hopper; here the
// unpack is two LOP3s per pair of nibbles (magic-number fp16 construction)
// and the products run as mixed-precision fp16 x fp16 -> fp32 FMAs, so every
// product is exact and every sum is fp32.
//
// Dequant trick, per packed word w (nibbles u0..u7, u = q + 8):
//   (w      & 0x000F000F) | 0x64006400 = half2{1024 + u0, 1024 + u4}
//   (w      & 0x00F000F0) | 0x64006400 = half2{1024 + 16 u1, 1024 + 16 u5}
//   (w >> 8 & 0x000F000F) | 0x64006400 = half2{1024 + u2, 1024 + u6}
//   (w >> 8 & 0x00F000F0) | 0x64006400 = half2{1024 + 16 u3, 1024 + 16 u7}
// One HSUB2 each turns these into exact codes: minus 1032 gives q for the
// even nibbles, minus 1152 gives 16 q for the odd ones.  The activations are
// staged once per CTA in shared memory in the matching order, with the
// odd-nibble ones pre-divided by 16 (exact), so every product (16 q)(x / 16)
// is exact in fp32.  That is one shift, four LOP3, four HSUB2 and eight FMAs
// per 8 weights.  (Folding the 1032 offset into the sum instead would save
// the HSUB2s but costs about eight bits of the fp32 sum when |x| is large.)
//
// Work split: LPR lanes cooperate on one weight row (LPR = 16 when K/32 is a
// multiple of 16, else 8 or 4); a warp covers 32/LPR rows at a time; each
// lane streams 16-byte words with 128-bit non-allocating loads, GEMV_U of
// them in flight, and the row sum is a shuffle reduction over LPR lanes.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "kernels.h"

namespace w4 {

constexpr int GEMV_WPB = 8;  // warps per block
constexpr int GEMV_U = 8;    // 16-byte weight loads in flight per lane

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

template <int LPR, int MT, bool SILU>
__global__ void __launch_bounds__(GEMV_WPB * 32) gemv_w4a16_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int RPW = 32 / LPR;               // row slots per warp
  constexpr int RPT = SILU ? RPW / 2 : RPW;   // output rows per warp task
  constexpr uint32_t MAGIC = 0x64006400u;     // half2{1024, 1024}
  constexpr uint32_t EVEN_OFF = 0x64086408u;  // half2{1032, 1032}
  constexpr uint32_t ODD_OFF = 0x64806480u;   // half2{1152, 1152}
  extern __shared__ uint4 smem[];
  const int K = a.K, M = a.M;
  const int NCH = K >> 5;      // 32-weight chunks per row
  const int NIT = NCH / LPR;   // chunks per lane per row
  uint4* xs = smem;  // [MT][4][NCH]
  __shared__ float red[GEMV_WPB][MT];
  __shared__ float rscale[MT];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = lane / LPR, lr = lane % LPR;
  const int ntask = (a.N + RPT - 1) / RPT;
  const int nwarps = gridDim.x * GEMV_WPB;

  // Weights do not depend on the previous kernel: let the next kernel start
  // early and issue this warp's first batch of weight loads before waiting.
  pdl_launch_dependents();

  int task = blockIdx.x * GEMV_WPB + warp;
  uint4 wb[GEMV_U];
  __half sb[GEMV_U];

  // Resolve (weight row pointer, scale row pointer, bias, output row) for a task.
  const uint32_t* qrow = nullptr;
  const __half* srow = nullptr;
  const __half* brow = nullptr;
  int out_row = 0;
  bool valid = false;
  auto resolve = [&](int t) {
    if (SILU) {
      out_row = t * RPT + (slot % RPT);
      const GemvSeg& sg = a.seg[slot / RPT];
      valid = out_row < a.N;
      int r = valid ? out_row : 0;
      qrow = sg.qw + (size_t)r * (K >> 3);
      srow = sg.s + (size_t)r * (K >> 7);
      brow = nullptr;
    } else {
      out_row = t * RPT + slot;
      valid = out_row < a.N;
      int r = valid ? out_row : 0;
      int si = 0;
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (si < a.nseg - 1 && r >= a.seg[si].rows) { r -= a.seg[si].rows; ++si; }
      const GemvSeg& sg = a.seg[si];
      qrow = sg.qw + (size_t)r * (K >> 3);
      srow = sg.s + (size_t)r * (K >> 7);
      brow = sg.bias ? sg.bias + r : nullptr;
    }
  };

  if (task < ntask) {
    resolve(task);
#pragma unroll
    for (int u = 0; u < GEMV_U; ++u) {
      if (u < NIT && valid) {
        int j = lr + LPR * u;
        wb[u] = ldg_stream(qrow + 4 * j);
        sb[u] = srow[j >> 2];
      }
    }
  }

  pdl_wait();  // x (and residual) come from the previous kernel

  // ---- stage x' (permuted, odd nibbles pre-scaled by 1/16) and C ----------
  if (a.gamma != nullptr) {
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        uint4 raw = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + k);
        const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v = __half2float(h[i]);
          ss = fmaf(v, v, ss);
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp][0] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < GEMV_WPB; ++w) t += red[w][0];
        rscale[m] = 1.0f / sqrtf(t / (float)K + a.eps);
      }
      __syncthreads();
    }
  }
  const __half sixteenth = __float2half(0.0625f);
  for (int idx = threadIdx.x; idx < M * NCH; idx += blockDim.x) {
    const int m = idx / NCH, j = idx - m * NCH;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)m * K + 32 * j);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint4 raw = src[wi];
      __half h[8];
      *reinterpret_cast<uint4*>(h) = raw;
      if (a.gamma != nullptr) {
        uint4 graw = *reinterpret_cast<const uint4*>(a.gamma + 32 * j + 8 * wi);
        const __half* g = reinterpret_cast<const __half*>(&graw);
        const float r = rscale[m];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __float2half_rn(__half2float(h[i]) * r * __half2float(g[i]));
      }
      uint4 o;
      o.x = pack_h2(h[0], h[4]);
      o.y = pack_h2(__hmul(h[1], sixteenth), __hmul(h[5], sixteenth));
      o.z = pack_h2(h[2], h[6]);
      o.w = pack_h2(__hmul(h[3], sixteenth), __hmul(h[7], sixteenth));
      xs[(size_t)(m * 4 + wi) * NCH + j] = o;
    }
  }
  __syncthreads();

  // ---- main loop over this warp's tasks -----------------------------------
  for (; task < ntask; task += nwarps) {
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;

    for (int it0 = 0; it0 < NIT; it0 += GEMV_U) {
      uint4 wc[GEMV_U];
      __half sc[GEMV_U];
#pragma unroll
      for (int u = 0; u < GEMV_U; ++u) {
        wc[u] = wb[u];
        sc[u] = sb[u];
      }
      // prefetch the next batch of this row
      if (it0 + GEMV_U < NIT && valid) {
#pragma unroll
        for (int u = 0; u < GEMV_U; ++u) {
          int it = it0 + GEMV_U + u;
          if (it < NIT) {
            int j = lr + LPR * it;
            wb[u] = ldg_stream(qrow + 4 * j);
            sb[u] = srow[j >> 2];
          }
        }
      }
      if (valid) {
#pragma unroll
        for (int u = 0; u < GEMV_U; ++u) {
          const int it = it0 + u;
          if (it < NIT) {
            const int j = lr + LPR * it;
            const uint32_t* wv = reinterpret_cast<const uint32_t*>(&wc[u]);
            const float s = __half2float(sc[u]);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m < M) {
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                  const uint32_t w = wv[wi];
                  const uint32_t w8 = w >> 8;
                  const uint4 xv = xs[(size_t)(m * 4 + wi) * NCH + j];
                  fma2_f16_f32_split(p0, p1, hsub2(and_or(w, 0x000F000Fu, MAGIC), EVEN_OFF), xv.x);
                  fma2_f16_f32_split(p0, p1, hsub2(and_or(w, 0x00F000F0u, MAGIC), ODD_OFF), xv.y);
                  fma2_f16_f32_split(p0, p1, hsub2(and_or(w8, 0x000F000Fu, MAGIC), EVEN_OFF), xv.z);
                  fma2_f16_f32_split(p0, p1, hsub2(and_or(w8, 0x00F000F0u, MAGIC), ODD_OFF), xv.w);
                }
                acc[m] = fmaf(p0 + p1, s, acc[m]);
              }
            }
          }
        }
      }
    }

    // ---- reduce over the LPR lanes of each row, epilogue ------------------
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
    }
    if (SILU) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float other = __shfl_xor_sync(0xffffffffu, acc[m], 16);
        if (m < M && valid && lr == 0 && slot < RPT) {
          // gate and up are rounded to fp16 like two separate GEMV outputs
          const float g = __half2float(__float2half_rn(acc[m]));
          const float u = __half2float(__float2half_rn(other));
          const float silu = g / (1.0f + expf(-g));
          a.y[(size_t)m * a.N + out_row] = __float2half_rn(silu * u);
        }
      }
    } else if (valid && lr == 0) {
      const float b = brow ? __half2float(*brow) : 0.f;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          float v = acc[m] + b;
          if (a.residual) v += __half2float(a.residual[(size_t)m * a.N + out_row]);
          a.y[(size_t)m * a.N + out_row] = __float2half_rn(v);
        }
      }
    }

    // issue the first batch of the next task
    const int nt = task + nwarps;
    if (nt < ntask) {
      resolve(nt);
      if (valid) {
#pragma unroll
        for (int u = 0; u < GEMV_U; ++u) {
          if (u < NIT) {
            int j = lr + LPR * u;
            wb[u] = ldg_stream(qrow + 4 * j);
            sb[u] = srow[j >> 2];
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int LPR, int MT, bool SILU>
static int launch_one(const GemvArgs& a, cudaStream_t s) {
  auto kern = gemv_w4a16_kernel<LPR, MT, SILU>;
  const size_t smem = (size_t)MT * a.K * 2;
  static int configured = 0;
  static int blocks_per_sm = 0;
  if (!configured) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 110 * 1024);
    configured = 1;
  }
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, GEMV_WPB * 32, smem) != cudaSuccess || bps < 1)
    bps = 1;
  (void)blocks_per_sm;
  constexpr int RPT = SILU ? (32 / LPR) / 2 : 32 / LPR;
  const int ntask = (a.N + RPT - 1) / RPT;
  int blocks = (ntask + GEMV_WPB - 1) / GEMV_WPB;
  blocks = std::min(blocks, bps * num_sms());
  blocks = std::max(blocks, 1);
  cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(GEMV_WPB * 32), smem, s, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

template <int MT, bool SILU>
static int dispatch_lpr(const GemvArgs& a, cudaStream_t s) {
  const int nch = a.K / 32;
  if (nch % 16 == 0) return launch_one<16, MT, SILU>(a, s);
  if (nch % 8 == 0) return launch_one<8, MT, SILU>(a, s);
  return launch_one<4, MT, SILU>(a, s);
}

int gemv_cuda_core_supported(int M, int K) { return M >= 1 && M <= 4 && (long)M * K <= 49152; }

int launch_gemv(const GemvArgs& a, bool silu, cudaStream_t s) {
  if (!gemv_cuda_core_supported(a.M, a.K))
    return set_error(W4A16_ERR_SHAPE, "gemv: M=%d K=%d outside the CUDA-core path (M<=4, M*K<=49152)", a.M, a.K);
  if (silu) {
    if (a.M == 1) return dispatch_lpr<1, true>(a, s);
    if (a.M == 2) return dispatch_lpr<2, true>(a, s);
    return dispatch_lpr<4, true>(a, s);
  }
  if (a.M == 1) return dispatch_lpr<1, false>(a, s);
  if (a.M == 2) return dispatch_lpr<2, false>(a, s);
  return dispatch_lpr<4, false>(a, s);
}

}  // namespace w4

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
using namespace w4;

static int check_gemv_common(const uint16_t* x, int M, int K, int N, const uint16_t* y) {
  W4_CHECK_ARG(x && y, "gemv: x and y must be non-null");
  W4_CHECK_ARG(M >= 1 && K >= 1 && N >= 1, "gemv: sizes must be positive (M=%d K=%d N=%d)", M, K, N);
  W4_CHECK_SHAPE(K % 128 == 0, "gemv: K=%d must be a multiple of 128", K);
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(y, 128, "y");
  return W4A16_OK;
}

extern "C" int w4a16_gemv(const uint16_t* x, int M, int K, const uint32_t* qweight, const uint16_t* scales,
                          int N, const uint16_t* bias, const uint16_t* residual, uint16_t* y,
                          w4a16_stream_t stream) {
  int rc = check_gemv_common(x, M, K, N, y);
  if (rc) return rc;
  W4_CHECK_ARG(qweight && scales, "w4a16_gemv: qweight and scales must be non-null");
  W4_CHECK_ALIGN(qweight, 128, "qweight");
  W4_CHECK_ALIGN(scales, 128, "scales");
  W4_CHECK_ALIGN(bias, 128, "bias");
  W4_CHECK_ALIGN(residual, 128, "residual");
  GemvArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.residual = reinterpret_cast<const __half*>(residual);
  a.y = reinterpret_cast<__half*>(y);
  a.seg[0] = {qweight, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(bias), N};
  a.nseg = 1;
  a.M = M;
  a.K = K;
  a.N = N;
  return launch_gemv(a, false, (cudaStream_t)stream);
}

extern "C" int w4a16_gemv_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                                  const uint32_t* qweight, const uint16_t* scales, int N,
                                  const uint16_t* bias, uint16_t* y, w4a16_stream_t stream) {
  int rc = check_gemv_common(x, M, K, N, y);
  if (rc) return rc;
  W4_CHECK_ARG(qweight && scales && gamma, "w4a16_gemv_rmsnorm: qweight, scales, gamma must be non-null");
  W4_CHECK_ARG(eps >= 0.f, "w4a16_gemv_rmsnorm: eps must be >= 0");
  W4_CHECK_ALIGN(qweight, 128, "qweight");
  W4_CHECK_ALIGN(scales, 128, "scales");
  W4_CHECK_ALIGN(gamma, 128, "gamma");
  W4_CHECK_ALIGN(bias, 128, "bias");
  GemvArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.gamma = reinterpret_cast<const __half*>(gamma);
  a.eps = eps;
  a.y = reinterpret_cast<__half*>(y);
  a.seg[0] = {qweight, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(bias), N};
  a.nseg = 1;
  a.M = M;
  a.K = K;
  a.N = N;
  return launch_gemv(a, false, (cudaStream_t)stream);
}

extern "C" int w4a16_gemv_silu_mul(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                                   const uint32_t* qweight_gate, const uint16_t* scales_gate,
                                   const uint32_t* qweight_up, const uint16_t* scales_up, int N, uint16_t* y,
                                   w4a16_stream_t stream) {
  int rc = check_gemv_common(x, M, K, N, y);
  if (rc) return rc;
  W4_CHECK_ARG(qweight_gate && scales_gate && qweight_up && scales_up,
               "w4a16_gemv_silu_mul: weights and scales must be non-null");
  W4_CHECK_ARG(eps >= 0.f, "w4a16_gemv_silu_mul: eps must be >= 0");
  W4_CHECK_ALIGN(qweight_gate, 128, "qweight_gate");
  W4_CHECK_ALIGN(scales_gate, 128, "scales_gate");
  W4_CHECK_ALIGN(qweight_up, 128, "qweight_up");
  W4_CHECK_ALIGN(scales_up, 128, "scales_up");
  W4_CHECK_ALIGN(gamma, 128, "gamma");
  GemvArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.gamma = reinterpret_cast<const __half*>(gamma);
  a.eps = eps;
  a.y = reinterpret_cast<__half*>(y);
  a.seg[0] = {qweight_gate, reinterpret_cast<const __half*>(scales_gate), nullptr, N};
  a.seg[1] = {qweight_up, reinterpret_cast<const __half*>(scales_up), nullptr, N};
  a.nseg = 2;
  a.M = M;
  a.K = K;
  a.N = N;
  return launch_gemv(a, true, (cudaStream_t)stream);
}
