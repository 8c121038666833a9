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
// Dequant trick, per packed word w (nibbles u0..u7, u = q + 8).  Nibbles i
// and i + 4 sit 16 bits apart, so one LOP3 drops a pair into the two halves
// of a half2 whose exponent field is that of 1024:
//   (w        & 0x000F000F) | 0x64006400 = half2{1024 + u0,    1024 + u4}
//   (w        & 0x00F000F0) | 0x64006400 = half2{1024 + 16 u1, 1024 + 16 u5}
//   ((w >> 8) & 0x000F000F) | 0x64006400 = half2{1024 + u2,    1024 + u6}
//   ((w >> 8) & 0x00F000F0) | 0x64006400 = half2{1024 + 16 u3, 1024 + 16 u7}
// all exact.  The activations are staged once per CTA in shared memory in the
// matching order, and mixed-precision fp16 x fp16 -> fp32 FMAs (exact
// products) give over a 32-weight chunk
//   A = sum_{i even} x_i (1024 + u_i),  B = sum_{i odd} x_i (1024 + 16 u_i),
//   sum_i q_i x_i = A + B/16 - (1032 sum_{i even} x_i + 72 sum_{i odd} x_i),
// with the bracket (one fp32 per chunk, shared by every row) staged beside x.
// The 1024 offset costs about ten bits of the fp32 sums, which leaves the
// chunk sums some 100x more accurate than an fp16 output needs.  That is one
// shift, four LOP3 and eight FMAs per eight weights, with no fp16-pipe work.
//
// Work split: LPR lanes cooperate on one weight row (LPR = 16 when K/32 is a
// multiple of 16, else 8 or 4); a warp covers 32/LPR rows at a time; each
// lane streams 16-byte words with 128-bit non-allocating loads, GEMV_U of
// them in flight, and the row sum is a shuffle reduction over LPR lanes.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "int4_dot.cuh"
#include "kernels.h"

namespace w4 {

constexpr int GEMV_WPB = 8;  // warps per block
constexpr int GEMV_U = 8;    // 16-byte weight loads in flight per lane

// gpre: gamma's groups already in registers (loaded before the dependency
// wait by the caller), or null to load them here.
template <int MT>
__device__ __forceinline__ void stage_activations(const GemvArgs& a, uint4* xs, float* cs, float (*red)[MT],
                                                  float* rscale, const uint4* gpre = nullptr) {
  const int K = a.K, M = a.M, NCH = K >> 5, NG = K >> 3;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarp = nthr >> 5;
  if (a.gamma != nullptr && NG <= STAGE_GMAX * nthr) {
    // one read of x and gamma into registers, sums of squares, one barrier
    uint4 xr[MT][STAGE_GMAX], gr[STAGE_GMAX];
    float ss[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) ss[m] = 0.f;
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      const int g = tid + i * nthr;
      if (g < NG) {
        gr[i] = gpre ? gpre[i] : *reinterpret_cast<const uint4*>(a.gamma + 8 * g);
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < M) xr[m][i] = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + 8 * g);
      }
    }
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      if (tid + i * nthr < NG) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const __half* h = reinterpret_cast<const __half*>(&xr[m][i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float v = __half2float(h[e]);
              ss[m] = fmaf(v, v, ss[m]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float t = warp_sum(ss[m]);
      if (lane == 0) red[warp][m] = t;
    }
    __syncthreads();
    // every warp adds the warps' sums in the same shuffle tree (one shared
    // load per lane instead of nwarp dependent ones per thread)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float t = warp_sum(lane < nwarp ? red[lane][m] : 0.f);
      rscale[m] = 1.0f / sqrtf(t / (float)K + a.eps);  // the same value from every thread
    }
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      const int g = tid + i * nthr;
      if (i * nthr + warp * 32 >= NG) break;  // warp-uniform: no group of this warp is left
      const bool active = g < NG;
      const __half* gh = reinterpret_cast<const __half*>(&gr[i]);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          __half h[8];
          if (active) {
            const __half* xh = reinterpret_cast<const __half*>(&xr[m][i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(__half2float(xh[e]) * rscale[m] * __half2float(gh[e]));
          }
          stage_group(xs, cs, NCH, m, g, h, active);
        }
      }
    }
  } else {
    // plain copy (or, past the register budget, RMSNorm in two reads): one
    // 32-element chunk per thread and step, its four loads in flight together
    if (a.gamma != nullptr) {
      for (int m = 0; m < M; ++m) {
        float ss = 0.f;
        for (int g = tid; g < NG; g += nthr) {
          const uint4 raw = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + 8 * g);
          const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float v = __half2float(h[e]);
            ss = fmaf(v, v, ss);
          }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp][m] = ss;
      }
      __syncthreads();
      for (int m = 0; m < M; ++m) {
        float t = 0.f;
        for (int w = 0; w < nwarp; ++w) t += red[w][m];
        rscale[m] = 1.0f / sqrtf(t / (float)K + a.eps);
      }
    }
    for (int idx = tid; idx < M * NCH; idx += nthr) {
      const int m = idx / NCH, j = idx - m * NCH;
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)m * K + 32 * j);
      uint4 raw[4];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) raw[wi] = src[wi];
      float se = 0.f, so = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        __half h[8];
        *reinterpret_cast<uint4*>(h) = raw[wi];
        if (a.gamma != nullptr) {
          const uint4 graw = *reinterpret_cast<const uint4*>(a.gamma + 32 * j + 8 * wi);
          const __half* gh = reinterpret_cast<const __half*>(&graw);
#pragma unroll
          for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(__half2float(h[e]) * rscale[m] * __half2float(gh[e]));
        }
        uint4 o;
        o.x = pack_h2(h[0], h[4]);
        o.y = pack_h2(h[1], h[5]);
        o.z = pack_h2(h[2], h[6]);
        o.w = pack_h2(h[3], h[7]);
        xs[(size_t)(m * 4 + wi) * NCH + j] = o;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          se += __half2float(h[e]);
          so += __half2float(h[e + 1]);
        }
      }
      cs[(size_t)m * NCH + j] = 1032.0f * se + 72.0f * so;
    }
  }
  __syncthreads();
}

template <int LPR, int MT, bool SILU>
__global__ void __launch_bounds__(GEMV_WPB * 32) w4pg_matvec_int4(const __grid_constant__ GemvArgs a) {
  constexpr int RPW = 32 / LPR;               // row slots per warp
  constexpr int RPT = SILU ? RPW / 2 : RPW;   // output rows per warp task
  extern __shared__ uint4 smem[];
  const int K = a.K, M = a.M;
  const int NCH = K >> 5;      // 32-weight chunks per row
  const int NIT = NCH / LPR;   // chunks per lane per row
  uint4* xs = smem;                                                   // [MT][4][NCH]
  float* cs = reinterpret_cast<float*>(smem + (size_t)MT * 4 * NCH);  // [MT][NCH]
  __shared__ float red[GEMV_WPB][MT];
  __shared__ float rscale[MT];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = lane / LPR, lr = lane % LPR;
  const int ntask = (a.N + RPT - 1) / RPT;
  const int nwarps = gridDim.x * GEMV_WPB;
  W4_TRACE_SCOPE(a.tag);

  // Weights do not depend on the previous kernel: issue this warp's first
  // batch of weight loads before waiting for it.

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

  pdl_wait_then_trigger();  // x (and residual) come from the previous kernel
  W4_TRACE_WAITED();

  stage_activations<MT>(a, xs, cs, red, rscale);

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
                float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) word_dot(p, wv[wi], xs[(size_t)(m * 4 + wi) * NCH + j]);
                acc[m] = fmaf(chunk_sum(p, cs[(size_t)m * NCH + j]), s, acc[m]);
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
// Fast path for K a multiple of 512 known at compile time (the model's
// K = 3584 and 18944).  16 lanes per weight row.  Each lane streams the
// 16-byte chunks it will use into its own slots of a shared-memory ring with
// cp.async (a lane only ever reads what it copied, so no barrier is needed),
// one batch of GEMV_RU chunks ahead of the batch it computes; bytes in
// flight therefore cost shared memory, not registers.  Task shapes:
//   KS = 1: each half-warp owns R rows (non-SiLU task = 2R rows; SiLU task =
//           R output rows, half-warp 0 on the gate rows, 1 on the up rows);
//   KS = 2: both half-warps work on the same R rows and split K (long K).
// All strides are compile-time immediates.
// ---------------------------------------------------------------------------
// RU: chunks per lane per batch (R rows x U chunks).  K = 3584 uses 8 so a
// whole row (7 chunks per lane) is in flight before the dependency wait;
// the long-K down projection uses 4 to fit more CTAs per SM.
template <int NCH, int R, int KS, int MT, bool SILU, int RU, int WPB, int NS>
__global__ void __launch_bounds__(WPB * 32, 32 / WPB) w4pg_matvec_int4_ring(const __grid_constant__ GemvArgs a) {
  constexpr int LPR = 16, U = RU / R;
  constexpr int K = NCH * 32;
  constexpr int NIT = NCH / LPR;                 // chunks per lane when one half-warp covers K
  constexpr int NIT_L = (NIT + KS - 1) / KS;     // this lane's share (upper bound)
  constexpr int NB = (NIT_L + U - 1) / U;        // batches per task
  // batches per unrolled round: a multiple of NB and of the NS ring slots,
  // so every slot index is a compile-time constant
  constexpr int NBT = lcm_c(NB, NS);
  constexpr int WROW = K / 8;
  constexpr int SROW = K / 128;
  constexpr int RPT = SILU ? R : (KS == 2 ? R : 2 * R);
  constexpr int NT = WPB * 32;
  static_assert(RU % R == 0, "R must divide RU");
  static_assert(!(SILU && KS == 2), "SiLU pairs gate and up across half-warps");
  static_assert(NCH % LPR == 0, "every lane takes the same number of chunks");
  extern __shared__ uint4 smem[];
  uint4* xs = smem;                                          // [MT][4][NCH]
  uint4* ring = smem + MT * 4 * NCH;                          // [NS][RU][NT], each lane its own column
  float* cs = reinterpret_cast<float*>(ring + NS * RU * NT);  // [MT][NCH]
  __shared__ float red[WPB][MT];
  __shared__ float rscale[MT];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int hw = lane >> 4, lr = lane & 15;
  const int M = a.M;
  const int ntask = (a.N + RPT - 1) / RPT;
  const int nwarps = gridDim.x * WPB;
  // chunk index of (batch b, word u) for this lane: j = jl + JSTEP * (b * U + u)
  constexpr int JSTEP = LPR * KS;
  const int jl = lr + (KS == 2 ? LPR * hw : 0);
  auto it_ok = [&](int i) { return KS == 2 ? (2 * i + hw < NIT) : (i < NIT); };
  W4_TRACE_SCOPE(a.tag);

  // first output row of this lane's rows for task t, and the weight-row base
  auto rows_of = [&](int t, int& out0, const uint32_t*& q, const __half*& sp, const __half*& bp) {
    if (SILU) {
      out0 = t * RPT;
      const int r = max(min(out0, a.N - R), 0);
      q = a.seg[hw].qw + (size_t)r * WROW;
      sp = a.seg[hw].s + (size_t)r * SROW;
      bp = nullptr;
    } else {
      out0 = KS == 2 ? t * RPT : t * RPT + hw * R;
      int r = max(min(out0, a.N - R), 0);
      int si = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (si < a.nseg - 1 && r >= a.seg[si].rows) { r -= a.seg[si].rows; ++si; }
      q = a.seg[si].qw + (size_t)r * WROW;
      sp = a.seg[si].s + (size_t)r * SROW;
      bp = a.seg[si].bias ? a.seg[si].bias + r : nullptr;
    }
  };

  // issue side: the task whose batches are being loaded
  int i_task = blockIdx.x * WPB + warp, i_out0;
  const uint32_t* i_q = nullptr;
  const __half *i_s = nullptr, *i_bias;
  if (i_task < ntask) {
    rows_of(i_task, i_out0, i_q, i_s, i_bias);
    i_q += 4 * jl;         // this lane's first 16-byte word
    i_s += jl >> 2;
  }
  __half sc[NS][RU];
  // batch b of the issue task into ring slot `slot` (b, slot compile-time once unrolled)
  auto issue = [&](const int slot, const int b) {
    if (i_task < ntask) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b * U + u;
        if (i < NIT_L && it_ok(i)) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            cp_async16(&ring[(slot * RU + r * U + u) * NT + tid], i_q + r * WROW + 4 * JSTEP * i);
            sc[slot][r * U + u] = i_s[r * SROW + (JSTEP * i) / 4];
          }
        }
      }
    }
    cp_async_commit();
  };
  auto next_issue_task = [&]() {
    i_task += nwarps;
    if (i_task < ntask) {
      rows_of(i_task, i_out0, i_q, i_s, i_bias);
      i_q += 4 * jl;
      i_s += jl >> 2;
    }
  };

  // RMSNorm weight first: like the weights it does not depend on the
  // previous kernel, and it is rarely still in L2 when its layer comes round
  uint4 gpre[STAGE_GMAX];
  const bool gp = a.gamma != nullptr && (K >> 3) <= STAGE_GMAX * NT;
  if (gp) {
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      const int g = tid + i * NT;
      if (g < (K >> 3)) gpre[i] = *reinterpret_cast<const uint4*>(a.gamma + 8 * g);
    }
  }
  // the first NS - 1 batches: weights do not depend on the previous kernel
#pragma unroll
  for (int q0 = 0; q0 < NS - 1; ++q0) {
    if (q0 > 0 && q0 % NB == 0) next_issue_task();
    issue(q0, q0 % NB);
  }
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  stage_activations<MT>(a, xs, cs, red, rscale, gp ? gpre : nullptr);
  W4_TRACE_MARK(0);

  // compute side
  int c_task = blockIdx.x * WPB + warp, c_out0 = 0;
  const uint32_t* c_q;
  const __half *c_s, *c_bias = nullptr;
  if (c_task < ntask) rows_of(c_task, c_out0, c_q, c_s, c_bias);
  const uint4* xl = xs + jl;                               // this lane's chunk column of x
  const float* csl = cs + jl;
  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

  auto compute = [&](const int slot, const int b) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = b * U + u;
      if (i < NIT_L && it_ok(i)) {
        const int jo = JSTEP * i;  // compile-time chunk offset
        uint4 wv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) wv[r] = ring[(slot * RU + r * U + u) * NT + tid];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const uint4* xc = xl + (size_t)(m * 4) * NCH + jo;
            float p[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) p[r][0] = p[r][1] = p[r][2] = p[r][3] = 0.f;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              const uint4 xv = xc[wi * NCH];
#pragma unroll
              for (int r = 0; r < R; ++r) word_dot(p[r], (&wv[r].x)[wi], xv);
            }
            const float c = csl[(size_t)m * NCH + jo];
#pragma unroll
            for (int r = 0; r < R; ++r)
              acc[r][m] = fmaf(chunk_sum(p[r], c), __half2float(sc[slot][r * U + u]), acc[r][m]);
          }
        }
      }
    }
  };
  // task complete: reduce over the half-warp (and across half-warps for KS = 2), write
  auto finish = [&]() {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int o = (KS == 2 ? 16 : 8); o > 0; o >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);
      }
    if (SILU) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float other = __shfl_xor_sync(0xffffffffu, acc[r][m], 16);
          const int row = c_out0 + r;
          if (m < M && hw == 0 && lr == 0 && row < a.N) {
            const float g = __half2float(__float2half_rn(acc[r][m]));
            const float uu = __half2float(__float2half_rn(other));
            a.y[(size_t)m * a.N + row] = __float2half_rn(g / (1.0f + expf(-g)) * uu);
          }
        }
    } else if (lr == 0 && (KS == 1 || hw == 0)) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = c_out0 + r;
        if (row < a.N) {
          const float bv = c_bias ? __half2float(c_bias[r]) : 0.f;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m < M) {
              float v = acc[r][m] + bv;
              if (a.residual) v += __half2float(a.residual[(size_t)m * a.N + row]);
              a.y[(size_t)m * a.N + row] = __float2half_rn(v);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
    c_task += nwarps;
    if (c_task < ntask) rows_of(c_task, c_out0, c_q, c_s, c_bias);
  };

  // rounds of NBT batches; the issue side runs NS - 1 batches ahead
  while (c_task < ntask) {
#pragma unroll
    for (int qq = 0; qq < NBT; ++qq) {
      const int b = qq % NB, bn = (qq + NS - 1) % NB;  // computed batch; batch issued NS - 1 ahead
      if (bn == 0) next_issue_task();
      issue((qq + NS - 1) % NS, bn);
      cp_async_wait<NS - 1>();  // this lane's batch in slot qq % NS has landed
      compute(qq % NS, b);
      if (b == NB - 1) {
        W4_TRACE_MARK(1);
        finish();
        if (c_task >= ntask) break;
      }
    }
  }
  cp_async_wait<0>();
}
template <int NCH, int R, int KS, int MT, bool SILU, int RU, int WPB = GEMV_WPB, int NS = 2>
static int launch_fast(const GemvArgs& a, cudaStream_t s) {
  auto kern = w4pg_matvec_int4_ring<NCH, R, KS, MT, SILU, RU, WPB, NS>;
  const size_t smem = (size_t)MT * a.K * 2 + (size_t)NS * RU * WPB * 32 * 16 + (size_t)MT * (a.K / 32) * 4;
  static PerDeviceOnce once;
  once_per_device(once, [&] { cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024); });
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, WPB * 32, smem) != cudaSuccess || bps < 1)
    bps = 1;
  constexpr int RPT = SILU ? R : (KS == 2 ? R : 2 * R);
  const int ntask = (a.N + RPT - 1) / RPT;
  int blocks = std::min((ntask + WPB - 1) / WPB, bps * num_sms());
  blocks = std::max(blocks, 1);
  cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(WPB * 32), smem, s, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

template <int MT, bool SILU>
static int dispatch_fast(const GemvArgs& a, cudaStream_t s, bool* used) {
  *used = true;
  if (SILU) {
    // one 32-warp CTA per SM: x staged once per SM instead of four times
    // (14.9 us per launch against 15.8 for four 8-warp CTAs)
    if (a.K == 3584) return launch_fast<112, 2, 1, MT, true, 4, 32, 2>(a, s);
  } else {
    if (a.K == 3584) return launch_fast<112, 1, 1, MT, false, 8>(a, s);
    // one 24-warp CTA per SM (ring and x fit once, not three times): 3584
    // rows on 3648 warps, one task each (9.4 us per launch against 11.1 for
    // three 8-warp CTAs; 11.4 for 32 warps)
    if (a.K == 18944) return launch_fast<592, 1, 2, MT, false, 4, 24, 2>(a, s);
  }
  *used = false;
  return W4A16_OK;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int LPR, int MT, bool SILU>
static int launch_one(const GemvArgs& a, cudaStream_t s) {
  auto kern = w4pg_matvec_int4<LPR, MT, SILU>;
  const size_t smem = (size_t)MT * a.K * 2 + (size_t)MT * (a.K / 32) * 4;
  static PerDeviceOnce once;
  once_per_device(once, [&] { cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 110 * 1024); });
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, GEMV_WPB * 32, smem) != cudaSuccess || bps < 1)
    bps = 1;
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
  if (a.M <= 4 && !gemv_cuda_core_supported(a.M, a.K) && gemv_cuda_core_supported(1, a.K)) {
    // up to four rows whose activations do not fit the shared-memory budget
    // together: launches of as many rows as fit (each streams the weights;
    // still far ahead of a tensor-core GEMM with no workspace to split K)
    const int per = 49152 / a.K;
    for (int r0 = 0; r0 < a.M; r0 += per) {
      GemvArgs c = a;
      c.M = std::min(per, a.M - r0);
      c.x = a.x + (size_t)r0 * a.K;
      c.residual = a.residual ? a.residual + (size_t)r0 * a.N : nullptr;
      c.y = a.y + (size_t)r0 * a.N;
      const int rc = launch_gemv(c, silu, s);
      if (rc) return rc;
    }
    return W4A16_OK;
  }
  if (!gemv_cuda_core_supported(a.M, a.K)) {
    // a real batch: the tensor-core GEMM (no RMSNorm prologue there)
    if (a.M <= 32 && a.gamma == nullptr) {
      TcArgs t = {};
      t.x = a.x;
      t.residual = a.residual;
      t.y = a.y;
      for (int i = 0; i < 3; ++i) t.seg[i] = a.seg[i];
      t.nseg = a.nseg;
      t.M = a.M;
      t.K = a.K;
      t.N = a.N;
      t.ldy = a.N;
      t.ksplit = 1;
      t.tag = a.tag;
      return launch_gemm_tc(t, true, silu, s);
    }
    return set_error(W4A16_ERR_SHAPE, "gemv: M=%d K=%d outside the built paths (M<=32; fused RMSNorm only for M<=4)",
                     a.M, a.K);
  }
  // the fast path moves two rows per half-warp: every segment (and N) even
  bool even_rows = a.N >= 2 && a.N % 2 == 0;
  for (int i = 0; i < a.nseg; ++i) even_rows = even_rows && (a.seg[i].rows % 2 == 0);
  if (even_rows) {
    bool used = false;
    int rc = W4A16_OK;
    if (silu) {
      rc = a.M == 1 ? dispatch_fast<1, true>(a, s, &used)
                    : (a.M == 2 ? dispatch_fast<2, true>(a, s, &used) : dispatch_fast<4, true>(a, s, &used));
    } else {
      rc = a.M == 1 ? dispatch_fast<1, false>(a, s, &used)
                    : (a.M == 2 ? dispatch_fast<2, false>(a, s, &used) : dispatch_fast<4, false>(a, s, &used));
    }
    if (used) return rc;
  }
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
