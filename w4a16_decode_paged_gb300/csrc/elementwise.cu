// elementwise.cu -- RMSNorm, embedding gather, and the FP16 lm_head GEMV with
// a fused argmax.
//
// The aikraft.ru article "How to build your own LLM runtime from scratch"
// ("Архитектурные решения и оптимизации") keeps RMSNorm and lm_head in FP16;
// the argmax is the greedy decode rule.  All sums here are fp32.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace w4 {

// ---------------------------------------------------------------------------
// RMSNorm: one CTA per row.  Rows of up to RN_THREADS * RN_HELD * 8 = 8192
// values (the model's hidden size is 3584) stay in registers between the sum
// of squares and the scaling, so x is read once, and gamma, which does not depend on the
// previous kernel, is loaded before the dependency wait.  Longer rows are
// read twice.  Either way each thread sums its words in the same order.
// ---------------------------------------------------------------------------
constexpr int RN_THREADS = 256;
constexpr int RN_HELD = 4;  // 16-byte words of the row each thread holds

__global__ void __launch_bounds__(RN_THREADS) w4pg_rmsnorm(const __half* __restrict__ x,
                                                             const __half* __restrict__ gamma, __half* y, int H,
                                                             float eps, int tag) {
  __shared__ float red[RN_THREADS / 32];
  __shared__ float rs;
  W4_TRACE_SCOPE(tag);
  const int m = blockIdx.x;
  const int nw = H / 8;  // 16-byte words per row
  const bool held = nw <= RN_THREADS * RN_HELD;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)m * H);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)m * H);
  uint4 xv[RN_HELD], gv[RN_HELD];
  if (held) {
#pragma unroll
    for (int i = 0; i < RN_HELD; ++i) {
      const int w = threadIdx.x + i * RN_THREADS;
      if (w < nw) gv[i] = gr[w];
    }
  }
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  auto sumsq = [](const uint4& raw, float ss) {
    const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v = __half2float(h[i]);
      ss = fmaf(v, v, ss);
    }
    return ss;
  };
  auto scaled = [](uint4 raw, const uint4& graw, float r) {
    __half* h = reinterpret_cast<__half*>(&raw);
    const __half* g = reinterpret_cast<const __half*>(&graw);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __float2half_rn(__half2float(h[i]) * r * __half2float(g[i]));
    return raw;
  };
  float ss = 0.f;
  if (held) {
#pragma unroll
    for (int i = 0; i < RN_HELD; ++i) {
      const int w = threadIdx.x + i * RN_THREADS;
      if (w < nw) xv[i] = xr[w];
    }
#pragma unroll
    for (int i = 0; i < RN_HELD; ++i)
      if (threadIdx.x + i * RN_THREADS < nw) ss = sumsq(xv[i], ss);
  } else {
    for (int w = threadIdx.x; w < nw; w += RN_THREADS) ss = sumsq(xr[w], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < RN_THREADS / 32; ++w) t += red[w];
    rs = 1.0f / sqrtf(t / (float)H + eps);
  }
  __syncthreads();
  const float r = rs;
  if (held) {
#pragma unroll
    for (int i = 0; i < RN_HELD; ++i) {
      const int w = threadIdx.x + i * RN_THREADS;
      if (w < nw) yr[w] = scaled(xv[i], gv[i], r);
    }
  } else {
    for (int w = threadIdx.x; w < nw; w += RN_THREADS) yr[w] = scaled(xr[w], gr[w], r);
  }
}

int launch_rmsnorm(const __half* x, const __half* gamma, __half* y, int M, int H, float eps, cudaStream_t s,
                   int tag) {
  cudaError_t e = launch_pdl(w4pg_rmsnorm, dim3(M), dim3(RN_THREADS), 0, s, x, gamma, y, H, eps, tag);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "rmsnorm launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

// ---------------------------------------------------------------------------
// Embedding gather (+ optional device-side context length advance).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) w4pg_embedding(const __half* __restrict__ embed, int vocab, int H,
                                                        const int32_t* tokens, __half* x, int32_t* err_flag,
                                                        int32_t* lens, int max_len, int tag) {
  W4_TRACE_SCOPE(tag);
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  const int b = blockIdx.x;
  const int tok = tokens[b];
  const bool ok = tok >= 0 && tok < vocab;
  if (!ok && threadIdx.x == 0 && err_flag) atomicOr(err_flag, 1);
  const uint4* src = reinterpret_cast<const uint4*>(embed + (size_t)(ok ? tok : 0) * H);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)b * H);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
  if (lens && threadIdx.x == 0) {
    // the model's buffers and attention partitions cover max_len tokens: a
    // longer context is reported, not silently truncated
    const int n = lens[b] + 1;
    if (n > max_len && err_flag) atomicOr(err_flag, 1);
    lens[b] = n;
  }
}

int launch_embedding(const __half* embed, int vocab, int H, const int32_t* tokens, int B, __half* x,
                     int32_t* err_flag, int32_t* lens_to_advance, int max_len, cudaStream_t s, int tag) {
  cudaError_t e = launch_pdl(w4pg_embedding, dim3(B), dim3(256), 0, s, embed, vocab, H, tokens, x, err_flag,
                             lens_to_advance, max_len, tag);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "embedding launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

// ---------------------------------------------------------------------------
// Prefill bookkeeping: the T prompt tokens of one sequence run as T rows
// whose lengths are len0 + 1 .. len0 + T over copies of the sequence's
// block-table row (token t attends to positions <= len0 + t); afterwards the
// sequence's length advances by T.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) w4pg_prefill_rows(const int32_t* __restrict__ bt_row, int max_blocks,
                                                         const int32_t* __restrict__ len0, int T,
                                                         int32_t* __restrict__ bt_rep, int32_t* __restrict__ lens) {
  pdl_wait_then_trigger();
  const int l0 = *len0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * max_blocks; i += gridDim.x * blockDim.x) {
    const int t = i / max_blocks, j = i - t * max_blocks;
    bt_rep[i] = bt_row[j];
    if (j == 0) lens[t] = l0 + t + 1;
  }
}
__global__ void __launch_bounds__(32) w4pg_advance_len(int32_t* len, int T, int max_len, int32_t* err_flag) {
  pdl_wait_then_trigger();
  if (threadIdx.x == 0) {
    const int n = *len + T;
    if (n > max_len && err_flag) atomicOr(err_flag, 1);
    *len = n;
  }
}
int launch_prefill_rows(const int32_t* bt_row, int max_blocks, const int32_t* len0, int T, int32_t* bt_rep,
                        int32_t* lens, cudaStream_t s) {
  const int blocks = std::max(1, std::min(1024, (T * max_blocks + 255) / 256));
  cudaError_t e = launch_pdl(w4pg_prefill_rows, dim3(blocks), dim3(256), 0, s, bt_row, max_blocks, len0, T, bt_rep,
                             lens);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "prefill rows launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}
int launch_advance_len(int32_t* len, int T, int max_len, int32_t* err_flag, cudaStream_t s) {
  cudaError_t e = launch_pdl(w4pg_advance_len, dim3(1), dim3(32), 0, s, len, T, max_len, err_flag);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "advance length launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

// ---------------------------------------------------------------------------
// lm_head (fp16 weight [vocab][H]) GEMV + argmax, B <= 4 sequences.
// A warp owns a row at a time (lanes stride the row in 16-byte chunks, two
// rows in flight); x (optionally RMS-normalised) sits in shared memory.
// Each CTA reduces its best (logit, index) per sequence into a packed 64-bit
// key; the last CTA to finish (atomic ticket) reduces the CTA keys.
// ---------------------------------------------------------------------------
constexpr int LM_WPB = 8;
constexpr int LM_MAXB = 4;
constexpr int LM_MAX_BLOCKS = 4096;

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  uint32_t bits = __float_as_uint(v);
  uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__global__ void __launch_bounds__(LM_WPB * 32) w4pg_lm_head_argmax(const __grid_constant__ LmHeadArgs a) {
  extern __shared__ uint4 xsm[];  // [B][H/8]
  __shared__ unsigned long long wbest[LM_WPB][LM_MAXB];
  __shared__ float red[LM_WPB];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H, NC = H / 8;
  W4_TRACE_SCOPE(a.tag);
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();

  // stage x (RMS-normalised when gamma is given)
  for (int b = 0; b < a.B; ++b) {
    float r = 1.f;
    if (a.gamma) {
      float ss = 0.f;
      for (int c = threadIdx.x; c < NC; c += blockDim.x) {
        uint4 raw = *reinterpret_cast<const uint4*>(a.x + (size_t)b * H + 8 * c);
        const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v = __half2float(h[i]);
          ss = fmaf(v, v, ss);
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float t = 0.f;
      for (int w = 0; w < LM_WPB; ++w) t += red[w];
      r = 1.0f / sqrtf(t / (float)H + a.eps);
      __syncthreads();
    }
    for (int c = threadIdx.x; c < NC; c += blockDim.x) {
      uint4 raw = *reinterpret_cast<const uint4*>(a.x + (size_t)b * H + 8 * c);
      if (a.gamma) {
        uint4 graw = *reinterpret_cast<const uint4*>(a.gamma + 8 * c);
        __half* h = reinterpret_cast<__half*>(&raw);
        const __half* g = reinterpret_cast<const __half*>(&graw);
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __float2half_rn(__half2float(h[i]) * r * __half2float(g[i]));
      }
      xsm[b * NC + c] = raw;
    }
  }
  __syncthreads();

  float best[LM_MAXB];
  int besti[LM_MAXB];
#pragma unroll
  for (int b = 0; b < LM_MAXB; ++b) {
    best[b] = -INFINITY;
    besti[b] = 0x7fffffff;
  }
  const int nwarps = gridDim.x * LM_WPB;
  const int per_lane = (NC + 31) / 32;
  for (int row0 = blockIdx.x * LM_WPB + warp; row0 < a.vocab; row0 += 2 * nwarps) {
    const int row1 = row0 + nwarps;
    const bool has1 = row1 < a.vocab;
    const uint4* w0 = reinterpret_cast<const uint4*>(a.w + (size_t)row0 * H);
    const uint4* w1 = reinterpret_cast<const uint4*>(a.w + (size_t)(has1 ? row1 : row0) * H);
    float acc0[LM_MAXB], acc1[LM_MAXB];
#pragma unroll
    for (int b = 0; b < LM_MAXB; ++b) acc0[b] = acc1[b] = 0.f;
    for (int i0 = 0; i0 < per_lane; i0 += 8) {
      uint4 r0[8], r1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = lane + 32 * (i0 + u);
        if (i0 + u < per_lane && c < NC) {
          r0[u] = ldg_stream(w0 + c);
          r1[u] = ldg_stream(w1 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = lane + 32 * (i0 + u);
        if (i0 + u < per_lane && c < NC) {
#pragma unroll
          for (int b = 0; b < LM_MAXB; ++b) {
            if (b < a.B) {
              const uint4 xv = xsm[b * NC + c];
              fma2_f16_f32(acc0[b], r0[u].x, xv.x);
              fma2_f16_f32(acc0[b], r0[u].y, xv.y);
              fma2_f16_f32(acc0[b], r0[u].z, xv.z);
              fma2_f16_f32(acc0[b], r0[u].w, xv.w);
              fma2_f16_f32(acc1[b], r1[u].x, xv.x);
              fma2_f16_f32(acc1[b], r1[u].y, xv.y);
              fma2_f16_f32(acc1[b], r1[u].z, xv.z);
              fma2_f16_f32(acc1[b], r1[u].w, xv.w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < LM_MAXB; ++b) {
      if (b < a.B) {
        const float v0 = warp_sum(acc0[b]);
        const float v1 = warp_sum(acc1[b]);
        if (v0 > best[b]) { best[b] = v0; besti[b] = row0; }
        if (has1 && v1 > best[b]) { best[b] = v1; besti[b] = row1; }
        if (a.logits && lane == 0) {
          a.logits[(size_t)b * a.vocab + row0] = __float2half_rn(v0);
          if (has1) a.logits[(size_t)b * a.vocab + row1] = __float2half_rn(v1);
        }
      }
    }
  }
  // NOTE: within a warp rows are visited in increasing order, so '>' keeps
  // the lowest index among equal values; keys break ties across warps/CTAs.
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < LM_MAXB; ++b)
      wbest[warp][b] = (besti[b] == 0x7fffffff) ? 0ull : argmax_key(best[b], besti[b]);
  }
  __syncthreads();
  if (threadIdx.x < a.B) {
    unsigned long long k = 0;
    for (int w = 0; w < LM_WPB; ++w) k = max(k, wbest[w][threadIdx.x]);
    a.partial[(size_t)threadIdx.x * LM_MAX_BLOCKS + blockIdx.x] = k;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counters, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = warp; b < a.B; b += LM_WPB) {
    unsigned long long k = 0;
    for (int i = lane; i < (int)gridDim.x; i += 32) k = max(k, __ldcg(&a.partial[(size_t)b * LM_MAX_BLOCKS + i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
    if (lane == 0) a.tokens_out[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
  }
  if (threadIdx.x == 0) *a.counters = 0u;
}

size_t lm_head_workspace_bytes(int B, int vocab) {
  (void)B;  // one fixed block: partial keys of up to LM_MAXB rows x LM_MAX_BLOCKS CTAs + counters
  (void)vocab;
  return (size_t)LM_MAXB * LM_MAX_BLOCKS * 8 + 256;
}

int launch_lm_head_argmax(const LmHeadArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)a.B * a.H * 2;
  static PerDeviceOnce once;
  once_per_device(once,
                  [] { cudaFuncSetAttribute(w4pg_lm_head_argmax, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024); });
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, w4pg_lm_head_argmax, LM_WPB * 32, smem) != cudaSuccess ||
      bps < 1)
    bps = 1;
  int blocks = std::min((a.vocab + 2 * LM_WPB - 1) / (2 * LM_WPB), bps * num_sms());
  blocks = std::max(1, std::min(blocks, LM_MAX_BLOCKS));
  cudaError_t e = launch_pdl(w4pg_lm_head_argmax, dim3(blocks), dim3(LM_WPB * 32), smem, s, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "lm_head launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

}  // namespace w4

using namespace w4;

extern "C" int rmsnorm(const uint16_t* x, const uint16_t* gamma, uint16_t* y, int M, int H, float eps,
                       w4a16_stream_t stream) {
  W4_CHECK_ARG(x && gamma && y, "rmsnorm: null pointer");
  W4_CHECK_ARG(M >= 1 && H >= 1, "rmsnorm: sizes must be positive");
  W4_CHECK_SHAPE(H % 8 == 0, "rmsnorm: H=%d must be a multiple of 8", H);
  W4_CHECK_ARG(eps >= 0.f, "rmsnorm: eps must be >= 0");
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(gamma, 128, "gamma");
  W4_CHECK_ALIGN(y, 128, "y");
  return launch_rmsnorm(reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(gamma),
                        reinterpret_cast<__half*>(y), M, H, eps, (cudaStream_t)stream);
}

extern "C" int embedding_gather(const uint16_t* embed, int vocab, int H, const int32_t* tokens, int B, uint16_t* x,
                                int32_t* err_flag, w4a16_stream_t stream) {
  W4_CHECK_ARG(embed && tokens && x, "embedding_gather: null pointer");
  W4_CHECK_ARG(vocab >= 1 && H >= 1 && B >= 1, "embedding_gather: sizes must be positive");
  W4_CHECK_SHAPE(H % 8 == 0, "embedding_gather: H %% 8 != 0");
  W4_CHECK_ALIGN(embed, 128, "embed");
  W4_CHECK_ALIGN(x, 128, "x");
  return launch_embedding(reinterpret_cast<const __half*>(embed), vocab, H, tokens, B, reinterpret_cast<__half*>(x),
                          err_flag, nullptr, 0, (cudaStream_t)stream);
}

extern "C" size_t lm_head_argmax_workspace_size(int B, int vocab) { return lm_head_workspace_bytes(B, vocab); }

extern "C" int lm_head_argmax(const uint16_t* x, int B, int H, const uint16_t* lm_head, int vocab, uint16_t* logits,
                              int32_t* tokens_out, void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  W4_CHECK_ARG(x && lm_head && tokens_out && workspace, "lm_head_argmax: null pointer");
  W4_CHECK_ARG(B >= 1 && H >= 1 && vocab >= 1, "lm_head_argmax: sizes must be positive");
  W4_CHECK_SHAPE(B <= LM_MAXB, "lm_head_argmax: B=%d > %d", B, LM_MAXB);
  W4_CHECK_SHAPE(H % 8 == 0 && H <= 16384, "lm_head_argmax: H=%d", H);
  W4_CHECK_ARG(workspace_bytes >= lm_head_workspace_bytes(B, vocab), "lm_head_argmax: workspace too small");
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(lm_head, 128, "lm_head");
  W4_CHECK_ALIGN(logits, 128, "logits");
  W4_CHECK_ALIGN(workspace, 128, "workspace");
  LmHeadArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.w = reinterpret_cast<const __half*>(lm_head);
  a.logits = reinterpret_cast<__half*>(logits);
  a.tokens_out = tokens_out;
  a.partial = reinterpret_cast<unsigned long long*>(workspace);
  a.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + (size_t)LM_MAXB * LM_MAX_BLOCKS * 8);
  a.B = B;
  a.H = H;
  a.vocab = vocab;
  return launch_lm_head_argmax(a, (cudaStream_t)stream);
}
