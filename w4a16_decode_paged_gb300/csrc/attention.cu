// attention.cu -- paged GQA decode attention with a fused split-K combine,
// and RoPE + KV append.
//
// Paging follows "Building a Custom LLM Inference Runtime on H100"
// (explore.n1n.ai), "2. The KV Cache and PagedAttention" and "Bug 1: The KV
// Cache Indexing 'Off-By-One'": token t of sequence b is slot t % 16 of page
// block_table[b][t / 16].  The pool layout [page][kv_head][16][128] fp16 makes
// each (page, kv head) slice one contiguous 4 KiB run, the unit the aikraft.ru
// article ("Архитектурные решения и оптимизации") aligns to cache lines; here
// one warp copies it into shared memory with 16-byte cp.async copies (512
// contiguous bytes per instruction) into rows padded for ldmatrix.
//
// One CTA handles (sequence b, kv head, partition p) for all G = Hq/Hkv query
// heads that share the kv head (7:1 GQA in the article).  Its eight warps take
// the partition's pages round-robin; each warp owns a private ring of
// 2 or 3 (K, V) page slots, filled with 16-byte cp.async copies (the 32 lanes
// move 512 contiguous bytes per instruction into padded rows), so no warp
// waits on another inside the page loop.  Because the G query heads read
// the same K and V, a page is a small dense contraction and runs on the tensor
// cores with warp-level mma.sync (m16n8k16, fp16 in, fp32 accumulate): the
// scores S[head][token] = Q K^T with the heads as the M rows (padded to 16),
// an fp32 online softmax in registers (exp2, scale folded in), and O += P V
// with the probabilities rounded to fp16 as the A operand (the score
// accumulator layout is the A-fragment layout) and V read with ldmatrix.trans.
// The warps' states are merged in shared memory; partitions are merged through
// distributed shared memory when they fit one thread-block cluster, else their
// (max, sum, weighted V) partials go to the workspace and the last CTA of the
// (b, kv head) group to finish (an atomic ticket, no spin) merges them and
// writes the output.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "attn_core.cuh"
#include "common.cuh"
#include "kernels.h"

namespace w4 {

#ifdef W4A16_TRACE
__device__ TraceRec* g_trace_buf = nullptr;
__device__ unsigned int g_trace_cap = 0;
__device__ unsigned int g_trace_n = 0;
#endif

constexpr int ATT_NW = 8;          // warps per CTA (small grids); large grids use 4 so that
                                   // three CTAs share an SM
constexpr int ATT_MAX_CLUSTER = 8; // partitions merged through distributed shared memory
constexpr int ATT_STAGES = 2;      // page slots per warp (CTA per partition)
constexpr int ATT_STAGES_WP = 3;   // page slots per warp (warp per partition: deeper, the
                                   // warp streams a whole partition alone)
constexpr int att_stages(bool wp) { return wp ? ATT_STAGES_WP : ATT_STAGES; }
constexpr size_t att_slot_bytes(bool kv8) { return kv8 ? (size_t)ATT8_SLOT : (size_t)2 * ATT_SSLICE * 2; }
constexpr size_t att_ring_bytes(int nw, int st, bool kv8) { return (size_t)nw * st * att_slot_bytes(kv8); }
constexpr size_t att_smem(int nw, int st, bool kv8) {
  // the ring is reused for the warps' merge ([NW][8][128 + 2] floats)
  return att_ring_bytes(nw, st, kv8) > (size_t)nw * 8 * (ATT_D + 2) * 4 + 64 * 4 * 4
             ? att_ring_bytes(nw, st, kv8)
             : (size_t)nw * 8 * (ATT_D + 2) * 4 + 64 * 4 * 4;
}

template <int G, bool FUSE, int NW, bool WP, bool KV8>
__global__ void __launch_bounds__(NW * 32) w4pg_paged_attn(const __grid_constant__ AttnArgs a) {
  constexpr int ST = att_stages(WP);      // page slots per warp
  constexpr int SLOT = (int)att_slot_bytes(KV8);
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ __align__(16) float s_q[G][ATT_D];   // this group's q (rotated in the fused variant)
  __shared__ __align__(16) __half s_knew[ATT_D];  // fused: rotated new k and new v (read as uint2)
  __shared__ __align__(16) __half s_vnew[ATT_D];
  __shared__ __align__(16) unsigned char s_new8[2][ATT_D];  // fused, FP8 pages: codes of the new k, v
  __shared__ float s_new8_scale[2];
  __shared__ int s_last;
  // cluster partial table (used in the leader CTA): [partition][head][128 + M, den, pad]
  __shared__ __align__(16) float s_clu[WP ? 4 : ATT_MAX_CLUSTER * G * (ATT_D + 4)];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.z, kvh = blockIdx.y;
  // WP: each warp owns partition p (its pages, its own partial); else the
  // CTA owns partition p and its warps share the pages round-robin
  const int p = WP ? blockIdx.x * NW + warp : blockIdx.x;
  W4_TRACE_SCOPE(a.tag);

  // The fused variant writes the only KV slot that changes in this step
  // itself, and the lengths were written at the start of the step, so it
  // may fetch pages before its predecessor (the q|k|v GEMV) finishes.  The
  // plain variant may be preceded by a kernel that appended to the pools.
  if (!FUSE) {
    pdl_wait_then_trigger();
    W4_TRACE_WAITED();
  }

  // plain variant: this group's q (G x 128 fp16, one 16-byte word per
  // thread) is requested first, so its latency overlaps the page-table reads
  uint4 q_word = make_uint4(0u, 0u, 0u, 0u);
  if (!FUSE && tid < G * ATT_D / 8)
    q_word = __ldcg(reinterpret_cast<const uint4*>(a.q + (size_t)b * a.q_stride + (size_t)kvh * G * ATT_D) + tid);
  const int L = __ldcg(&a.context_lens[b]);
  // the grid covers P partitions: tokens past them would be dropped (and, in
  // the fused variant, the new token never appended), so such a length is
  // reported instead of silently truncated
  if (L > a.P * a.part_tokens && blockIdx.x == 0 && tid == 0 && a.err_flag) atomicOr(a.err_flag, 1);
  const int t_begin = p * a.part_tokens;
  const int t_end = min(L, t_begin + a.part_tokens);
  const int npages = t_end > t_begin ? (t_end - t_begin + ATT_PAGE - 1) / ATT_PAGE : 0;
  const int pg0 = t_begin / ATT_PAGE;
  // tokens of this CTA (decides which CTA appends the new token)
  const int cta_t0 = WP ? blockIdx.x * NW * a.part_tokens : t_begin;
  const int cta_t1 = WP ? min(L, cta_t0 + NW * a.part_tokens) : t_end;
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;

  // this warp's pages: i = warp, warp + NW, ...
  const int my_pages = WP ? npages : (npages > warp ? (npages - warp + NW - 1) / NW : 0);
  unsigned char* myring = smraw + (size_t)warp * ST * SLOT;

  auto page_load = [&](int li) -> int {  // li: index into this warp's page list
    const int gi = pg0 + (WP ? li : warp + li * NW);
    const int pg = (gi < a.max_blocks) ? __ldcg(&bt[gi]) : -1;
    return (pg >= 0 && pg < a.num_pages) ? pg : -1;
  };
  // Each lane loads one of this warp's page ids up front (one L2 round trip
  // for all of them); page_of() broadcasts it.  Must be called warp-wide.
  const int pg_lane = lane < my_pages ? page_load(lane) : -1;
  auto page_of = [&](int li) -> int { return li < 32 ? __shfl_sync(0xffffffffu, pg_lane, li) : page_load(li); };
  // page li of this warp into its ring slot with 16-byte cp.async copies:
  // the 32 lanes move 512 contiguous bytes per instruction, 16 instructions
  // per page (K rows 0-15, then V rows 0-15), into the padded rows.  One
  // commit group per page (empty for a missing page).  Warp-wide.
  auto issue = [&](int li, int pg) {
    unsigned char* dst = myring + (size_t)(li % ST) * SLOT;
    if (pg >= 0 && KV8) {
      // FP8: 2 x 2 KiB of codes (8 x 16 bytes per row) and 2 x 64 bytes of row scales
      const size_t row0 = ((size_t)pg * a.Hkv + kvh) * ATT_PAGE;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;  // [K|V][row][8]
        const int which = c >> 7, row = (c >> 3) & 15, col = c & 7;
        cp_async16(dst + which * ATT8_CODES + row * ATT8_PITCH + col * 16,
                   (which ? a.v8 : a.k8) + (row0 + row) * ATT_D + col * 16);
      }
      if (lane < 8) {
        const int which = lane >> 2, part = lane & 3;
        cp_async16(dst + 2 * ATT8_CODES + which * ATT_PAGE * 4 + part * 16, (which ? a.vs : a.ks) + row0 + 4 * part);
      }
    } else if (pg >= 0) {
      const size_t off = ((size_t)pg * a.Hkv + kvh) * ATT_SLICE;
      __half* dh = reinterpret_cast<__half*>(dst);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = lane + 32 * i;  // 16-byte chunk of the page: [K|V][row][16]
        const int which = c >> 8, row = (c >> 4) & 15, col = c & 15;
        cp_async16(dh + which * ATT_SSLICE + row * ATT_PITCH + col * 8,
                   (which ? a.v_pool : a.k_pool) + off + row * ATT_D + col * 8);
      }
    } else if (lane == 0 && li < my_pages && a.err_flag) {
      atomicOr(a.err_flag, 1);
    }
    cp_async_commit();
  };
  for (int li = 0; li < ST; ++li) issue(li, li < my_pages ? page_of(li) : -1);
  const int pos = L - 1;
  // fused: the 64 (cos, sin) pairs of this position, each computed once and
  // before the dependency wait (the position comes from the lengths, which
  // an older kernel of the step wrote)
  __shared__ float s_cos[ATT_D / 2], s_sin[ATT_D / 2];
  if (FUSE && tid < ATT_D / 2) {
    const float ang = __fmul_rn((float)(pos > 0 ? pos : 0), a.inv_freq[tid]);  // the fp32 product
    sincosf(ang, &s_sin[tid], &s_cos[tid]);
  }
  if (FUSE) {
    pdl_wait_then_trigger();
    W4_TRACE_WAITED();
  }

  // ---- q (and, fused, RoPE of q and the new k; append of k and v) ----------
  const __half* qb = a.q + (size_t)b * a.q_stride + (size_t)kvh * G * ATT_D;
  if (FUSE) {
    // each thread rotates pairs (i, i + 64) of q heads / the new k straight
    // from the q|k|v rows (the q|k|v GEMV's output, read through L2)
    const __half* kn = a.q + (size_t)b * a.q_stride + (size_t)(a.Hq + kvh) * ATT_D;
    const __half* vn = a.q + (size_t)b * a.q_stride + (size_t)(a.Hq + a.Hkv + kvh) * ATT_D;
    constexpr int NPAIR = (G + 1) * (ATT_D / 2);
    constexpr int PER = (NPAIR + NW * 32 - 1) / (NW * 32);
    __half x0h[PER], x1h[PER], vh = __float2half(0.f);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = tid + u * NW * 32;
      if (idx < NPAIR) {
        const int h = idx / (ATT_D / 2), i = idx % (ATT_D / 2);
        const __half* src = h < G ? qb + h * ATT_D : kn;
        x0h[u] = __ldcg(src + i);
        x1h[u] = __ldcg(src + i + ATT_D / 2);
      }
    }
    if (tid < ATT_D) vh = __ldcg(vn + tid);
    __syncthreads();  // s_cos / s_sin
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = tid + u * NW * 32;
      if (idx < NPAIR) {
        const int h = idx / (ATT_D / 2), i = idx % (ATT_D / 2);
        const float cs = s_cos[i], sn = s_sin[i];
        const float x0 = __half2float(x0h[u]), x1 = __half2float(x1h[u]);
        const __half r0 = __float2half_rn(x0 * cs - x1 * sn);
        const __half r1 = __float2half_rn(x1 * cs + x0 * sn);
        if (h < G) {
          s_q[h][i] = __half2float(r0);
          s_q[h][i + ATT_D / 2] = __half2float(r1);
        } else {
          s_knew[i] = r0;
          s_knew[i + ATT_D / 2] = r1;
        }
      }
    }
    if (tid < ATT_D) s_vnew[tid] = vh;
    __syncthreads();
    if (KV8 && warp < 2) {
      // quantise the new k (warp 0) and v (warp 1) rows: the largest
      // magnitude maps to 448, codes in fp32 round-to-nearest-even
      const __half* src = warp == 0 ? s_knew : s_vnew;
      const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
      const __half* h4 = reinterpret_cast<const __half*>(&raw);
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(__half2float(h4[e])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
      const uint32_t c01 = f32x2_to_e4m3x2(__fmul_rn(__half2float(h4[0]), inv), __fmul_rn(__half2float(h4[1]), inv));
      const uint32_t c23 = f32x2_to_e4m3x2(__fmul_rn(__half2float(h4[2]), inv), __fmul_rn(__half2float(h4[3]), inv));
      *reinterpret_cast<uint32_t*>(&s_new8[warp][4 * lane]) = c01 | (c23 << 16);
      if (lane == 0) s_new8_scale[warp] = __fdiv_rn(amax, 448.0f);
    }
    if (KV8) __syncthreads();
    if (pos >= cta_t0 && pos < cta_t1) {  // this CTA holds the new token: append it
      const int blk = pos / ATT_PAGE;
      const int pg = (blk < a.max_blocks) ? __ldcg(&bt[blk]) : -1;
      if (pg >= 0 && pg < a.num_pages) {
        const size_t row = ((size_t)pg * a.Hkv + kvh) * ATT_PAGE + pos % ATT_PAGE;
        if (KV8) {
          for (int d = tid; d < ATT_D; d += blockDim.x) {
            a.k8[row * ATT_D + d] = s_new8[0][d];
            a.v8[row * ATT_D + d] = s_new8[1][d];
          }
          if (tid == 0) {
            a.ks[row] = s_new8_scale[0];
            a.vs[row] = s_new8_scale[1];
          }
        } else {
          for (int d = tid; d < ATT_D; d += blockDim.x) {
            a.k_pool[row * ATT_D + d] = s_knew[d];
            a.v_pool[row * ATT_D + d] = s_vnew[d];
          }
        }
      } else if (tid == 0 && a.err_flag) {
        atomicOr(a.err_flag, 1);
      }
    }
  } else {
    static_assert(G * ATT_D / 8 <= 4 * 32, "one q word per thread of the smallest CTA");
    if (tid < G * ATT_D / 8) {
      const __half* hq = reinterpret_cast<const __half*>(&q_word);
#pragma unroll
      for (int i = 0; i < 8; ++i) s_q[(tid * 8 + i) / ATT_D][(tid * 8 + i) % ATT_D] = __half2float(hq[i]);
    }
    __syncthreads();
  }

  W4_TRACE_MARK(0);
  // ---- tensor-core fragments (mma.sync m16n8k16): lane = (g, t) ------------
  // A rows are the query heads (rows >= G and the upper 8 rows are zero),
  // B columns are tokens (scores) or dims (P.V).  This lane holds rows g of
  // every accumulator, columns 2t, 2t+1.
  const int g = lane >> 2, t4 = lane & 3;
  const bool head_ok = g < G;
  uint32_t qa[8][2];  // q of head g, dims 16s + 2t4 + {0,1} and 16s + 8 + 2t4 + {0,1}, fp16 (FP8: attn8_qdim)
  if (KV8) attn_q_frags_fp8(s_q, G, g, t4, qa);
  else attn_q_frags(s_q, G, g, t4, qa);
  float m_run = -INFINITY, l_run = 0.f;  // head g's running max (log2 domain) and sum
  float o[16][4];                        // P.V accumulators, n-block nb = dims 8nb..8nb+7 (FP8: attn8_odim)
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  const uint32_t k_off = attn_k_off(lane), v_off = attn_v_off(lane);

  for (int li = 0; li < my_pages; ++li) {
    const int stage = li % ST;
    cp_async_wait<ST - 1>();  // this lane's copies of page li landed
    __syncwarp();             // ... and every other lane's
    unsigned char* sl = myring + (size_t)stage * SLOT;
    __half* Ks = reinterpret_cast<__half*>(sl);
    __half* Vs = Ks + ATT_SSLICE;
    const int gi = WP ? li : warp + li * NW;  // page index within the partition
    const int tok0 = (pg0 + gi) * ATT_PAGE;
    const bool page_ok = page_of(li) >= 0;
    const int nv = page_ok ? min(ATT_PAGE, t_end - tok0) : 0;
    if (FUSE && page_ok && pos >= tok0 && pos < tok0 + ATT_PAGE) {
      // the page was fetched before the append: patch the new token's row
      const int slot = pos - tok0;
      if (KV8) {
        *reinterpret_cast<uint32_t*>(sl + slot * ATT8_PITCH + 4 * lane) =
            *reinterpret_cast<const uint32_t*>(&s_new8[0][4 * lane]);
        *reinterpret_cast<uint32_t*>(sl + ATT8_CODES + slot * ATT8_PITCH + 4 * lane) =
            *reinterpret_cast<const uint32_t*>(&s_new8[1][4 * lane]);
        if (lane == 0) {
          reinterpret_cast<float*>(sl + 2 * ATT8_CODES)[slot] = s_new8_scale[0];
          reinterpret_cast<float*>(sl + 2 * ATT8_CODES)[ATT_PAGE + slot] = s_new8_scale[1];
        }
      } else {
        *reinterpret_cast<uint2*>(Ks + slot * ATT_PITCH + 4 * lane) = *reinterpret_cast<const uint2*>(s_knew + 4 * lane);
        *reinterpret_cast<uint2*>(Vs + slot * ATT_PITCH + 4 * lane) = *reinterpret_cast<const uint2*>(s_vnew + 4 * lane);
      }
      __syncwarp();
    }
    if (nv > 0) {
      if (KV8) attn_page_fp8(sl, nv, qa, a.scale_log2, g, t4, m_run, l_run, o);
      else attn_page(Ks, Vs, nv, qa, a.scale_log2, k_off, v_off, t4, m_run, l_run, o);
    }
    __syncwarp();
    // refill this stage with the page ST ahead (an empty group past the end)
    issue(li + ST, li + ST < my_pages ? page_of(li + ST) : -1);
  }
  cp_async_wait<0>();
  __syncthreads();  // all warps done with their rings
  W4_TRACE_MARK(1);

  // ---- merge the warps' states in shared memory (ring reused).  In the
  // warp-per-partition variant these are NW whole partitions, merged by the
  // same online-softmax rule as any two partials. -----------------------------
  const size_t qh0 = (size_t)b * a.Hq + (size_t)kvh * G;
  const int PC = gridDim.x;         // CTA partials per (sequence, kv head)
  const int pc = blockIdx.x;
  const bool clu = !WP && a.use_cluster && PC > 1;
  float* mo = reinterpret_cast<float*>(smraw);          // [NW][8][128]
  float* mml = mo + NW * 8 * ATT_D;                     // [NW][8][2]
  if (head_ok) {
    if (KV8) {
#pragma unroll
      for (int nb = 0; nb < 16; ++nb) {
        mo[(warp * 8 + g) * ATT_D + attn8_odim(nb, t4, 0)] = o[nb][0];
        mo[(warp * 8 + g) * ATT_D + attn8_odim(nb, t4, 1)] = o[nb][1];
      }
    } else {
#pragma unroll
      for (int nb = 0; nb < 16; ++nb)
        *reinterpret_cast<float2*>(mo + (warp * 8 + g) * ATT_D + 8 * nb + 2 * t4) = make_float2(o[nb][0], o[nb][1]);
    }
    if (t4 == 0) {
      mml[(warp * 8 + g) * 2 + 0] = m_run;
      mml[(warp * 8 + g) * 2 + 1] = l_run;
    }
  }
  __syncthreads();
  // thread (h, 4 dims): this CTA's merged state; M = max m, den = sum e^(m-M) l,
  // acc = sum e^(m-M) o.  It goes to the output (one partial), to the cluster
  // leader's shared memory, or to the workspace.
  float* cp_o = mml + NW * 8 * 2;  // [G][128] (workspace path)
  float* cp_ml = cp_o + G * ATT_D; // [G][2]
  for (int idx = tid; idx < G * (ATT_D / 4); idx += blockDim.x) {
    const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mml[(w * 8 + h) * 2]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = mml[(w * 8 + h) * 2];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        const float4 v = *reinterpret_cast<const float4*>(mo + (w * 8 + h) * ATT_D + 4 * d4);
        acc.x = fmaf(v.x, f, acc.x);
        acc.y = fmaf(v.y, f, acc.y);
        acc.z = fmaf(v.z, f, acc.z);
        acc.w = fmaf(v.w, f, acc.w);
        den = fmaf(mml[(w * 8 + h) * 2 + 1], f, den);
      }
    }
    if (PC == 1) {
      const float inv = den > 0.f ? 1.f / den : 0.f;
      __half2* dst = reinterpret_cast<__half2*>(a.out + (qh0 + h) * ATT_D + 4 * d4);
      dst[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
      dst[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
    } else if (clu) {
      // into slot `pc` of the leader's (rank 0's) partial table
      st_dsmem4(&s_clu[(pc * G + h) * (ATT_D + 4) + 4 * d4], 0, acc);
      if (d4 == 0) st_dsmem2(&s_clu[(pc * G + h) * (ATT_D + 4) + ATT_D], 0, make_float2(M, den));
    } else {
      *reinterpret_cast<float4*>(cp_o + h * ATT_D + 4 * d4) = acc;
      if (d4 == 0) {
        cp_ml[h * 2] = M;
        cp_ml[h * 2 + 1] = den;
      }
    }
  }
  if (PC == 1) return;
  W4_TRACE_MARK(2);

  if (clu) {
    // one cluster barrier: every CTA's partial has landed in the leader's
    // table; the leader merges them (partitions with no tokens carry M = -inf)
    cluster_sync();
    if (pc != 0) return;
    for (int idx = tid; idx < G * (ATT_D / 4); idx += blockDim.x) {
      const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
      float M = -INFINITY;
      for (int j = 0; j < PC; ++j) M = fmaxf(M, s_clu[(j * G + h) * (ATT_D + 4) + ATT_D]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
      if (M != -INFINITY) {
        for (int j = 0; j < PC; ++j) {
          const float* e = &s_clu[(j * G + h) * (ATT_D + 4)];
          const float mj = e[ATT_D];
          const float f = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
          const float4 v = *reinterpret_cast<const float4*>(e + 4 * d4);
          acc.x = fmaf(v.x, f, acc.x);
          acc.y = fmaf(v.y, f, acc.y);
          acc.z = fmaf(v.z, f, acc.z);
          acc.w = fmaf(v.w, f, acc.w);
          den = fmaf(e[ATT_D + 1], f, den);
        }
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      __half2* dst = reinterpret_cast<__half2*>(a.out + (qh0 + h) * ATT_D + 4 * d4);
      dst[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
      dst[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
    }
    return;
  }

  // several CTA partials without a cluster: this CTA's partial goes to the
  // workspace ([qh][PC][128]), then the ticket
  const int cta_tokens = (WP ? NW : 1) * a.part_tokens;
  __syncthreads();
  if (pc * cta_tokens < L) {
    for (int idx = tid; idx < G * ATT_D / 4; idx += blockDim.x) {
      const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
      *reinterpret_cast<float4*>(a.ws_o + ((qh0 + h) * PC + pc) * ATT_D + 4 * d4) =
          *reinterpret_cast<const float4*>(cp_o + h * ATT_D + 4 * d4);
    }
    if (tid < G) {
      a.ws_ml[((qh0 + tid) * PC + pc) * 2 + 0] = cp_ml[tid * 2];
      a.ws_ml[((qh0 + tid) * PC + pc) * 2 + 1] = cp_ml[tid * 2 + 1];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int ticket = atomicAdd(&a.counters[(size_t)b * a.Hkv + kvh], 1u);
    s_last = (ticket == (unsigned int)(PC - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Combine, in parallel: (1) all (max, sum) pairs into shared memory,
  // (2) one thread per head turns them into weights, (3) the weighted
  // partial outputs are summed four dims per thread (16-byte loads, all
  // partials of a head in flight together).
  const int Pv = L > 0 ? min(PC, (L + cta_tokens - 1) / cta_tokens) : 0;
  float* cw = reinterpret_cast<float*>(smraw);  // [G][Pv] maxima, then weights
  float* cl = cw + G * Pv;                      // [G][Pv] sums
  for (int idx = tid; idx < G * Pv; idx += blockDim.x) {
    const int h = idx / Pv, j = idx - h * Pv;
    const size_t slot = (qh0 + h) * PC + j;
    cw[idx] = __ldcg(&a.ws_ml[slot * 2]);
    cl[idx] = __ldcg(&a.ws_ml[slot * 2 + 1]);
  }
  __syncthreads();
  if (tid < G) {
    float* mw = cw + tid * Pv;
    float* lw = cl + tid * Pv;
    float M = -INFINITY;
    for (int j = 0; j < Pv; ++j) M = fmaxf(M, mw[j]);
    float den = 0.f;
    for (int j = 0; j < Pv; ++j) {
      const float f = (M == -INFINITY || mw[j] == -INFINITY) ? 0.f : exp2f(mw[j] - M);
      mw[j] = f;
      den += lw[j] * f;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int j = 0; j < Pv; ++j) mw[j] *= inv;
  }
  __syncthreads();
  // G x 32 (head, 4-dim) outputs over the CTA's threads
  for (int idx = tid; idx < G * (ATT_D / 4); idx += blockDim.x) {
    const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
    const float* wts = cw + h * Pv;
    const float4* src = reinterpret_cast<const float4*>(a.ws_o + ((qh0 + h) * PC) * ATT_D) + d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < Pv; ++j) {
      const float4 v = __ldcg(src + (size_t)j * (ATT_D / 4));
      const float w = wts[j];
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    __half2* dst = reinterpret_cast<__half2*>(a.out + (qh0 + h) * ATT_D + 4 * d4);
    dst[0] = __floats2half2_rn(acc.x, acc.y);
    dst[1] = __floats2half2_rn(acc.z, acc.w);
  }
  if (tid == 0) a.counters[(size_t)b * a.Hkv + kvh] = 0u;  // ready for the next call
}

size_t attention_workspace_bytes(int B, int Hq, int Hkv, int P) {
  (void)Hkv;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return ATT_TICKET_BYTES + up((size_t)B * Hq * P * ATT_D * 4) + up((size_t)B * Hq * P * 2 * 4);
}

void attention_workspace_layout(AttnArgs& a, void* ws, int B, int Hq, int P) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  char* w = static_cast<char*>(ws);
  a.counters = reinterpret_cast<unsigned int*>(w);
  a.ws_o = reinterpret_cast<float*>(w + ATT_TICKET_BYTES);
  a.ws_ml = reinterpret_cast<float*>(w + ATT_TICKET_BYTES + up((size_t)B * Hq * P * ATT_D * 4));
}

template <int G, int NW, bool WP, bool KV8>
static int launch_attn_gw(const AttnArgs& a, cudaStream_t s) {
  static PerDeviceOnce once;
  auto k0 = w4pg_paged_attn<G, false, NW, WP, KV8>;
  auto k1 = w4pg_paged_attn<G, true, NW, WP, KV8>;
  constexpr size_t smem = att_smem(NW, att_stages(WP), KV8);
  once_per_device(once, [&] {
    cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  dim3 grid(WP ? (a.P + NW - 1) / NW : a.P, a.Hkv, a.B);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.use_cluster ? a.P : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = a.fuse_rope_append ? cudaLaunchKernelEx(&cfg, k1, a) : cudaLaunchKernelEx(&cfg, k0, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "paged attention launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

// Many partitions (at least two per SM): every warp owns one partition and
// writes its partial itself (4-warp CTAs, three per SM); the last CTA of a
// (sequence, kv head) combines.  Fewer partitions: a CTA of 8 warps per
// partition, merged in shared memory (and across a cluster).
template <int G>
static int launch_attn_g(const AttnArgs& a, cudaStream_t s) {
  const long parts = (long)a.P * a.Hkv * a.B;
  const bool wp = !a.use_cluster && parts >= 2L * num_sms();
  if (a.kv8) return wp ? launch_attn_gw<G, 4, true, true>(a, s) : launch_attn_gw<G, ATT_NW, false, true>(a, s);
  return wp ? launch_attn_gw<G, 4, true, false>(a, s) : launch_attn_gw<G, ATT_NW, false, false>(a, s);
}

int launch_paged_attention(const AttnArgs& a_in, cudaStream_t s) {
  if (a_in.P > ATT_MAX_PARTITIONS)
    return set_error(W4A16_ERR_SHAPE, "paged attention: %d partitions > %d", a_in.P, ATT_MAX_PARTITIONS);
  if (a_in.P > 1 && (size_t)a_in.B * a_in.Hkv * 4 > ATT_TICKET_BYTES)
    return set_error(W4A16_ERR_SHAPE, "paged attention: B*Hkv=%d split-K tickets > %zu", a_in.B * a_in.Hkv,
                     ATT_TICKET_BYTES / 4);
  AttnArgs a = a_in;
  // up to 8 partitions (a portable cluster) merge through distributed shared
  // memory; more go through the workspace and a last-CTA ticket
  a.use_cluster = (a.P > 1 && a.P <= ATT_MAX_CLUSTER) ? 1 : 0;
  switch (a.Hq / a.Hkv) {
    case 1: return launch_attn_g<1>(a, s);
    case 2: return launch_attn_g<2>(a, s);
    case 4: return launch_attn_g<4>(a, s);
    case 7: return launch_attn_g<7>(a, s);
    case 8: return launch_attn_g<8>(a, s);
    default:
      return set_error(W4A16_ERR_SHAPE, "paged attention: Hq/Hkv=%d not built (1, 2, 4, 7, 8)", a.Hq / a.Hkv);
  }
}

// ---------------------------------------------------------------------------
// Causal attention of a prompt (prefill): row i of q (i < T) is the token at
// position context_lens[i] - 1 of ONE sequence, whose pages are row 0 of the
// block table, and attends to the keys at positions 0 .. its own.  A CTA
// takes 16 consecutive rows and one kv head; every K/V page of its range is
// copied once into a ring shared by the CTA's 8 warps, and warp w works on
// rows 2w and 2w + 1 together (the MMA's rows 0-7 and 8-15), so each page
// feeds 16 query tokens x G heads.  KV8: FP8 (E4M3) pages, codes and row
// scales, in the dim orders of the FP8 decode step (attn8_qdim, attn8_odim).
// ---------------------------------------------------------------------------
constexpr int PF_ROWS = 16;    // query rows per CTA
constexpr int PF_WARPS = 8;
constexpr int PF_STAGES = 3;   // page slots of the CTA's ring
constexpr size_t pf_slot_bytes(bool kv8) { return kv8 ? (size_t)ATT8_SLOT : (size_t)2 * ATT_SSLICE * 2; }

template <int G, bool KV8>
__global__ void __launch_bounds__(PF_WARPS * 32) w4pg_prefill_attn(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y;
  const int row0 = blockIdx.x * PF_ROWS;
  const int g = lane >> 2, t4 = lane & 3;
  W4_TRACE_SCOPE(a.tag);
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  // this warp's two rows and their positions (-1: no such row)
  const int rA = row0 + 2 * warp, rB = rA + 1;
  const int posA = rA < a.B ? __ldcg(&a.context_lens[rA]) - 1 : -1;
  const int posB = rB < a.B ? __ldcg(&a.context_lens[rB]) - 1 : -1;
  // the CTA's key range: up to its last row's position
  const int rl = min(a.B, row0 + PF_ROWS) - 1;
  const int L = __ldcg(&a.context_lens[rl]);
  const int npages = (L + ATT_PAGE - 1) / ATT_PAGE;
  if (L > a.max_blocks * ATT_PAGE && tid == 0 && a.err_flag) atomicOr(a.err_flag, 1);
  // query fragments: rows g (token A) and 8 + g (token B), head kvh G + g
  uint32_t qa[8][4];
#pragma unroll
  for (int st = 0; st < 8; ++st) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = r ? rB : rA;
      uint32_t lo = 0u, hi = 0u;
      if (g < G && row < a.B) {
        const __half* qh = a.q + (size_t)row * a.q_stride + (size_t)(kvh * G + g) * ATT_D;
        if (KV8) {
          // physical dims p0 .. p0 + 3 (see attn8_qdim)
          const uint2 q4 = __ldcg(reinterpret_cast<const uint2*>(qh + attn8_qdim(st, t4)));
          lo = q4.x;
          hi = q4.y;
        } else {
          lo = __ldcg(reinterpret_cast<const unsigned int*>(qh + 16 * st + 2 * t4));
          hi = __ldcg(reinterpret_cast<const unsigned int*>(qh + 16 * st + 8 + 2 * t4));
        }
      }
      qa[st][r] = lo;
      qa[st][2 + r] = hi;
    }
  }
  constexpr int SLOT = (int)pf_slot_bytes(KV8);  // K and V slices, padded rows (+ FP8 row scales)
  auto page_id = [&](int li) -> int {
    const int pg = li < a.max_blocks ? __ldcg(&a.block_table[li]) : -1;
    return (pg >= 0 && pg < a.num_pages) ? pg : -1;
  };
  // page li into slot li % PF_STAGES: 2 x 16 rows of 256 bytes, 512 16-byte
  // copies over the CTA's 256 threads; one commit group per page
  auto issue = [&](int li) {
    if (li < npages) {
      const int pg = page_id(li);
      if (pg >= 0 && KV8) {
        // 2 x 16 rows of 128 code bytes (256 16-byte copies) and the 2 x 16 row scales
        unsigned char* dst = smraw + (size_t)(li % PF_STAGES) * SLOT;
        const size_t row0 = ((size_t)pg * a.Hkv + kvh) * ATT_PAGE;
        const int which = tid >> 7, row = (tid >> 3) & 15, col = tid & 7;  // [K|V][row][8 chunks]
        cp_async16(dst + which * ATT8_CODES + row * ATT8_PITCH + col * 16,
                   (which ? a.v8 : a.k8) + (row0 + row) * ATT_D + col * 16);
        if (tid < 8) {
          const int w = tid >> 2, part = tid & 3;
          cp_async16(dst + 2 * ATT8_CODES + w * ATT_PAGE * 4 + part * 16, (w ? a.vs : a.ks) + row0 + 4 * part);
        }
      } else if (pg >= 0) {
        unsigned char* dst = smraw + (size_t)(li % PF_STAGES) * SLOT;
        const size_t off = ((size_t)pg * a.Hkv + kvh) * ATT_SLICE;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = tid + 256 * i;  // [K|V][row][16 chunks]
          const int which = c >> 8, row = (c >> 4) & 15, col = c & 15;
          cp_async16(dst + (size_t)which * ATT_SSLICE * 2 + row * ATT_PITCH * 2 + col * 16,
                     (which ? a.v_pool : a.k_pool) + off + (size_t)row * ATT_D + col * 8);
        }
      } else if (tid == 0 && a.err_flag) {
        atomicOr(a.err_flag, 1);
      }
    }
    cp_async_commit();
  };
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  const uint32_t k_off = attn_k_off(lane), v_off = attn_v_off(lane);
#pragma unroll
  for (int i = 0; i < PF_STAGES - 1; ++i) issue(i);
  for (int li = 0; li < npages; ++li) {
    cp_async_wait<PF_STAGES - 2>();  // this thread's copies of page li landed
    __syncthreads();                 // everyone's; and every warp is done with page li - 1
    issue(li + PF_STAGES - 1);       // into the slot page li - 1 used
    const int tok0 = li * ATT_PAGE;
    // rows whose position is before this page see nothing in it (posB is -1
    // when the warp has only row A)
    if (max(posA, posB) >= tok0 && page_id(li) >= 0) {
      const unsigned char* sl = smraw + (size_t)(li % PF_STAGES) * SLOT;
      if (KV8) {
        attn_page_pair_fp8(sl, tok0, posA, posB, qa, a.scale_log2, g, t4, m_run, l_run, o);
      } else {
        const __half* Ks = reinterpret_cast<const __half*>(sl);
        attn_page_pair(Ks, Ks + ATT_SSLICE, tok0, posA, posB, qa, a.scale_log2, k_off, v_off, t4, m_run, l_run, o);
      }
    }
  }
  cp_async_wait<0>();
  // normalise and write: row g -> token A, head kvh G + g; row 8 + g -> token B
  if (g < G) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = r ? rB : rA;
      if (row >= a.B) continue;
      const float inv = l_run[r] > 0.f ? 1.0f / l_run[r] : 0.f;
      __half* outh = a.out + (size_t)row * a.Hq * ATT_D + (size_t)(kvh * G + g) * ATT_D;
      if (KV8) {
#pragma unroll
        for (int nb = 0; nb < 16; ++nb) {
          outh[attn8_odim(nb, t4, 0)] = __float2half_rn(o[nb][2 * r] * inv);
          outh[attn8_odim(nb, t4, 1)] = __float2half_rn(o[nb][2 * r + 1] * inv);
        }
      } else {
#pragma unroll
        for (int nb = 0; nb < 16; ++nb)
          *reinterpret_cast<__half2*>(outh + 8 * nb + 2 * t4) =
              __floats2half2_rn(o[nb][2 * r] * inv, o[nb][2 * r + 1] * inv);
      }
    }
  }
}

template <int G, bool KV8>
static int launch_prefill_attn_g(const AttnArgs& a, cudaStream_t s) {
  constexpr size_t smem = (size_t)PF_STAGES * pf_slot_bytes(KV8);
  auto kern = w4pg_prefill_attn<G, KV8>;
  static PerDeviceOnce once;
  once_per_device(once, [&] { cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); });
  const dim3 grid((a.B + PF_ROWS - 1) / PF_ROWS, a.Hkv);
  cudaError_t e = launch_pdl(kern, grid, dim3(PF_WARPS * 32), smem, s, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "prefill attention launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

int launch_prefill_attention(const AttnArgs& a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return a.kv8 ? launch_prefill_attn_g<1, true>(a, s) : launch_prefill_attn_g<1, false>(a, s);
    case 2: return a.kv8 ? launch_prefill_attn_g<2, true>(a, s) : launch_prefill_attn_g<2, false>(a, s);
    case 4: return a.kv8 ? launch_prefill_attn_g<4, true>(a, s) : launch_prefill_attn_g<4, false>(a, s);
    case 7: return a.kv8 ? launch_prefill_attn_g<7, true>(a, s) : launch_prefill_attn_g<7, false>(a, s);
    case 8: return a.kv8 ? launch_prefill_attn_g<8, true>(a, s) : launch_prefill_attn_g<8, false>(a, s);
    default:
      return set_error(W4A16_ERR_SHAPE, "prefill attention: Hq/Hkv=%d not built (1, 2, 4, 7, 8)", a.Hq / a.Hkv);
  }
}

// ---------------------------------------------------------------------------
// RoPE + KV append: one CTA per sequence.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) w4pg_rope_append(const __grid_constant__ RopeArgs a) {
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int pos = a.context_lens[b] - 1;
  if (pos < 0) return;
  const int blk = pos / ATT_PAGE, slot = pos % ATT_PAGE;
  const int page = (blk < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + blk] : -1;
  const bool ok = page >= 0 && page < a.num_pages;
  if (!ok && threadIdx.x == 0 && a.err_flag) atomicOr(a.err_flag, 1);
  const float fpos = (float)pos;
  const int nrot = (a.Hq + a.Hkv) * (ATT_D / 2);
  for (int idx = threadIdx.x; idx < nrot; idx += blockDim.x) {
    const int head = idx / (ATT_D / 2), i = idx % (ATT_D / 2);
    const float ang = __fmul_rn(fpos, a.inv_freq[i]);  // the fp32 product, no contraction
    float sn, cs;
    sincosf(ang, &sn, &cs);
    if (head < a.Hq) {
      __half* x = a.q + (size_t)b * a.stride_q + (size_t)head * ATT_D;
      const float x0 = __half2float(x[i]), x1 = __half2float(x[i + ATT_D / 2]);
      x[i] = __float2half_rn(x0 * cs - x1 * sn);
      x[i + ATT_D / 2] = __float2half_rn(x1 * cs + x0 * sn);
    } else if (ok) {
      const int kh = head - a.Hq;
      const __half* x = a.k + (size_t)b * a.stride_kv + (size_t)kh * ATT_D;
      const float x0 = __half2float(x[i]), x1 = __half2float(x[i + ATT_D / 2]);
      __half* dst = a.k_pool + (((size_t)page * a.Hkv + kh) * ATT_PAGE + slot) * ATT_D;
      dst[i] = __float2half_rn(x0 * cs - x1 * sn);
      dst[i + ATT_D / 2] = __float2half_rn(x1 * cs + x0 * sn);
    }
  }
  if (ok) {
    for (int idx = threadIdx.x; idx < a.Hkv * ATT_D; idx += blockDim.x) {
      const int kh = idx / ATT_D, dd = idx % ATT_D;
      a.v_pool[(((size_t)page * a.Hkv + kh) * ATT_PAGE + slot) * ATT_D + dd] =
          a.v[(size_t)b * a.stride_kv + (size_t)kh * ATT_D + dd];
    }
  }
}

// RoPE + FP8 append: one CTA per sequence; q heads rotated in place, each kv
// head's rotated k row and v row quantised by one warp (largest magnitude to
// 448, fp32 round-to-nearest-even codes) into its slot.
__global__ void __launch_bounds__(256) w4pg_rope_append_fp8(const __grid_constant__ RopeArgs a) {
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait();
  const int pos = a.context_lens[b] - 1;
  if (pos < 0) return;
  const int blk = pos / ATT_PAGE, slot = pos % ATT_PAGE;
  const int page = (blk < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + blk] : -1;
  const bool ok = page >= 0 && page < a.num_pages;
  if (!ok && threadIdx.x == 0 && a.err_flag) atomicOr(a.err_flag, 1);
  const float fpos = (float)pos;
  for (int idx = threadIdx.x; idx < a.Hq * (ATT_D / 2); idx += blockDim.x) {
    const int head = idx / (ATT_D / 2), i = idx % (ATT_D / 2);
    float sn, cs;
    sincosf(__fmul_rn(fpos, a.inv_freq[i]), &sn, &cs);
    __half* x = a.q + (size_t)b * a.stride_q + (size_t)head * ATT_D;
    const float x0 = __half2float(x[i]), x1 = __half2float(x[i + ATT_D / 2]);
    x[i] = __float2half_rn(x0 * cs - x1 * sn);
    x[i + ATT_D / 2] = __float2half_rn(x1 * cs + x0 * sn);
  }
  if (!ok) return;
  for (int kh = warp; kh < a.Hkv; kh += blockDim.x / 32) {
    const __half* kx = a.k + (size_t)b * a.stride_kv + (size_t)kh * ATT_D;
    const __half* vx = a.v + (size_t)b * a.stride_kv + (size_t)kh * ATT_D;
    float kr[4], vr[4];  // dims lane, lane + 32, lane + 64, lane + 96
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = lane + 32 * e;
      float sn, cs;
      sincosf(__fmul_rn(fpos, a.inv_freq[i]), &sn, &cs);
      const float x0 = __half2float(kx[i]), x1 = __half2float(kx[i + ATT_D / 2]);
      kr[e] = __half2float(__float2half_rn(x0 * cs - x1 * sn));
      kr[e + 2] = __half2float(__float2half_rn(x1 * cs + x0 * sn));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) vr[e] = __half2float(vx[lane + 32 * e]);
    const size_t row = ((size_t)page * a.Hkv + kh) * ATT_PAGE + slot;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float* r = which ? vr : kr;
      float amax = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
      uint8_t* dst = (which ? a.v8 : a.k8) + row * ATT_D;
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = (uint8_t)(f32x2_to_e4m3x2(__fmul_rn(r[e], inv), 0.f) & 0xFFu);
      if (lane == 0) (which ? a.vs : a.ks)[row] = __fdiv_rn(amax, 448.0f);
    }
  }
}

void rope_inv_freq_table(float theta, int D, float* out) {
  for (int i = 0; i < D / 2; ++i) out[i] = (float)std::pow((double)theta, -2.0 * (double)i / (double)D);
}

int launch_rope_append(const RopeArgs& a, cudaStream_t s) {
  cudaError_t e = a.k8 ? launch_pdl(w4pg_rope_append_fp8, dim3(a.B), dim3(256), 0, s, a)
                       : launch_pdl(w4pg_rope_append, dim3(a.B), dim3(256), 0, s, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "rope/append launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

// Partition size: up to 1024 tokens, 128-token partitions (one page per warp,
// every page fetched before the CTA's dependency wait) merged within one
// cluster.  Longer contexts: with many (sequence, kv head) pairs, 256-token
// partitions, one warp each (the 28-layer batch-32 step with lengths up to
// 4096 measured 5.00 ms against 6.03 with 512 and 5.09 with 128); with few,
// 512-token partitions.
int default_partition(int B, int Hkv, int max_context) {
  if (max_context <= ATT_MAX_CLUSTER * 128) return 128;  // one page per warp, one cluster
  if ((long)B * Hkv >= 64) return 256;
  return 512;
}

}  // namespace w4

using namespace w4;

extern "C" int paged_gqa_decode_default_partition(int B, int Hkv, int max_context) {
  if (B < 1 || Hkv < 1 || max_context < 1) return 64;
  return default_partition(B, Hkv, max_context);
}

extern "C" size_t paged_gqa_decode_workspace_size(int B, int Hq, int Hkv, int max_context, int partition_tokens,
                                                  int D) {
  (void)D;
  if (B < 1 || Hq < 1 || Hkv < 1 || max_context < 1) return 0;
  if (partition_tokens <= 0) partition_tokens = default_partition(B, Hkv, max_context);
  const int P = (max_context + partition_tokens - 1) / partition_tokens;
  return attention_workspace_bytes(B, Hq, Hkv, P);
}

extern "C" int w4a16_workspace_clear(void* workspace, size_t bytes, w4a16_stream_t stream) {
  W4_CHECK_ARG(workspace || bytes == 0, "workspace_clear: null workspace");
  if (bytes == 0) return W4A16_OK;
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "workspace_clear: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

extern "C" int paged_gqa_decode(const uint16_t* q, int q_stride, const uint16_t* k_pool, const uint16_t* v_pool,
                                int num_pages, const int32_t* block_table, int max_blocks,
                                const int32_t* context_lens, int max_context, int B, int Hq, int Hkv, int D,
                                float sm_scale, int partition_tokens, void* workspace, size_t workspace_bytes,
                                uint16_t* out, int32_t* err_flag, w4a16_stream_t stream) {
  W4_CHECK_ARG(q && k_pool && v_pool && block_table && context_lens && out,
               "paged_gqa_decode: null tensor pointer");
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1 && max_context >= 1,
               "paged_gqa_decode: sizes must be positive");
  W4_CHECK_SHAPE(D == ATT_D, "paged_gqa_decode: D=%d, only 128 is built", D);
  W4_CHECK_SHAPE(Hq % Hkv == 0 && Hq / Hkv <= 8, "paged_gqa_decode: Hq=%d Hkv=%d", Hq, Hkv);
  W4_CHECK_SHAPE(max_context <= max_blocks * ATT_PAGE, "paged_gqa_decode: max_context %d > max_blocks*16",
                 max_context);
  if (partition_tokens <= 0) partition_tokens = default_partition(B, Hkv, max_context);
  W4_CHECK_SHAPE(partition_tokens % ATT_PAGE == 0, "paged_gqa_decode: partition_tokens %% 16 != 0");
  if (q_stride == 0) q_stride = Hq * D;
  W4_CHECK_ARG(q_stride >= Hq * D, "paged_gqa_decode: q_stride too small");
  W4_CHECK_ALIGN(q, 128, "q");
  W4_CHECK_ALIGN(k_pool, 128, "k_pool");
  W4_CHECK_ALIGN(v_pool, 128, "v_pool");
  W4_CHECK_ALIGN(out, 128, "out");
  W4_CHECK_ARG((q_stride * 2) % 16 == 0, "paged_gqa_decode: q_stride*2 must be a multiple of 16 bytes");
  const int P = (max_context + partition_tokens - 1) / partition_tokens;
  AttnArgs a = {};
  if (P > 1) {
    const size_t need = attention_workspace_bytes(B, Hq, Hkv, P);
    W4_CHECK_ARG(workspace != nullptr && workspace_bytes >= need,
                 "paged_gqa_decode: workspace of %zu bytes needed", need);
    W4_CHECK_ALIGN(workspace, 128, "workspace");
    attention_workspace_layout(a, workspace, B, Hq, P);
  }
  a.q = reinterpret_cast<const __half*>(q);
  a.k_pool = reinterpret_cast<__half*>(const_cast<uint16_t*>(k_pool));
  a.v_pool = reinterpret_cast<__half*>(const_cast<uint16_t*>(v_pool));
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = reinterpret_cast<__half*>(out);
  a.err_flag = err_flag;
  a.q_stride = q_stride;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = P;
  a.part_tokens = partition_tokens;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  return launch_paged_attention(a, (cudaStream_t)stream);
}

extern "C" int paged_gqa_decode_rope_append(const uint16_t* qkv, int qkv_stride, uint16_t* k_pool, uint16_t* v_pool,
                                            int num_pages, const int32_t* block_table, int max_blocks,
                                            const int32_t* context_lens, int max_context, int B, int Hq, int Hkv,
                                            int D, float theta, float sm_scale, int partition_tokens,
                                            void* workspace, size_t workspace_bytes, uint16_t* out, int32_t* err_flag,
                                            w4a16_stream_t stream) {
  W4_CHECK_ARG(qkv && k_pool && v_pool && block_table && context_lens && out,
               "paged_gqa_decode_rope_append: null tensor pointer");
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1 && max_context >= 1,
               "paged_gqa_decode_rope_append: sizes must be positive");
  W4_CHECK_SHAPE(D == ATT_D, "paged_gqa_decode_rope_append: D=%d, only 128 is built", D);
  W4_CHECK_SHAPE(Hq % Hkv == 0 && Hq / Hkv <= 8, "paged_gqa_decode_rope_append: Hq=%d Hkv=%d", Hq, Hkv);
  W4_CHECK_SHAPE(max_context <= max_blocks * ATT_PAGE, "paged_gqa_decode_rope_append: max_context > max_blocks*16");
  W4_CHECK_ARG(theta > 0.f, "paged_gqa_decode_rope_append: theta must be positive");
  if (partition_tokens <= 0) partition_tokens = default_partition(B, Hkv, max_context);
  W4_CHECK_SHAPE(partition_tokens % ATT_PAGE == 0, "paged_gqa_decode_rope_append: partition_tokens %% 16 != 0");
  if (qkv_stride == 0) qkv_stride = (Hq + 2 * Hkv) * D;
  W4_CHECK_ARG(qkv_stride >= (Hq + 2 * Hkv) * D && (qkv_stride * 2) % 16 == 0,
               "paged_gqa_decode_rope_append: bad qkv_stride");
  W4_CHECK_ALIGN(qkv, 128, "qkv");
  W4_CHECK_ALIGN(k_pool, 128, "k_pool");
  W4_CHECK_ALIGN(v_pool, 128, "v_pool");
  W4_CHECK_ALIGN(out, 128, "out");
  const int P = (max_context + partition_tokens - 1) / partition_tokens;
  AttnArgs a = {};
  if (P > 1) {
    const size_t need = attention_workspace_bytes(B, Hq, Hkv, P);
    W4_CHECK_ARG(workspace != nullptr && workspace_bytes >= need,
                 "paged_gqa_decode_rope_append: workspace of %zu bytes needed", need);
    W4_CHECK_ALIGN(workspace, 128, "workspace");
    attention_workspace_layout(a, workspace, B, Hq, P);
  }
  a.q = reinterpret_cast<const __half*>(qkv);
  a.k_pool = reinterpret_cast<__half*>(k_pool);
  a.v_pool = reinterpret_cast<__half*>(v_pool);
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = reinterpret_cast<__half*>(out);
  a.err_flag = err_flag;
  a.q_stride = qkv_stride;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = P;
  a.part_tokens = partition_tokens;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.fuse_rope_append = 1;
  rope_inv_freq_table(theta, D, a.inv_freq);
  return launch_paged_attention(a, (cudaStream_t)stream);
}

extern "C" int kv_append_rope(uint16_t* q, const uint16_t* k, const uint16_t* v, int row_stride, uint16_t* k_pool,
                              uint16_t* v_pool, int num_pages, const int32_t* block_table, int max_blocks,
                              const int32_t* context_lens, int B, int Hq, int Hkv, int D, float theta,
                              int32_t* err_flag, w4a16_stream_t stream) {
  W4_CHECK_ARG(q && k && v && k_pool && v_pool && block_table && context_lens, "kv_append_rope: null pointer");
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1, "kv_append_rope: sizes");
  W4_CHECK_SHAPE(D == ATT_D, "kv_append_rope: D=%d, only 128 is built", D);
  W4_CHECK_SHAPE(Hq % Hkv == 0, "kv_append_rope: Hq %% Hkv != 0");
  W4_CHECK_ARG(theta > 0.f, "kv_append_rope: theta must be positive");
  W4_CHECK_ARG(row_stride >= 0, "kv_append_rope: negative row_stride");
  W4_CHECK_ALIGN(q, 128, "q");
  W4_CHECK_ALIGN(k, 128, "k");
  W4_CHECK_ALIGN(v, 128, "v");
  W4_CHECK_ALIGN(k_pool, 128, "k_pool");
  W4_CHECK_ALIGN(v_pool, 128, "v_pool");
  RopeArgs a = {};
  a.q = reinterpret_cast<__half*>(q);
  a.k = reinterpret_cast<__half*>(const_cast<uint16_t*>(k));
  a.v = reinterpret_cast<const __half*>(v);
  a.k_pool = reinterpret_cast<__half*>(k_pool);
  a.v_pool = reinterpret_cast<__half*>(v_pool);
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.err_flag = err_flag;
  a.stride_q = row_stride ? row_stride : Hq * D;
  a.stride_kv = row_stride ? row_stride : Hkv * D;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  rope_inv_freq_table(theta, D, a.inv_freq);
  return launch_rope_append(a, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) KV pages
// ---------------------------------------------------------------------------
static int check_fp8_pools(const uint8_t* k8, const uint8_t* v8, const float* ks, const float* vs, const char* who) {
  W4_CHECK_ARG(k8 && v8 && ks && vs, "%s: null FP8 pool or scale pointer", who);
  W4_CHECK_ALIGN(k8, 128, "k_pool");
  W4_CHECK_ALIGN(v8, 128, "v_pool");
  W4_CHECK_ALIGN(ks, 128, "k_scale");
  W4_CHECK_ALIGN(vs, 128, "v_scale");
  return W4A16_OK;
}

static int fp8_attention(const uint16_t* q, int q_stride, int fuse, uint8_t* k8, uint8_t* v8, float* ks, float* vs,
                         int num_pages, const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                         int max_context, int B, int Hq, int Hkv, int D, float theta, float sm_scale,
                         int partition_tokens, void* workspace, size_t workspace_bytes, uint16_t* out,
                         int32_t* err_flag, cudaStream_t stream, const char* who) {
  W4_CHECK_ARG(q && block_table && context_lens && out, "%s: null tensor pointer", who);
  int rc = check_fp8_pools(k8, v8, ks, vs, who);
  if (rc) return rc;
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1 && max_context >= 1,
               "%s: sizes must be positive", who);
  W4_CHECK_SHAPE(D == ATT_D, "%s: D=%d, only 128 is built", who, D);
  W4_CHECK_SHAPE(Hq % Hkv == 0 && Hq / Hkv <= 8, "%s: Hq=%d Hkv=%d", who, Hq, Hkv);
  W4_CHECK_SHAPE(max_context <= max_blocks * ATT_PAGE, "%s: max_context > max_blocks*16", who);
  if (fuse) W4_CHECK_ARG(theta > 0.f, "%s: theta must be positive", who);
  if (partition_tokens <= 0) partition_tokens = default_partition(B, Hkv, max_context);
  W4_CHECK_SHAPE(partition_tokens % ATT_PAGE == 0, "%s: partition_tokens %% 16 != 0", who);
  const int min_stride = fuse ? (Hq + 2 * Hkv) * D : Hq * D;
  if (q_stride == 0) q_stride = min_stride;
  W4_CHECK_ARG(q_stride >= min_stride && (q_stride * 2) % 16 == 0, "%s: bad q_stride", who);
  W4_CHECK_ALIGN(q, 128, "q");
  W4_CHECK_ALIGN(out, 128, "out");
  const int P = (max_context + partition_tokens - 1) / partition_tokens;
  AttnArgs a = {};
  if (P > 1) {
    const size_t need = attention_workspace_bytes(B, Hq, Hkv, P);
    W4_CHECK_ARG(workspace != nullptr && workspace_bytes >= need, "%s: workspace of %zu bytes needed", who, need);
    W4_CHECK_ALIGN(workspace, 128, "workspace");
    attention_workspace_layout(a, workspace, B, Hq, P);
  }
  a.q = reinterpret_cast<const __half*>(q);
  a.kv8 = 1;
  a.k8 = k8;
  a.v8 = v8;
  a.ks = ks;
  a.vs = vs;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = reinterpret_cast<__half*>(out);
  a.err_flag = err_flag;
  a.q_stride = q_stride;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = P;
  a.part_tokens = partition_tokens;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.fuse_rope_append = fuse;
  if (fuse) rope_inv_freq_table(theta, D, a.inv_freq);
  return launch_paged_attention(a, stream);
}

extern "C" int paged_gqa_decode_fp8(const uint16_t* q, int q_stride, const uint8_t* k_pool, const uint8_t* v_pool,
                                    const float* k_scale, const float* v_scale, int num_pages,
                                    const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                    int max_context, int B, int Hq, int Hkv, int D, float sm_scale,
                                    int partition_tokens, void* workspace, size_t workspace_bytes, uint16_t* out,
                                    int32_t* err_flag, w4a16_stream_t stream) {
  return fp8_attention(q, q_stride, 0, const_cast<uint8_t*>(k_pool), const_cast<uint8_t*>(v_pool),
                       const_cast<float*>(k_scale), const_cast<float*>(v_scale), num_pages, block_table, max_blocks,
                       context_lens, max_context, B, Hq, Hkv, D, 0.f, sm_scale, partition_tokens, workspace,
                       workspace_bytes, out, err_flag, (cudaStream_t)stream, "paged_gqa_decode_fp8");
}

extern "C" int paged_gqa_decode_rope_append_fp8(const uint16_t* qkv, int qkv_stride, uint8_t* k_pool,
                                                uint8_t* v_pool, float* k_scale, float* v_scale, int num_pages,
                                                const int32_t* block_table, int max_blocks,
                                                const int32_t* context_lens, int max_context, int B, int Hq,
                                                int Hkv, int D, float theta, float sm_scale, int partition_tokens,
                                                void* workspace, size_t workspace_bytes, uint16_t* out,
                                                int32_t* err_flag, w4a16_stream_t stream) {
  return fp8_attention(qkv, qkv_stride, 1, k_pool, v_pool, k_scale, v_scale, num_pages, block_table, max_blocks,
                       context_lens, max_context, B, Hq, Hkv, D, theta, sm_scale, partition_tokens, workspace,
                       workspace_bytes, out, err_flag, (cudaStream_t)stream, "paged_gqa_decode_rope_append_fp8");
}

extern "C" int kv_append_rope_fp8(uint16_t* q, const uint16_t* k, const uint16_t* v, int row_stride,
                                  uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale, int num_pages,
                                  const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B,
                                  int Hq, int Hkv, int D, float theta, int32_t* err_flag, w4a16_stream_t stream) {
  W4_CHECK_ARG(q && k && v && block_table && context_lens, "kv_append_rope_fp8: null pointer");
  int rc = check_fp8_pools(k_pool, v_pool, k_scale, v_scale, "kv_append_rope_fp8");
  if (rc) return rc;
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1, "kv_append_rope_fp8: sizes");
  W4_CHECK_SHAPE(D == ATT_D, "kv_append_rope_fp8: D=%d, only 128 is built", D);
  W4_CHECK_SHAPE(Hq % Hkv == 0, "kv_append_rope_fp8: Hq %% Hkv != 0");
  W4_CHECK_ARG(theta > 0.f, "kv_append_rope_fp8: theta must be positive");
  W4_CHECK_ARG(row_stride >= 0, "kv_append_rope_fp8: negative row_stride");
  W4_CHECK_ALIGN(q, 128, "q");
  W4_CHECK_ALIGN(k, 128, "k");
  W4_CHECK_ALIGN(v, 128, "v");
  RopeArgs a = {};
  a.q = reinterpret_cast<__half*>(q);
  a.k = reinterpret_cast<__half*>(const_cast<uint16_t*>(k));
  a.v = reinterpret_cast<const __half*>(v);
  a.k8 = k_pool;
  a.v8 = v_pool;
  a.ks = k_scale;
  a.vs = v_scale;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.err_flag = err_flag;
  a.stride_q = row_stride ? row_stride : Hq * D;
  a.stride_kv = row_stride ? row_stride : Hkv * D;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  rope_inv_freq_table(theta, D, a.inv_freq);
  return launch_rope_append(a, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the split-K scratch is a static device array.
// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory, so its device address is looked up once per device and passed to
// the kernel like any workspace pointer.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A16_NOALLOC_SCRATCH_BYTES];

static int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "paged_gqa_decode_noalloc: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(W4A16_ERR_INVALID_ARG, "paged_gqa_decode_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(W4A16_ERR_CUDA, "paged_gqa_decode_noalloc: scratch address lookup: %s", cudaGetErrorString(e));
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return W4A16_OK;
}

extern "C" int paged_gqa_decode_noalloc(const uint16_t* q, int q_stride, const uint16_t* k_pool,
                                        const uint16_t* v_pool, int num_pages, const int32_t* block_table,
                                        int max_blocks, const int32_t* context_lens, int max_context, int B, int Hq,
                                        int Hkv, int D, float sm_scale, int partition_tokens, uint16_t* out,
                                        int32_t* err_flag, w4a16_stream_t stream) {
  W4_CHECK_ARG(q && k_pool && v_pool && block_table && context_lens && out,
               "paged_gqa_decode_noalloc: null tensor pointer");
  W4_CHECK_ARG(B >= 1 && Hq >= 1 && Hkv >= 1 && num_pages >= 1 && max_blocks >= 1 && max_context >= 1,
               "paged_gqa_decode_noalloc: sizes must be positive");
  W4_CHECK_SHAPE(D == ATT_D, "paged_gqa_decode_noalloc: D=%d, only 128 is built", D);
  W4_CHECK_SHAPE(Hq % Hkv == 0 && Hq / Hkv <= 8, "paged_gqa_decode_noalloc: Hq=%d Hkv=%d", Hq, Hkv);
  W4_CHECK_SHAPE(max_context <= max_blocks * ATT_PAGE, "paged_gqa_decode_noalloc: max_context %d > max_blocks*16",
                 max_context);
  if (partition_tokens <= 0) partition_tokens = default_partition(B, Hkv, max_context);
  W4_CHECK_SHAPE(partition_tokens % ATT_PAGE == 0, "paged_gqa_decode_noalloc: partition_tokens %% 16 != 0");
  if (q_stride == 0) q_stride = Hq * D;
  W4_CHECK_ARG(q_stride >= Hq * D, "paged_gqa_decode_noalloc: q_stride too small");
  W4_CHECK_ALIGN(q, 128, "q");
  W4_CHECK_ALIGN(k_pool, 128, "k_pool");
  W4_CHECK_ALIGN(v_pool, 128, "v_pool");
  W4_CHECK_ALIGN(out, 128, "out");
  W4_CHECK_ARG((q_stride * 2) % 16 == 0, "paged_gqa_decode_noalloc: q_stride*2 must be a multiple of 16 bytes");
  const int P = (max_context + partition_tokens - 1) / partition_tokens;
  AttnArgs a = {};
  if (P > 1) {
    const size_t need = attention_workspace_bytes(B, Hq, Hkv, P);
    if (need > W4A16_NOALLOC_SCRATCH_BYTES)
      return set_error(W4A16_ERR_SHAPE,
                       "paged_gqa_decode_noalloc: these sizes need %zu bytes of scratch; the static array holds %u",
                       need, (unsigned)W4A16_NOALLOC_SCRATCH_BYTES);
    // the launcher repeats these checks; they come first here so that nothing
    // is cleared for a call that is then refused
    W4_CHECK_SHAPE(P <= ATT_MAX_PARTITIONS, "paged_gqa_decode_noalloc: %d partitions > %d", P, ATT_MAX_PARTITIONS);
    W4_CHECK_SHAPE((size_t)B * Hkv * 4 <= ATT_TICKET_BYTES, "paged_gqa_decode_noalloc: B*Hkv=%d split-K tickets > %zu",
                   B * Hkv, ATT_TICKET_BYTES / 4);
    void* base = nullptr;
    int rc = noalloc_scratch(&base);
    if (rc) return rc;
    attention_workspace_layout(a, base, B, Hq, P);
    // the array keeps the previous call's contents: the tickets must start at zero
    cudaError_t e = cudaMemsetAsync(a.counters, 0, (size_t)B * Hkv * sizeof(unsigned int), (cudaStream_t)stream);
    if (e != cudaSuccess)
      return set_error(W4A16_ERR_CUDA, "paged_gqa_decode_noalloc: clearing counters: %s", cudaGetErrorString(e));
  }
  a.q = reinterpret_cast<const __half*>(q);
  a.k_pool = reinterpret_cast<__half*>(const_cast<uint16_t*>(k_pool));
  a.v_pool = reinterpret_cast<__half*>(const_cast<uint16_t*>(v_pool));
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = reinterpret_cast<__half*>(out);
  a.err_flag = err_flag;
  a.q_stride = q_stride;
  a.num_pages = num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = P;
  a.part_tokens = partition_tokens;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  return launch_paged_attention(a, (cudaStream_t)stream);
}
