// persistent.cu -- one persistent kernel per decode step (one sequence).
//
// "Building a Custom LLM Inference Runtime on H100" (explore.n1n.ai), "3. CUDA
// Graph Capture", and the aikraft.ru article ("Ключевые метрики
// производительности": ~119 ms eager vs ~17 ms graph-captured per token) put
// the cost of a decode step that is not bandwidth in kernel launches.  This
// kernel removes the launches altogether: one cooperative launch walks the
// whole step -- embedding, for each layer the q|k|v GEMV (RMSNorm in front),
// RoPE + KV append + paged GQA attention, the o GEMV + residual, the gate|up
// GEMV + SiLU-mul (RMSNorm in front) and the down GEMV + residual, then the
// final RMSNorm, lm_head and argmax -- with a grid-wide barrier between the
// phases.
//
// Why it is faster than a stream of kernels: weights never depend on the
// previous phase, so every thread streams its share of the step's weights
// through its own FIFO of shared-memory slots (16-byte cp.async copies, one
// commit group per copy) a fixed number of copies ahead of what it computes.
// At a phase boundary that FIFO is already filling with the next phase's
// weights -- the whole of a small projection fits -- while the CTA waits at
// the barrier and stages the new activations; the attention CTAs fetch their
// KV pages (bulk copies into padded rows, completion on mbarriers) before the
// barrier too.
//
// Work split of a GEMV phase: the output rows come in pairs (gate|up: the
// gate and up rows of a pair of outputs, four weight rows); a CTA owns a
// contiguous run of pairs, and the run's (pair, 16-chunk column block) items
// are cut into 32 contiguous ranges, one per half-warp.  Lane l of a
// half-warp takes chunk 16 b + l of every weight row of its items.  A
// half-warp that covers a whole pair writes the outputs itself; a pair cut by
// range boundaries is finished, after a CTA barrier, by the half-warp that
// holds its last item, adding the others' partial sums in half-warp order,
// so every sum has a fixed order and the result is deterministic.
//
// Every wait is bounded (%globaltimer): a barrier that does not complete in
// time sets bit 1 of the error word and an abort flag, and every CTA leaves
// at its next barrier after its own copies have landed.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "attn_core.cuh"
#include "common.cuh"
#include "int4_dot.cuh"
#include "kernels.h"
#include "persistent.h"

namespace w4 {

constexpr int PK_THREADS = 512;
constexpr int PK_WARPS = PK_THREADS / 32;
constexpr int PK_HW = 2 * PK_WARPS;  // half-warps per CTA
constexpr int PK_DEPTH = 16;         // FIFO slots per thread (16 bytes each)
constexpr int PK_AHEAD = 12;         // copies in flight ahead of the computed item (+ up to 4 of the item)
constexpr int PK_ATT_PAGES = 4;      // pages of an attention unit (one slot each)
constexpr int PK_ATT_WARPS = 2 * PK_ATT_PAGES;  // two warps per page: each does P V for half the dims
constexpr int PK_PART = PK_ATT_PAGES * ATT_PAGE;  // tokens per attention partition
constexpr int PK_MAX_K = 18944;      // largest GEMV input the activation staging holds
constexpr size_t PK_RING_BYTES = (size_t)PK_DEPTH * PK_THREADS * 16;
constexpr size_t PK_SFIFO_BYTES = (size_t)PK_DEPTH * PK_THREADS * 4;
constexpr size_t PK_XS_BYTES = ((size_t)PK_MAX_K * 2 + (size_t)(PK_MAX_K / 32) * 4 + 1023) / 1024 * 1024;
constexpr size_t PK_SMEM = PK_RING_BYTES + PK_SFIFO_BYTES + PK_XS_BYTES;
static_assert((size_t)PK_ATT_PAGES * 2 * ATT_SSLICE * 2 <= PK_XS_BYTES, "attention pages reuse the staging area");
static_assert((size_t)PK_ATT_PAGES * 8 * (ATT_D + 2) * 4 <= PK_XS_BYTES, "attention merge reuses the staging area");
// one head's partial attention state in the workspace: 128 weighted-V sums,
// the running max and the sum, padded so every record starts 16-byte aligned
// (the sums are read and written as float4)
constexpr int PK_PREC = ATT_D + 4;
static_assert(PK_AHEAD + 4 <= PK_DEPTH, "an item's copies and the copies ahead of it share the FIFO");

enum PkPhase { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3, PH_LM = 4, PH_END = 5 };

// ---------------------------------------------------------------------------
// Geometry of one GEMV phase for one half-warp.
// ---------------------------------------------------------------------------
struct PkGeo {
  int nr;         // weight rows (chunks per lane) per item: 2, or 4 for gate|up
  int nch;        // 16-byte chunks per weight row
  int ipp;        // items per pair: ceil(nch / 16)
  int p0, np;     // this CTA's pairs [p0, p0 + np)
  int it0, it1;   // this half-warp's items [it0, it1), local to the CTA's run
  int K;          // input width (fp16 elements)
  int N;          // output rows
};

__device__ __forceinline__ int pk_phase_n(const PkArgs& a, int ph) {
  switch (ph) {
    case PH_QKV: return (a.Hq + 2 * a.Hkv) * ATT_D;
    case PH_O: return a.H;
    case PH_GU: return a.I;
    case PH_D: return a.H;
    default: return a.vocab;
  }
}
__device__ __forceinline__ int pk_phase_k(const PkArgs& a, int ph) {
  switch (ph) {
    case PH_O: return a.Hq * ATT_D;
    case PH_D: return a.I;
    default: return a.H;
  }
}

__device__ __forceinline__ PkGeo pk_geo(const PkArgs& a, int ph, int hw_id) {
  PkGeo g;
  g.N = pk_phase_n(a, ph);
  g.K = pk_phase_k(a, ph);
  g.nr = ph == PH_GU ? 4 : 2;
  g.nch = ph == PH_LM ? g.K / 8 : g.K / 32;
  g.ipp = (g.nch + 15) / 16;
  const int pairs = g.N / 2;
  const int c = blockIdx.x, G = gridDim.x;
  g.p0 = (int)((long)c * pairs / G);
  g.np = (int)((long)(c + 1) * pairs / G) - g.p0;
  const int T = g.np * g.ipp;
  g.it0 = (int)((long)hw_id * T / PK_HW);
  g.it1 = (int)((long)(hw_id + 1) * T / PK_HW);
  return g;
}
__device__ __forceinline__ int pk_range_start(const PkGeo& g, int hw_id) {
  return (int)((long)hw_id * (g.np * g.ipp) / PK_HW);
}

// Weight row `row` of phase ph in layer L: packed words (int4) and scales.
__device__ __forceinline__ void pk_int4_row(const PkArgs& a, const PkLayer& L, int ph, int row, const uint32_t*& q,
                                            const __half*& s) {
  if (ph == PH_QKV) {
    const int nq = a.Hq * ATT_D, nk = a.Hkv * ATT_D;
    if (row < nq) {
      q = L.wq + (size_t)row * (a.H / 8);
      s = L.sq + (size_t)row * (a.H / 128);
    } else if (row < nq + nk) {
      q = L.wk + (size_t)(row - nq) * (a.H / 8);
      s = L.sk + (size_t)(row - nq) * (a.H / 128);
    } else {
      q = L.wv + (size_t)(row - nq - nk) * (a.H / 8);
      s = L.sv + (size_t)(row - nq - nk) * (a.H / 128);
    }
  } else if (ph == PH_O) {
    q = L.wo + (size_t)row * (a.Hq * ATT_D / 8);
    s = L.so + (size_t)row * (a.Hq * ATT_D / 128);
  } else if (ph == PH_D) {
    q = L.wd + (size_t)row * (a.I / 8);
    s = L.sd + (size_t)row * (a.I / 128);
  } else {  // gate|up: rows 0..N-1 gate, N..2N-1 up
    if (row < a.I) {
      q = L.wg + (size_t)row * (a.H / 8);
      s = L.sg + (size_t)row * (a.H / 128);
    } else {
      q = L.wu + (size_t)(row - a.I) * (a.H / 8);
      s = L.su + (size_t)(row - a.I) * (a.H / 128);
    }
  }
}

// ---------------------------------------------------------------------------
// The issue side of a thread's weight FIFO: walks the step's phases in order
// and copies the chunks this thread will compute, PK_AHEAD copies ahead.
// ---------------------------------------------------------------------------
struct PkIssuer {
  int layer, ph;         // position in the step's stream: phase,
  int it, it1;           // item and end of this half-warp's range,
  int k, nr;             // weight row within the item and rows per item,
  int pair, cb, ipp;     // the item's pair and column block,
  int nch;               // chunks per weight row
  const char* wa;        // the item's chunk in the first row of matrix A (gate, or the only one)
  const char* wb;        //   ... and in matrix B (up); the second row is rowb bytes on
  const char* sa;        // the first row's scale of that chunk (not yet aligned), matrix A
  const char* sb;        //   ... matrix B
  int rowb, srowb;       // bytes per weight row and per scale row
  bool valid;            // the chunk index of this lane exists in the row
  unsigned seq;          // copies issued so far

  __device__ __forceinline__ void load_item(const PkArgs& a, int lr) {
    const int j = 16 * cb + lr;
    valid = j < nch;
    const int jj = valid ? j : 0;
    if (ph == PH_LM) {
      wa = reinterpret_cast<const char*>(a.lm_head + (size_t)(2 * pair) * a.H) + 16 * jj;
      wb = wa;
      return;
    }
    const PkLayer& L = a.layers[layer];
    const uint32_t* q;
    const __half* s;
    pk_int4_row(a, L, ph, 2 * pair, q, s);
    wa = reinterpret_cast<const char*>(q) + 16 * jj;
    sa = reinterpret_cast<const char*>(s + (jj >> 2));
    if (ph == PH_GU) {
      pk_int4_row(a, L, ph, a.I + 2 * pair, q, s);
      wb = reinterpret_cast<const char*>(q) + 16 * jj;
      sb = reinterpret_cast<const char*>(s + (jj >> 2));
    } else {
      wb = wa;
      sb = sa;
    }
  }
  // enter phase `ph` of `layer`: its geometry for this half-warp
  __device__ __forceinline__ bool enter(const PkArgs& a, int hw_id, int lr) {
    const PkGeo g = pk_geo(a, ph, hw_id);
    if (g.it0 >= g.it1) return false;
    it = g.it0;
    it1 = g.it1;
    nr = g.nr;
    ipp = g.ipp;
    nch = g.nch;
    pair = g.p0 + g.it0 / g.ipp;
    cb = g.it0 % g.ipp;
    rowb = ph == PH_LM ? g.K * 2 : g.K / 2;
    srowb = (g.K / 128) * 2;
    k = 0;
    load_item(a, lr);
    return true;
  }
  // first item of the next phase that has one for this half-warp
  __device__ __forceinline__ void next_phase(const PkArgs& a, int hw_id, int lr) {
    while (true) {
      if (ph == PH_LM) {
        ph = PH_END;
        return;
      }
      if (ph == PH_D) {
        ++layer;
        ph = layer < a.n_layers ? PH_QKV : PH_LM;
      } else {
        ++ph;
      }
      if (enter(a, hw_id, lr)) return;
    }
  }
  // the step's first phase (the kernel runs only with n_layers >= 1)
  __device__ __forceinline__ void init(const PkArgs& a, int hw_id, int lr) {
    layer = 0;
    seq = 0;
    ph = PH_QKV;
    if (!enter(a, hw_id, lr)) next_phase(a, hw_id, lr);
  }
  // one copy (or an empty group past the end of the stream)
  __device__ __forceinline__ void issue_one(const PkArgs& a, uint4* ring, uint32_t* sfifo, int tid, int hw_id, int lr) {
    if (ph != PH_END) {
      const unsigned slot = seq & (PK_DEPTH - 1);
      const int odd = k & 1;
      const char* w = ((k & 2) ? wb : wa) + (odd ? rowb : 0);
      cp_async16_zfill(ring + (size_t)slot * PK_THREADS + tid, w, valid);
      if (ph != PH_LM) {
        const char* sp = ((k & 2) ? sb : sa) + (odd ? srowb : 0);
        cp_async4_zfill(sfifo + (size_t)slot * PK_THREADS + tid,
                        reinterpret_cast<const void*>(reinterpret_cast<uintptr_t>(sp) & ~uintptr_t(3)), valid);
      }
      if (++k == nr) {
        k = 0;
        if (++it == it1) {
          next_phase(a, hw_id, lr);
        } else {
          if (++cb == ipp) {
            cb = 0;
            ++pair;
          }
          load_item(a, lr);
        }
      }
    }
    cp_async_commit();
    ++seq;
  }
};

// ---------------------------------------------------------------------------
// Grid barrier: a counter that only grows; barrier j of step s completes when
// it reaches (s * barriers_per_step + j + 1) * gridDim.x (mod 2^32).  Bounded:
// on time-out it raises the abort flag and reports bit 1 of the error word.
// Returns false when the kernel must stop.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __noinline__ bool pk_grid_sync(const PkArgs& a, unsigned target, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    red_release_add(&a.ctl[PK_CTL_BAR], 1u);
    unsigned long long t0 = 0;
    for (unsigned n = 0;; ++n) {
      const unsigned v = ld_acquire_u32(&a.ctl[PK_CTL_BAR]);
      if ((int)(v - target) >= 0) break;
      if (a.wait_limit_ns == 0) {  // test hook: give up at the first wait that is not already over
        atomicOr(a.err_flag, 2);
        atomicExch(&a.ctl[PK_CTL_ABORT], 1u);
        ok = 0;
        break;
      }
      if ((n & 63) == 63) {
        if (ld_acquire_u32(&a.ctl[PK_CTL_ABORT]) != 0u) {
          ok = 0;
          break;
        }
        const unsigned long long t = globaltimer();
        if (t0 == 0) {
          t0 = t;
        } else if (t - t0 > a.wait_limit_ns) {
          atomicOr(a.err_flag, 2);
          atomicExch(&a.ctl[PK_CTL_ABORT], 1u);
          ok = 0;
          break;
        }
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// ---------------------------------------------------------------------------
// Activation staging (one sequence): xs in the nibble order of the int4
// product plus the per-chunk bracket cs, optionally RMS-normalised; or, for
// the fp16 lm_head, plain fp16 (RMS-normalised).
// ---------------------------------------------------------------------------
// x == nullptr stages zeros (a token outside the vocabulary).
__device__ __forceinline__ void pk_stage_int4(const __half* x, const __half* gamma, int K, float eps, uint4* xs,
                                              float* cs, float* red) {
  const int NCH = K >> 5, NG = K >> 3;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (gamma != nullptr && NG <= STAGE_GMAX * PK_THREADS) {
    uint4 xr[STAGE_GMAX], gr[STAGE_GMAX];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      const int g = tid + i * PK_THREADS;
      if (g < NG) {
        xr[i] = x ? __ldcg(reinterpret_cast<const uint4*>(x) + g) : make_uint4(0u, 0u, 0u, 0u);
        gr[i] = __ldg(reinterpret_cast<const uint4*>(gamma) + g);
      }
    }
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      if (tid + i * PK_THREADS < NG) {
        const __half* h = reinterpret_cast<const __half*>(&xr[i]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float v = __half2float(h[e]);
          ss = fmaf(v, v, ss);
        }
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < PK_WARPS; ++w) t += red[w];
    const float rscale = 1.0f / sqrtf(t / (float)K + eps);
#pragma unroll
    for (int i = 0; i < STAGE_GMAX; ++i) {
      const int g = tid + i * PK_THREADS;
      if (i * PK_THREADS + warp * 32 >= NG) break;  // warp-uniform
      const bool active = g < NG;
      __half h[8];
      if (active) {
        const __half* xh = reinterpret_cast<const __half*>(&xr[i]);
        const __half* gh = reinterpret_cast<const __half*>(&gr[i]);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(__half2float(xh[e]) * rscale * __half2float(gh[e]));
      }
      stage_group(xs, cs, NCH, 0, g, h, active);
    }
  } else {
    for (int j = tid; j < NCH; j += PK_THREADS) {
      const uint4* src = reinterpret_cast<const uint4*>(x + 32 * (size_t)j);
      uint4 raw[4];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) raw[wi] = x ? __ldcg(src + wi) : make_uint4(0u, 0u, 0u, 0u);
      float se = 0.f, so = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const __half* h = reinterpret_cast<const __half*>(&raw[wi]);
        uint4 o;
        o.x = pack_h2(h[0], h[4]);
        o.y = pack_h2(h[1], h[5]);
        o.z = pack_h2(h[2], h[6]);
        o.w = pack_h2(h[3], h[7]);
        xs[(size_t)wi * NCH + j] = o;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          se += __half2float(h[e]);
          so += __half2float(h[e + 1]);
        }
      }
      cs[j] = 1032.0f * se + 72.0f * so;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void pk_stage_fp16(const __half* x, const __half* gamma, int K, float eps, uint4* xs,
                                              float* red) {
  const int NG = K >> 3;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float ss = 0.f;
  for (int g = tid; g < NG; g += PK_THREADS) {
    const uint4 raw = x ? __ldcg(reinterpret_cast<const uint4*>(x) + g) : make_uint4(0u, 0u, 0u, 0u);
    const __half* h = reinterpret_cast<const __half*>(&raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float v = __half2float(h[e]);
      ss = fmaf(v, v, ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < PK_WARPS; ++w) t += red[w];
  const float rscale = 1.0f / sqrtf(t / (float)K + eps);
  for (int g = tid; g < NG; g += PK_THREADS) {
    uint4 raw = x ? __ldcg(reinterpret_cast<const uint4*>(x) + g) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 graw = __ldg(reinterpret_cast<const uint4*>(gamma) + g);
    __half* h = reinterpret_cast<__half*>(&raw);
    const __half* gh = reinterpret_cast<const __half*>(&graw);
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(__half2float(h[e]) * rscale * __half2float(gh[e]));
    xs[g] = raw;
  }
  __syncthreads();
}

__device__ __forceinline__ unsigned long long pk_argmax_key(float v, int idx) {
  uint32_t bits = __float_as_uint(v);
  uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

// Shared scratch of the GEMV phases (static shared memory).
struct PkShared {
  float rec[PK_HW][2][4];  // partial sums of cut pairs: [half-warp][first | last pair][row]
  float red[PK_WARPS];
  unsigned long long key[PK_HW];
  int flag;
};

// ---------------------------------------------------------------------------
// Epilogue of one finished pair (v: the sums of its weight rows; add: the
// bias (q|k|v) or residual (o, down) of its two output rows, loaded when the
// pair was started so the load's latency is hidden by the pair's work).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float pk_epi_operand(const PkArgs& a, const PkLayer* L, int ph, int row) {
  if (ph == PH_QKV) {
    const int nq = a.Hq * ATT_D, nk = a.Hkv * ATT_D;
    const __half* b = row < nq ? L->bq : (row < nq + nk ? L->bk : L->bv);
    const int br = row < nq ? row : (row < nq + nk ? row - nq : row - nq - nk);
    return b ? __half2float(__ldg(b + br)) : 0.f;
  }
  if (ph == PH_O) return __half2float(__ldcg(a.x + row));
  if (ph == PH_D) return __half2float(__ldcg(a.h + row));
  return 0.f;
}

__device__ __forceinline__ void pk_epilogue(const PkArgs& a, int ph, int pair, const float (&v)[4],
                                            const float (&add)[2], unsigned long long& key) {
  if (ph == PH_QKV) {
#pragma unroll
    for (int r = 0; r < 2; ++r) a.qkv[2 * pair + r] = __float2half_rn(v[r] + add[r]);
  } else if (ph == PH_O) {
#pragma unroll
    for (int r = 0; r < 2; ++r) a.h[2 * pair + r] = __float2half_rn(v[r] + add[r]);
  } else if (ph == PH_GU) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float gv = __half2float(__float2half_rn(v[r]));
      const float uv = __half2float(__float2half_rn(v[2 + r]));
      a.mlp[2 * pair + r] = __float2half_rn(gv / (1.0f + expf(-gv)) * uv);
    }
  } else if (ph == PH_D) {
#pragma unroll
    for (int r = 0; r < 2; ++r) a.x[2 * pair + r] = __float2half_rn(v[r] + add[r]);
  } else {  // lm_head: logits and the running argmax (lowest index on ties)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = 2 * pair + r;
      if (a.logits) a.logits[row] = __float2half_rn(v[r]);
      key = max(key, pk_argmax_key(v[r], row));
    }
  }
}

// ---------------------------------------------------------------------------
// One GEMV phase: the compute side of the FIFO.  xs holds the staged input.
// Returns this half-warp's lane-0 argmax key (lm_head) through key.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pk_gemv_phase(const PkArgs& a, int ph, int layer, PkIssuer& is, unsigned& cseq,
                                              uint4* ring, uint32_t* sfifo, const uint4* xs, const float* cs,
                                              PkShared& sh, unsigned long long& key) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int hw_id = tid >> 4, lr = lane & 15;
  const unsigned hmask = 0xFFFFu << (lane & 16);
  const PkGeo g = pk_geo(a, ph, hw_id);
  const PkLayer* L = ph == PH_LM ? nullptr : &a.layers[layer];
  const bool int4 = ph != PH_LM;
  const int nr = g.nr, NCH = g.nch;
  const int godd = (g.K >> 7) & 1;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int pair = g.p0 + (g.it1 > g.it0 ? g.it0 / g.ipp : 0);
  int cb = g.it1 > g.it0 ? g.it0 % g.ipp : 0;
  bool whole = cb == 0;  // this half-warp holds the pair's first item
  const bool has_add = ph == PH_QKV || ph == PH_O || ph == PH_D;
  float add[2] = {0.f, 0.f};
  if (has_add && lr == 0 && g.it1 > g.it0) {
    add[0] = pk_epi_operand(a, L, ph, 2 * pair);
    add[1] = pk_epi_operand(a, L, ph, 2 * pair + 1);
  }
  for (int it = g.it0; it < g.it1; ++it) {
    for (int r = 0; r < nr; ++r) is.issue_one(a, ring, sfifo, tid, hw_id, lr);
    cp_async_wait<PK_AHEAD>();
    const int j = 16 * cb + lr;
    if (j < NCH) {
      if (int4) {
        const uint4 x0 = xs[j], x1 = xs[NCH + j], x2 = xs[2 * NCH + j], x3 = xs[3 * NCH + j];
        const float c = cs[j];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (r < nr) {
            const unsigned slot = (cseq + r) & (PK_DEPTH - 1);
            const uint4 w = ring[(size_t)slot * PK_THREADS + tid];
            const uint32_t sw = sfifo[(size_t)slot * PK_THREADS + tid];
            // the scale of chunk j is element j / 4 of its row; the copied word
            // is the aligned 4 bytes around it (rows start 128-byte aligned
            // matrices at row * K/128 elements), so the half is the parity of
            // row * K/128 + j / 4
            float p[4] = {0.f, 0.f, 0.f, 0.f};
            word_dot(p, w.x, x0);
            word_dot(p, w.y, x1);
            word_dot(p, w.z, x2);
            word_dot(p, w.w, x3);
            const uint32_t sel = (uint32_t)(((r & 1) & godd) ^ ((j >> 2) & 1));
            const __half sh16 = __ushort_as_half((unsigned short)(sel ? (sw >> 16) : (sw & 0xFFFFu)));
            acc[r] = fmaf(chunk_sum(p, c), __half2float(sh16), acc[r]);
          }
        }
      } else {
        const uint4 xv = xs[j];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const unsigned slot = (cseq + r) & (PK_DEPTH - 1);
          const uint4 w = ring[(size_t)slot * PK_THREADS + tid];
          fma2_f16_f32(acc[r], w.x, xv.x);
          fma2_f16_f32(acc[r], w.y, xv.y);
          fma2_f16_f32(acc[r], w.z, xv.z);
          fma2_f16_f32(acc[r], w.w, xv.w);
        }
      }
    }
    cseq += nr;
    ++cb;
    const bool pair_done = cb == g.ipp;
    if (pair_done || it == g.it1 - 1) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(hmask, acc[r], o);
      }
      if (lr == 0) {
        if (pair_done && whole) {
          pk_epilogue(a, ph, pair, acc, add, key);
        } else {
          // cut pair: the first pair of this range if it ends here (we hold
          // its last item), else the last pair of this range
          const int slot = pair_done ? 0 : 1;
#pragma unroll
          for (int r = 0; r < 4; ++r) sh.rec[hw_id][slot][r] = acc[r];
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[r] = 0.f;
      if (pair_done) {
        cb = 0;
        ++pair;
        whole = true;
        if (has_add && lr == 0 && it + 1 < g.it1) {
          add[0] = pk_epi_operand(a, L, ph, 2 * pair);
          add[1] = pk_epi_operand(a, L, ph, 2 * pair + 1);
        }
      }
    }
  }
  __syncthreads();
  // cut pairs: the half-warp holding a pair's last item adds the partials of
  // the half-warps before it (in order) to its own and finishes the pair
  if (tid < PK_HW) {
    const int h = tid;
    const PkGeo gh = pk_geo(a, ph, h);
    if (gh.it1 > gh.it0 && gh.it0 % gh.ipp != 0) {
      const int lp = gh.it0 / gh.ipp;          // local pair cut at this range's start
      const int last_item = lp * gh.ipp + gh.ipp - 1;
      if (last_item < gh.it1) {                // this range holds its last item: finish it
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        int h0 = h - 1;
        while (h0 > 0 && pk_range_start(gh, h0) > lp * gh.ipp) --h0;  // first half-warp on the pair
        for (int hh = h0; hh < h; ++hh) {
          const PkGeo gx = pk_geo(a, ph, hh);
          if (gx.it1 <= gx.it0) continue;
#pragma unroll
          for (int r = 0; r < 4; ++r) v[r] += sh.rec[hh][1][r];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) v[r] += sh.rec[h][0][r];
        const int pr = gh.p0 + lp;
        const float ad[2] = {has_add ? pk_epi_operand(a, L, ph, 2 * pr) : 0.f,
                             has_add ? pk_epi_operand(a, L, ph, 2 * pr + 1) : 0.f};
        pk_epilogue(a, ph, pr, v, ad, key);
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Attention: unit u = (kv head u / P, partition u % P) of the one sequence;
// warps 0..PK_ATT_WARPS-1 each take one 16-token page of the partition.
// ---------------------------------------------------------------------------
struct PkAttn {
  int kvh, p, t0, t1;  // unit, its tokens [t0, t1)
  int page;            // this warp's page id (-1: none or outside the pool)
  bool in_use;         // this warp's page slot has a copy in flight
  unsigned parity;     // phase parity of this warp's page barrier
};

// Copies of this warp's page of unit u (lane 0 issues 32 row copies of 256
// bytes into the padded slot; completion on the warp's mbarrier).  Needs the
// generic-proxy accesses of the slot ordered before it by the caller.
__device__ __forceinline__ void pk_att_fetch(const PkArgs& a, const PkLayer& Lw, int u, int L, int warp, int lane,
                                             __half* slot, uint64_t* bar, PkAttn& st) {
  st.kvh = u / a.P;
  st.p = u % a.P;
  st.t0 = st.p * PK_PART;
  st.t1 = min(L, st.t0 + PK_PART);
  st.page = -1;
  st.in_use = false;
  if (warp >= PK_ATT_WARPS) return;
  const int pg_i = warp >> 1;  // the page this warp pair shares
  const int tok0 = st.t0 + pg_i * ATT_PAGE;
  if (tok0 >= st.t1) return;
  const int blk = tok0 / ATT_PAGE;
  const int pg = blk < a.max_blocks ? __ldg(&a.block_table[blk]) : -1;
  if (pg < 0 || pg >= a.num_pages) {
    if (lane == 0 && (warp & 1) == 0) atomicOr(a.err_flag, 1);
    return;
  }
  st.page = pg;
  st.in_use = true;
  if (lane == 0 && (warp & 1) == 0) {  // the even warp of the pair issues the copies
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * ATT_PAGE * ATT_D * 2);
    const size_t off = ((size_t)pg * a.Hkv + st.kvh) * ATT_SLICE;
#pragma unroll 4
    for (int r = 0; r < 2 * ATT_PAGE; ++r) {
      const __half* src = (r < ATT_PAGE ? Lw.k_pool : Lw.v_pool) + off + (size_t)(r % ATT_PAGE) * ATT_D;
      __half* dst = slot + (r < ATT_PAGE ? 0 : ATT_SSLICE) + (r % ATT_PAGE) * ATT_PITCH;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
          "l"(src), "r"(ATT_D * 2), "r"(smem_u32(bar))
          : "memory");
    }
  }
}

// Bounded wait of this warp for its page; false on time-out.
__device__ __forceinline__ bool pk_att_wait(uint64_t* bar, PkAttn& st, unsigned long long limit) {
  if (!st.in_use) return true;
  bool ok = mbar_try_wait(bar, st.parity);
  if (!ok) {
    const unsigned long long t0 = globaltimer();
    while (!ok) {
      for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait(bar, st.parity);
      if (!ok && globaltimer() - t0 > (limit > 0 ? limit : ATT_TIMEOUT_NS)) break;
    }
  }
  if (ok) {
    st.parity ^= 1u;
    st.in_use = false;
  }
  return ok;
}

template <int G>
__device__ __noinline__ bool pk_attention_unit(const PkArgs& a, const PkLayer& Lw, int L, PkAttn& st,
                                                  unsigned char* area, uint64_t* pbar, float (*s_q)[ATT_D],
                                                  __half* s_knew, __half* s_vnew, const float* s_cos,
                                                  const float* s_sin, int* s_last) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pos = L - 1;
  const int kvh = st.kvh;
  // ---- RoPE of this kv head's G query heads and the new k; new v ----------
  {
    const __half* qb = a.qkv + (size_t)kvh * G * ATT_D;
    const __half* kn = a.qkv + (size_t)(a.Hq + kvh) * ATT_D;
    const __half* vn = a.qkv + (size_t)(a.Hq + a.Hkv + kvh) * ATT_D;
    constexpr int NPAIR = (G + 1) * (ATT_D / 2);
    for (int idx = tid; idx < NPAIR; idx += PK_THREADS) {
      const int h = idx / (ATT_D / 2), i = idx % (ATT_D / 2);
      const __half* src = h < G ? qb + h * ATT_D : kn;
      const float x0 = __half2float(__ldcg(src + i)), x1 = __half2float(__ldcg(src + i + ATT_D / 2));
      const float cs = s_cos[i], sn = s_sin[i];
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
    for (int d = tid; d < ATT_D; d += PK_THREADS) s_vnew[d] = __ldcg(vn + d);
  }
  __syncthreads();
  // ---- append the new token (the unit whose partition holds it) ------------
  if (pos >= st.t0 && pos < st.t0 + PK_PART && tid < ATT_D) {
    const int blk = pos / ATT_PAGE;
    const int pg = blk < a.max_blocks ? __ldg(&a.block_table[blk]) : -1;
    if (pg >= 0 && pg < a.num_pages) {
      const size_t off = (((size_t)pg * a.Hkv + kvh) * ATT_PAGE + pos % ATT_PAGE) * ATT_D + tid;
      Lw.k_pool[off] = s_knew[tid];
      Lw.v_pool[off] = s_vnew[tid];
    } else if (tid == 0) {
      atomicOr(a.err_flag, 1);
    }
  }
  // ---- pages: scores, online softmax, P V (warps 0..PK_ATT_WARPS-1) -------
  const int g = lane >> 2, t4 = lane & 3;
  float m_run = -INFINITY, l_run = 0.f;
  float o[8][4];  // this warp's half of the dims
#pragma unroll
  for (int nb = 0; nb < 8; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  bool ok = true;
  const int pg_i = warp >> 1, dh = warp & 1;
  if (warp < PK_ATT_WARPS) {
    uint64_t* bar = pbar + pg_i;
    ok = pk_att_wait(bar, st, a.wait_limit_ns);
    const int tok0 = st.t0 + pg_i * ATT_PAGE;
    if (ok && st.page >= 0) {
      __half* Ks = reinterpret_cast<__half*>(area) + (size_t)pg_i * 2 * ATT_SSLICE;
      __half* Vs = Ks + ATT_SSLICE;
      // the page was fetched before the append: the new token's row comes
      // from the rotated k / new v (each warp of the pair patches the rows
      // it reads: K in full, V in its half of the dims)
      const bool has_new = pos >= tok0 && pos < tok0 + ATT_PAGE;
      const int slot = pos - tok0;
      uint32_t qa[8][2];
      attn_q_frags(s_q, G, g, t4, qa);
      if (has_new) {
        // a private copy of the K row is not needed: both warps write the
        // same values, and each only after its own wait
        *reinterpret_cast<uint2*>(Ks + slot * ATT_PITCH + 4 * lane) = *reinterpret_cast<const uint2*>(s_knew + 4 * lane);
        if (lane < 16)
          *reinterpret_cast<uint2*>(Vs + slot * ATT_PITCH + 64 * dh + 4 * lane) =
              *reinterpret_cast<const uint2*>(s_vnew + 64 * dh + 4 * lane);
        __syncwarp();
      }
      const int nv = min(ATT_PAGE, st.t1 - tok0);
      attn_page_half(Ks, Vs, nv, qa, a.scale_log2, attn_k_off(lane), attn_v_off(lane), t4, dh, m_run, l_run, o);
    }
  }
  if (!ok && lane == 0) {
    atomicOr(a.err_flag, 2);
    atomicExch(&a.ctl[PK_CTL_ABORT], 1u);
  }
  // pages consumed: the area becomes the merge buffer; the outcome is made
  // the same for every thread so the caller's barriers stay matched
  ok = __syncthreads_or(!ok) == 0;
  // ---- merge the warps' states ------------------------------------------------
  float* mo = reinterpret_cast<float*>(area);   // [PK_ATT_PAGES][8][128]
  float* mml = mo + PK_ATT_PAGES * 8 * ATT_D;  // [PK_ATT_PAGES][8][2]
  if (warp < PK_ATT_WARPS && g < G) {
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
      *reinterpret_cast<float2*>(mo + (pg_i * 8 + g) * ATT_D + 64 * dh + 8 * nb + 2 * t4) =
          make_float2(o[nb][0], o[nb][1]);
    if (t4 == 0 && dh == 0) {
      mml[(pg_i * 8 + g) * 2 + 0] = m_run;
      mml[(pg_i * 8 + g) * 2 + 1] = l_run;
    }
  }
  __syncthreads();
  float* part = a.att_part + ((size_t)(kvh * a.P + st.p) * G) * PK_PREC;
  for (int idx = tid; idx < G * (ATT_D / 4); idx += PK_THREADS) {
    const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < PK_ATT_PAGES; ++w) M = fmaxf(M, mml[(w * 8 + h) * 2]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < PK_ATT_PAGES; ++w) {
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
    if (a.P == 1) {
      const float inv = den > 0.f ? 1.f / den : 0.f;
      __half2* dst = reinterpret_cast<__half2*>(a.att + ((size_t)kvh * G + h) * ATT_D + 4 * d4);
      dst[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
      dst[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
    } else {
      *reinterpret_cast<float4*>(part + h * PK_PREC + 4 * d4) = acc;
      if (d4 == 0) {
        part[h * PK_PREC + ATT_D] = M;
        part[h * PK_PREC + ATT_D + 1] = den;
      }
    }
  }
  if (a.P == 1) return ok;
  // ---- the last unit of this kv head to finish merges the P partials -------
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = (atomicAdd(&a.att_tickets[kvh], 1u) == (unsigned)(a.P - 1));
  __syncthreads();
  if (!*s_last) return ok;
  __threadfence();
  const int Pv = min(a.P, (L + PK_PART - 1) / PK_PART);  // partitions with tokens
  float* cw = mo;                  // [G][Pv] maxima, then weights
  float* cl = cw + G * Pv;         // [G][Pv] sums
  const float* base = a.att_part + (size_t)kvh * a.P * G * PK_PREC;
  // every (max, sum) pair in flight at once, then one thread per head
  for (int idx = tid; idx < G * Pv; idx += PK_THREADS) {
    const int h = idx / Pv, j = idx - h * Pv;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + ((size_t)j * G + h) * PK_PREC + ATT_D));
    cw[idx] = ml.x;
    cl[idx] = ml.y;
  }
  __syncthreads();
  if (tid < G) {
    float* mw = cw + tid * Pv;
    const float* lw = cl + tid * Pv;
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
  for (int idx = tid; idx < G * (ATT_D / 4); idx += PK_THREADS) {
    const int h = idx / (ATT_D / 4), d4 = idx % (ATT_D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < Pv; ++j) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + ((size_t)j * G + h) * PK_PREC) + d4);
      const float w = cw[h * Pv + j];
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    __half2* dst = reinterpret_cast<__half2*>(a.att + ((size_t)kvh * G + h) * ATT_D + 4 * d4);
    dst[0] = __floats2half2_rn(acc.x, acc.y);
    dst[1] = __floats2half2_rn(acc.z, acc.w);
  }
  if (tid == 0) a.att_tickets[kvh] = 0u;  // ready for the next layer
  return ok;
}

// ---------------------------------------------------------------------------
// Phase timeline (kernel-timeline builds only): thread 0 of every CTA
// records, per phase, when it started (the previous barrier passed), when
// its staging ended, when its share of the phase was done (it arrives at the
// barrier) and when the barrier passed.  Record tag = 5 * layer + phase
// (0 q|k|v, 1 attention, 2 o, 3 gate|up, 4 down; 5 * layers: lm_head).
// ---------------------------------------------------------------------------
#ifdef W4A16_TRACE
#define PK_NOW(v) v = trace_now()
__device__ __forceinline__ void pk_trace(unsigned tag, unsigned long long t0, unsigned long long t1,
                                         unsigned long long t2, unsigned long long t3) {
  if (threadIdx.x == 0 && g_trace_buf != nullptr) {
    const unsigned int i = atomicAdd(&g_trace_n, 1u);
    if (i < g_trace_cap) {
      unsigned int sm;
      asm volatile("mov.u32 %0, %smid;" : "=r"(sm));
      g_trace_buf[i] = TraceRec{t0, t1, t2, {t3, 0, 0}, tag, (unsigned int)blockIdx.x, sm, 0u};
    }
  }
}
#define PK_TRACE(tag, t0, t1, t2, t3) pk_trace(tag, t0, t1, t2, t3)
#else
#define PK_NOW(v) (void)0
#define PK_TRACE(tag, t0, t1, t2, t3) (void)0
#endif

// ---------------------------------------------------------------------------
// The kernel: one decode step of one sequence.
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(PK_THREADS, 1) w4pg_decode_persistent(const __grid_constant__ PkArgs a) {
  extern __shared__ __align__(16) unsigned char pk_smem[];
  uint4* ring = reinterpret_cast<uint4*>(pk_smem);
  uint32_t* sfifo = reinterpret_cast<uint32_t*>(pk_smem + PK_RING_BYTES);
  unsigned char* area = pk_smem + PK_RING_BYTES + PK_SFIFO_BYTES;  // staging / attention pages / merges
  uint4* xs = reinterpret_cast<uint4*>(area);
  float* cs = reinterpret_cast<float*>(area + (size_t)PK_MAX_K * 2);
  __shared__ PkShared sh;
  __shared__ __align__(8) uint64_t pbar[PK_ATT_PAGES];
  __shared__ __align__(16) float s_q[G][ATT_D];
  __shared__ __align__(16) __half s_knew[ATT_D];
  __shared__ __align__(16) __half s_vnew[ATT_D];
  __shared__ float s_cos[ATT_D / 2], s_sin[ATT_D / 2];
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hw_id = tid >> 4, lr = lane & 15;
  const unsigned nctas = gridDim.x;
  // step state: written by the previous step's kernel (read before the first
  // barrier; the lengths and the step counter are written after the last)
  const unsigned step = __ldcg(&a.ctl[PK_CTL_STEP]);
  const unsigned per_step = 5u * (unsigned)a.n_layers;
  const unsigned bar_base = step * per_step * nctas;
  unsigned nbar = 0;
  const int tok = __ldcg(a.tokens_in);
  const int L = __ldcg(a.context_lens) + 1;  // after this step's append
  const int pos = L - 1;
  const bool tok_ok = tok >= 0 && tok < a.vocab;
  const __half* xe = tok_ok ? a.embed + (size_t)tok * a.H : nullptr;

  if (tid == 0) {
    for (int w = 0; w < PK_ATT_PAGES; ++w) mbar_init(&pbar[w], 1);
    fence_mbar_init();
    if (blockIdx.x == 0) {
      if (!tok_ok) atomicOr(a.err_flag, 1);
      if (L > a.max_context) atomicOr(a.err_flag, 1);
    }
  }
  if (tid < ATT_D / 2) {
    const float ang = __fmul_rn((float)(pos > 0 ? pos : 0), a.inv_freq[tid]);  // the fp32 product
    sincosf(ang, &s_sin[tid], &s_cos[tid]);
  }
  // the residual stream of layer 0 is the embedding row
  if (blockIdx.x == 0) {
    for (int i = tid; i < a.H / 8; i += PK_THREADS)
      reinterpret_cast<uint4*>(a.x)[i] = xe ? __ldg(reinterpret_cast<const uint4*>(xe) + i) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  // the weight FIFO: PK_AHEAD copies in flight before the first item
  PkIssuer is;
  is.init(a, hw_id, lr);
#pragma unroll 1
  for (int i = 0; i < PK_AHEAD; ++i) is.issue_one(a, ring, sfifo, tid, hw_id, lr);
  unsigned cseq = 0;
  unsigned long long nokey = 0ull;  // the projections keep no argmax
  PkAttn st;
  st.parity = 0u;
  st.in_use = false;
  const int n_units = a.Hkv * a.P;
  bool alive = true;

  unsigned long long t_start = 0, t_staged = 0, t_done = 0, t_pass = 0;
  PK_NOW(t_start);
#pragma unroll 1
  for (int l = 0; l < a.n_layers && alive; ++l) {
    const PkLayer& Lw = a.layers[l];
    // ---- RMSNorm + q|k|v --------------------------------------------------
    pk_stage_int4(l == 0 ? xe : a.x, Lw.ln1, a.H, a.eps, xs, cs, sh.red);
    PK_NOW(t_staged);
    pk_gemv_phase(a, PH_QKV, l, is, cseq, ring, sfifo, xs, cs, sh, nokey);
    __syncthreads();  // the staging area is free: fetch this CTA's first attention pages
    int u = blockIdx.x;
    if (u < n_units)
      pk_att_fetch(a, Lw, u, L, warp, lane, reinterpret_cast<__half*>(area) + (size_t)(warp >> 1) * 2 * ATT_SSLICE,
                   pbar + (warp < PK_ATT_WARPS ? warp >> 1 : 0), st);
    PK_NOW(t_done);
    if (!(alive = pk_grid_sync(a, bar_base + (++nbar) * nctas, &sh.flag))) break;
    PK_NOW(t_pass);
    PK_TRACE(5 * l + 0, t_start, t_staged, t_done, t_pass);
    t_start = t_pass;
    // ---- RoPE + append + attention -------------------------------------------
#pragma unroll 1
    for (; u < n_units; u += nctas) {
      if (u != (int)blockIdx.x) {
        __syncthreads();  // the previous unit's merge buffer is no longer read
        pk_att_fetch(a, Lw, u, L, warp, lane, reinterpret_cast<__half*>(area) + (size_t)(warp >> 1) * 2 * ATT_SSLICE,
                     pbar + (warp < PK_ATT_WARPS ? warp >> 1 : 0), st);
      }
      if (!pk_attention_unit<G>(a, Lw, L, st, area, pbar, s_q, s_knew, s_vnew, s_cos, s_sin, &s_last)) break;
      __syncthreads();
    }
    PK_NOW(t_done);
    if (!(alive = pk_grid_sync(a, bar_base + (++nbar) * nctas, &sh.flag))) break;
    PK_NOW(t_pass);
    PK_TRACE(5 * l + 1, t_start, t_start, t_done, t_pass);
    t_start = t_pass;
    // ---- o + residual -------------------------------------------------------
    pk_stage_int4(a.att, nullptr, a.Hq * ATT_D, a.eps, xs, cs, sh.red);
    PK_NOW(t_staged);
    pk_gemv_phase(a, PH_O, l, is, cseq, ring, sfifo, xs, cs, sh, nokey);
    PK_NOW(t_done);
    if (!(alive = pk_grid_sync(a, bar_base + (++nbar) * nctas, &sh.flag))) break;
    PK_NOW(t_pass);
    PK_TRACE(5 * l + 2, t_start, t_staged, t_done, t_pass);
    t_start = t_pass;
    // ---- RMSNorm + gate|up + SiLU-mul ---------------------------------------
    pk_stage_int4(a.h, Lw.ln2, a.H, a.eps, xs, cs, sh.red);
    PK_NOW(t_staged);
    pk_gemv_phase(a, PH_GU, l, is, cseq, ring, sfifo, xs, cs, sh, nokey);
    PK_NOW(t_done);
    if (!(alive = pk_grid_sync(a, bar_base + (++nbar) * nctas, &sh.flag))) break;
    PK_NOW(t_pass);
    PK_TRACE(5 * l + 3, t_start, t_staged, t_done, t_pass);
    t_start = t_pass;
    // ---- down + residual ----------------------------------------------------
    pk_stage_int4(a.mlp, nullptr, a.I, a.eps, xs, cs, sh.red);
    PK_NOW(t_staged);
    pk_gemv_phase(a, PH_D, l, is, cseq, ring, sfifo, xs, cs, sh, nokey);
    PK_NOW(t_done);
    if (!(alive = pk_grid_sync(a, bar_base + (++nbar) * nctas, &sh.flag))) break;
    PK_NOW(t_pass);
    PK_TRACE(5 * l + 4, t_start, t_staged, t_done, t_pass);
    t_start = t_pass;
  }

  if (alive) {
    // ---- final RMSNorm + lm_head + argmax -----------------------------------
    pk_stage_fp16(a.x, a.final_norm, a.H, a.eps, xs, sh.red);
    PK_NOW(t_staged);
    unsigned long long key = 0ull;
    pk_gemv_phase(a, PH_LM, 0, is, cseq, ring, sfifo, xs, cs, sh, key);
    PK_NOW(t_done);
    PK_TRACE(5 * a.n_layers, t_start, t_staged, t_done, t_done);
    // this CTA's best (value, lowest index) key, then the last CTA's reduction
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    if (lane == 0) sh.key[warp] = key;
    __syncthreads();
    if (tid == 0) {
      unsigned long long k = 0ull;
      for (int w = 0; w < PK_WARPS; ++w) k = max(k, sh.key[w]);
      a.lm_keys[blockIdx.x] = k;
      __threadfence();
      s_last = atomicAdd(&a.ctl[PK_CTL_LM_TICKET], 1u) == nctas - 1;
    }
    __syncthreads();
    if (s_last && warp == 0) {
      __threadfence();
      unsigned long long k = 0ull;
      for (unsigned i = lane; i < nctas; i += 32) k = max(k, __ldcg(&a.lm_keys[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
      if (lane == 0) {
        a.tokens_out[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
        a.ctl[PK_CTL_LM_TICKET] = 0u;
      }
    }
    // every CTA read the lengths and the step counter before the first barrier
    if (blockIdx.x == 0 && tid == 0) {
      a.context_lens[0] = L;
      a.ctl[PK_CTL_STEP] = step + 1u;
    }
  }
  // leave with no copy in flight
  cp_async_wait<0>();
  if (warp < PK_ATT_WARPS && st.in_use) (void)pk_att_wait(pbar + (warp >> 1), st, 0);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool persistent_supported(int hidden, int n_q_heads, int n_kv_heads, int head_dim, int inter, int n_layers,
                          int max_context) {
  return head_dim == ATT_D && n_kv_heads >= 1 && n_q_heads == 7 * n_kv_heads && n_layers >= 1 &&
         hidden % 128 == 0 && inter % 128 == 0 && inter <= PK_MAX_K && hidden <= 8192 && hidden <= PK_MAX_K &&
         n_q_heads * head_dim <= PK_MAX_K && max_context >= 1 && max_context <= PK_MAX_CONTEXT;
}

size_t persistent_workspace_bytes(int n_kv_heads, int max_context, int n_layers) {
  const int P = (max_context + PK_PART - 1) / PK_PART;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return up((size_t)n_layers * sizeof(PkLayer)) + up((size_t)n_kv_heads * P * 7 * PK_PREC * 4) +
         up((size_t)n_kv_heads * 4) + up((size_t)1024 * 8) + up((size_t)PK_CTL_WORDS * 4);
}

int launch_persistent(const PkArgs& a, cudaStream_t s) {
  static PerDeviceOnce once;
  static int ok_dev[64] = {};
  auto kern = w4pg_decode_persistent<7>;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PK_SMEM);
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, PK_THREADS, PK_SMEM) == cudaSuccess && bps >= 1)
      ok_dev[device_index() & 63] = 1;
  });
  if (!ok_dev[device_index() & 63])
    return set_error(W4A16_ERR_CUDA, "persistent decode: the kernel does not fit on an SM of this device");
  const int grid = std::min(num_sms(), 1024);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PK_THREADS);
  cfg.dynamicSmemBytes = PK_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "persistent decode launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

}  // namespace w4
