// gemm_tc.cu -- batched-decode W4A16 GEMM (M <= 32 sequences) on the
// 5th-generation tensor cores (tcgen05, accumulator in tensor memory).
//
// With a decode batch of 32 the q/k/v, o, gate/up and down projections
// become real dense contractions, y[m][n] = sum_k x[m][k] * w[n][k]
// ("Архитектурные решения и оптимизации" of the aikraft.ru article fixes the
// symmetric group-wise INT4 weights with group 128; the pages' "maximize
// batch sizes" motivates the batched form).  Swap-AB: the MMA's A operand is a
// 128-row weight tile, its B operand the (up to) 32 activation rows, so
// D[n][m] (128 lanes x 32 columns, fp32) lives in tensor memory.
//
// Per 64-wide K stage, 128 threads dequantise their weight row (int4 codes
// times the fp16 group scale, rounded to fp16) straight into the canonical
// no-swizzle K-major shared-memory layout -- core matrices of 8 rows x 16
// bytes; K-adjacent core matrices 128 B apart, 8-row groups 256 B apart --
// and stage the activations the same way; one thread then issues four
// kind::f16 MMAs (K = 16 each) and commits them to the stage's mbarrier.
// Two stage buffers let the dequant of stage s+1 overlap the MMAs of s.
// Within each 8-wide k group both operands use the order 0,4,1,5,2,6,3,7,
// which is the order the two-nibbles-per-LOP3 unpack produces.
//
// Small-N projections split K across CTAs: each split writes its fp32 tile
// to the workspace and the last split of a tile (atomic ticket) sums them
// and runs the epilogue.  Dense fp16 weights (the batched lm_head) skip the
// dequant and use the natural k order.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "kernels.h"

namespace w4 {

constexpr int TC_M = 128;      // weight rows per tile (MMA M)
constexpr int TC_N = 32;       // batch columns (MMA N)
constexpr int TC_K = 64;       // K per stage
constexpr int TC_THREADS = 128;
constexpr int TC_A_BYTES = TC_M * TC_K * 2;  // 16 KB per matrix per stage
constexpr int TC_B_BYTES = TC_N * TC_K * 2;  // 4 KB per stage
constexpr unsigned long long TC_TIMEOUT_NS = 2000000000ull;

__device__ __forceinline__ unsigned long long tc_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = tc_now();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (tc_now() - t0 > TC_TIMEOUT_NS) return false;
  }
}

// Shared-memory matrix descriptor: no swizzle, K-major, LBO = 128 B between
// K-adjacent core matrices, SBO = 256 B between 8-row groups.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(256 >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor: kind::f16, fp32 accumulate, fp16 A and B, both
// K-major, N = 32, M = 128.
constexpr uint32_t TC_IDESC = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(TC_N >> 3) << 17) |
                              ((uint32_t)(TC_M >> 4) << 24);

// byte offset of (row, 8-wide k group w) of a 64-wide stage in the canonical layout
__device__ __forceinline__ uint32_t tc_off(int row, int w, int slice_bytes) {
  return (uint32_t)((w >> 1) * slice_bytes + (row >> 3) * 256 + (w & 1) * 128 + (row & 7) * 16);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 8 codes of one packed word -> exact fp16 codes q in the order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ uint4 codes_word(uint32_t w) {
  constexpr uint32_t MAGIC = 0x64006400u;      // half2{1024, 1024}
  constexpr uint32_t OFF = 0x64086408u;        // half2{1032, 1032}
  constexpr uint32_t SIXTEENTH = 0x2C002C00u;  // half2{1/16, 1/16}
  constexpr uint32_t M72 = 0xD480D480u;        // half2{-72, -72}
  const uint32_t w8 = w >> 8;
  uint4 o;
  o.x = hsub2(and_or(w, 0x000F000Fu, MAGIC), OFF);                 // q0, q4
  o.y = hfma2_u32(and_or(w, 0x00F000F0u, MAGIC), SIXTEENTH, M72);  // q1, q5
  o.z = hsub2(and_or(w8, 0x000F000Fu, MAGIC), OFF);                // q2, q6
  o.w = hfma2_u32(and_or(w8, 0x00F000F0u, MAGIC), SIXTEENTH, M72); // q3, q7
  return o;
}

// fp16 x0..x7 -> order 0,4,1,5,2,6,3,7
__device__ __forceinline__ uint4 permute_k8(uint4 v) {
  uint4 o;
  o.x = prmt(v.x, v.z, 0x5410);
  o.y = prmt(v.x, v.z, 0x7632);
  o.z = prmt(v.y, v.w, 0x5410);
  o.w = prmt(v.y, v.w, 0x7632);
  return o;
}

template <bool INT4, bool SILU>
__global__ void __launch_bounds__(TC_THREADS) gemm_tc_kernel(const __grid_constant__ TcArgs a) {
  constexpr int NA = SILU ? 2 : 1;  // weight matrices per tile (gate and up)
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sA = smem;                               // [2][NA][TC_A_BYTES]
  unsigned char* sB = smem + 2 * NA * TC_A_BYTES;         // [2][TC_B_BYTES]
  __shared__ __align__(8) uint64_t bars[2];   // stage buffers free again
  __shared__ __align__(8) uint64_t gbars[2];  // a group's MMAs complete (per tensor-memory buffer)
  __shared__ uint32_t tmem_slot;
  __shared__ int s_last;
  __shared__ int s_ok;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int K = a.K, M = a.M, N = a.N;
  const int nst = K / TC_K;                               // stages over the whole K
  const int per_split = ((nst + a.ksplit - 1) / a.ksplit + 1) & ~1;  // even: splits start on a group
  const int ntiles = (N + TC_M - 1) / TC_M;
  const int nwork = ntiles * a.ksplit;
  W4_TRACE_SCOPE(a.tag);

  // tensor memory: NA accumulators of TC_N fp32 columns, allocated with a
  // factor-2 margin (power of two, >= 32 columns)
  constexpr uint32_t TMEM_COLS = 2 * NA * TC_N;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&gbars[0], 1);
    mbar_init(&gbars[1], 1);
    fence_mbar_init();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();

  bool ok = true;
  uint32_t it = 0;  // stages processed by this CTA (selects buffer and mbarrier phase)
  uint32_t gc = 0;  // 128-wide groups processed by this CTA (selects tensor-memory buffer)
  uint32_t issued = 0;  // stages whose MMAs were issued (drained before tensor memory is freed)
  for (int work = blockIdx.x; work < nwork && ok; work += gridDim.x) {
    const int tile = work / a.ksplit, split = work % a.ksplit;
    const int n0 = tile * TC_M;
    const int s_begin = split * per_split, s_end = min(nst, s_begin + per_split);
    // this thread's weight row (A operand row tid)
    const int row = n0 + tid;
    const bool row_ok = row < N;
    const uint32_t* qrow[NA];
    const __half* srow[NA];
    const __half* wrow16 = nullptr;
#pragma unroll
    for (int g = 0; g < NA; ++g) {
      qrow[g] = nullptr;
      srow[g] = nullptr;
    }
    if (row_ok) {
      if (INT4) {
        if (SILU) {
#pragma unroll
          for (int g = 0; g < NA; ++g) {
            qrow[g] = a.seg[g].qw + (size_t)row * (K / 8);
            srow[g] = a.seg[g].s + (size_t)row * (K / 128);
          }
        } else {
          int r = row, si = 0;
#pragma unroll
          for (int k = 0; k < 2; ++k)
            if (si < a.nseg - 1 && r >= a.seg[si].rows) { r -= a.seg[si].rows; ++si; }
          qrow[0] = a.seg[si].qw + (size_t)r * (K / 8);
          srow[0] = a.seg[si].s + (size_t)r * (K / 128);
        }
      } else {
        wrow16 = a.w16 + (size_t)row * K;
      }
    }

    // Per 128-wide group the MMAs accumulate exact codes x activations into
    // one of two tensor-memory buffers; the threads read a group's sums one
    // group later (while the tensor core works on the next group) and add
    // them, times the row's fp32 scale, to registers.
    float acc[NA][TC_N];
#pragma unroll
    for (int g = 0; g < NA; ++g)
#pragma unroll
      for (int j = 0; j < TC_N; ++j) acc[g][j] = 0.f;
    float sc_prev[NA];
#pragma unroll
    for (int g = 0; g < NA; ++g) sc_prev[g] = 0.f;
    auto read_group = [&](uint32_t grp, const float (&scale)[NA]) -> bool {
      // grp: this CTA's running group index; wait for its MMAs, then read
      if (tid == 0) s_ok = tc_wait(&gbars[grp & 1], (grp >> 1) & 1) ? 1 : 0;
      __syncthreads();
      if (!s_ok) return false;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (int g = 0; g < NA; ++g) {
        uint32_t r[32];
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (grp & 1) * (NA * TC_N) + (uint32_t)(g * TC_N);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
            "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
              "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < TC_N; ++j) acc[g][j] = fmaf(__uint_as_float(r[j]), scale[g], acc[g][j]);
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      return true;
    };
    // the row's scales live in the epilogue's lane mapping: thread (warp, lane) owns row n0 + 32 warp + lane
    const int erow = n0 + warp * 32 + lane;
    const __half* esrow[NA];
#pragma unroll
    for (int g = 0; g < NA; ++g) esrow[g] = nullptr;
    if (INT4 && erow < N) {
      if (SILU) {
#pragma unroll
        for (int g = 0; g < NA; ++g) esrow[g] = a.seg[g].s + (size_t)erow * (K / 128);
      } else {
        int r = erow, si = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (si < a.nseg - 1 && r >= a.seg[si].rows) { r -= a.seg[si].rows; ++si; }
        esrow[0] = a.seg[si].s + (size_t)r * (K / 128);
      }
    }

    for (int st = s_begin; st < s_end; ++st, ++it) {
      const int buf = it & 1;
      const int k0 = st * TC_K;
      const bool group_first = (st & 1) == 0, group_last = (st & 1) == 1;
      // the MMAs that last read this buffer (two stages ago) must be done;
      // thread 0 waits and the outcome is shared, so every thread decides alike
      if (it >= 2) {
        if (tid == 0) s_ok = tc_wait(&bars[buf], ((it - 2) >> 1) & 1) ? 1 : 0;
        __syncthreads();
        if (!s_ok) {
          ok = false;
          break;
        }
      }
      unsigned char* A = sA + buf * NA * TC_A_BYTES;
      unsigned char* Bt = sB + buf * TC_B_BYTES;
      // ---- A: this thread's row, 64 k (exact codes, no scale)
#pragma unroll
      for (int g = 0; g < NA; ++g) {
        unsigned char* Ag = A + g * TC_A_BYTES;
        if (INT4) {
          uint4 q0 = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u), q1 = q0;  // code 0
          if (row_ok) {
            q0 = ldg_stream(qrow[g] + k0 / 8);
            q1 = ldg_stream(qrow[g] + k0 / 8 + 4);
          }
          const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int w = 0; w < 8; ++w) *reinterpret_cast<uint4*>(Ag + tc_off(tid, w, TC_M * 32)) = codes_word(wv[w]);
        } else {
#pragma unroll
          for (int w = 0; w < 8; ++w)
            *reinterpret_cast<uint4*>(Ag + tc_off(tid, w, TC_M * 32)) =
                row_ok ? ldg_stream(wrow16 + k0 + 8 * w) : make_uint4(0, 0, 0, 0);
        }
      }
      // ---- B: 32 activation rows x 64 k (two 8-wide chunks per thread)
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c = tid + c2 * TC_THREADS;
        const int m = c >> 3, w = c & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < M) v = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + k0 + 8 * w);
        if (INT4) v = permute_k8(v);
        *reinterpret_cast<uint4*>(Bt + tc_off(m, w, TC_N * 32)) = v;
      }
      float sc_cur[NA];
#pragma unroll
      for (int g = 0; g < NA; ++g) sc_cur[g] = (INT4 && esrow[g]) ? __half2float(esrow[g][st >> 1]) : 1.0f;
      // generic-proxy writes -> visible to the tensor core (async proxy)
      fence_proxy_async_smem();
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncthreads();
      if (tid == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t gbase = tmem + (gc & 1) * (NA * TC_N);
#pragma unroll
        for (int g = 0; g < NA; ++g) {
#pragma unroll
          for (int kk = 0; kk < TC_K / 16; ++kk) {
            const uint64_t ad = tc_desc(smem_u32(A + g * TC_A_BYTES + kk * TC_M * 32));
            const uint64_t bd = tc_desc(smem_u32(Bt + kk * TC_N * 32));
            const uint32_t accum = (!group_first || kk > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(gbase + (uint32_t)(g * TC_N)),
                "l"(ad), "l"(bd), "r"(TC_IDESC), "r"(accum)
                : "memory");
          }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&bars[buf]))
                     : "memory");
        if (group_last)
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           smem_u32(&gbars[gc & 1]))
                       : "memory");
      }
      ++issued;
      if (group_first) {
        // the previous group of this work item (if any) is read now, while
        // the tensor core works on this group
        if (st > s_begin && !read_group(gc - 1, sc_prev)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int g = 0; g < NA; ++g) sc_prev[g] = sc_cur[g];
      }
      if (group_last) ++gc;
    }
    if (!ok) break;
    // ---- the last group of this work item
    const bool has_stages = s_end > s_begin;  // a split past the end of K contributes zeros
    if (has_stages && !read_group(gc - 1, sc_prev)) {
      ok = false;
      break;
    }
    const int orow = erow;  // output row (feature n) of this thread

    bool finish = true;
    if (a.ksplit > 1) {
      // split K: park the partial tile; the last split of the tile sums them
      float* ws = a.ws + ((size_t)tile * a.ksplit + split) * (size_t)(NA * TC_N * TC_M);
#pragma unroll
      for (int g = 0; g < NA; ++g)
#pragma unroll
        for (int j = 0; j < TC_N; ++j) ws[(g * TC_N + j) * TC_M + warp * 32 + lane] = acc[g][j];
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = (atomicAdd(&a.counters[tile], 1u) == (unsigned int)(a.ksplit - 1));
      __syncthreads();
      finish = s_last;
      if (finish) {
        __threadfence();
#pragma unroll
        for (int g = 0; g < NA; ++g)
#pragma unroll
          for (int j = 0; j < TC_N; ++j) acc[g][j] = 0.f;
        for (int sp = 0; sp < a.ksplit; ++sp) {
          const float* wp = a.ws + ((size_t)tile * a.ksplit + sp) * (size_t)(NA * TC_N * TC_M);
#pragma unroll
          for (int g = 0; g < NA; ++g)
#pragma unroll
            for (int j = 0; j < TC_N; ++j) acc[g][j] += __ldcg(&wp[(g * TC_N + j) * TC_M + warp * 32 + lane]);
        }
        if (tid == 0) a.counters[tile] = 0u;  // ready for the next call
      }
    }
    if (finish && orow < N && a.y32 != nullptr) {
#pragma unroll
      for (int j = 0; j < TC_N; ++j)
        if (j < M) a.y32[(size_t)j * a.ldy + orow] = acc[0][j];
    } else if (finish && orow < N) {
      if (SILU) {
#pragma unroll
        for (int j = 0; j < TC_N; ++j) {
          if (j < M) {
            const float g = __half2float(__float2half_rn(acc[0][j]));
            const float u = __half2float(__float2half_rn(acc[NA - 1][j]));
            a.y[(size_t)j * a.ldy + orow] = __float2half_rn(g / (1.0f + expf(-g)) * u);
          }
        }
      } else {
        float bv = 0.f;
        if (INT4) {
          int r = orow, si = 0;
#pragma unroll
          for (int k = 0; k < 2; ++k)
            if (si < a.nseg - 1 && r >= a.seg[si].rows) { r -= a.seg[si].rows; ++si; }
          if (a.seg[si].bias) bv = __half2float(a.seg[si].bias[r]);
        }
#pragma unroll
        for (int j = 0; j < TC_N; ++j) {
          if (j < M) {
            float v = acc[0][j] + bv;
            if (a.residual) v += __half2float(a.residual[(size_t)j * a.ldy + orow]);
            a.y[(size_t)j * a.ldy + orow] = __float2half_rn(v);
          }
        }
      }
    }
    __syncthreads();  // accumulator reads done before the next work item's MMAs
  }
  if (!ok && tid == 0 && a.err_flag) atomicOr(a.err_flag, 2);
  // before freeing tensor memory, no MMA of this CTA may still be in flight
  if (!ok && tid == 0) {
    for (uint32_t x = (issued >= 2 ? issued - 2 : 0); x < issued; ++x) (void)tc_wait(&bars[x & 1], (x >> 1) & 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

size_t tc_workspace_bytes(int N, int ksplit, bool silu) {
  const int ntiles = (N + TC_M - 1) / TC_M;
  const size_t na = silu ? 2 : 1;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return TC_TICKET_BYTES + up((size_t)ntiles * ksplit * na * TC_N * TC_M * 4);
}

void tc_workspace_layout(TcArgs& a, void* ws) {
  a.counters = static_cast<unsigned int*>(ws);
  a.ws = reinterpret_cast<float*>(static_cast<char*>(ws) + TC_TICKET_BYTES);
}

int tc_default_ksplit(int N, int K) {
  const int ntiles = (N + TC_M - 1) / TC_M;
  const int nst = K / TC_K;
  int ks = 1;
  if ((size_t)ntiles * 4 > TC_TICKET_BYTES) return 1;  // more tiles than tickets: no split
  while (ntiles * ks * 2 <= num_sms() * 2 && nst / (ks * 2) >= 8) ks *= 2;
  return ks;
}

int launch_gemm_tc(const TcArgs& a, bool int4, bool silu, cudaStream_t s) {
  if (a.M < 1 || a.M > TC_N) return set_error(W4A16_ERR_SHAPE, "gemm_tc: M=%d outside 1..%d", a.M, TC_N);
  // stages pair into 128-wide groups (the int4 scale group), dense weights too
  if (a.K % 128 != 0) return set_error(W4A16_ERR_SHAPE, "gemm_tc: K=%d not a multiple of 128", a.K);
  if (a.ksplit < 1) return set_error(W4A16_ERR_INVALID_ARG, "gemm_tc: ksplit < 1");
  const int na = silu ? 2 : 1;
  const size_t smem = (size_t)2 * na * TC_A_BYTES + (size_t)2 * TC_B_BYTES + 1024;
  const int ntiles = (a.N + TC_M - 1) / TC_M;
  const int nwork = ntiles * a.ksplit;
  static bool configured = false;  // all three instantiations share one function-pointer type
  if (!configured) {
    cudaFuncSetAttribute(gemm_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    cudaFuncSetAttribute(gemm_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    cudaFuncSetAttribute(gemm_tc_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    configured = true;
  }
  auto pick = [&](auto kern) -> int {
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, TC_THREADS, smem) != cudaSuccess || bps < 1) bps = 1;
    bps = std::min(bps, 4);  // tensor memory: <= 4 x 128 columns per SM of 512
    const int blocks = std::max(1, std::min(nwork, bps * num_sms()));
    cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(TC_THREADS), smem, s, a);
    if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "gemm_tc launch: %s", cudaGetErrorString(e));
    return W4A16_OK;
  };
  if (!int4) return pick(gemm_tc_kernel<false, false>);
  if (silu) return pick(gemm_tc_kernel<true, true>);
  return pick(gemm_tc_kernel<true, false>);
}

}  // namespace w4

// ---------------------------------------------------------------------------
// argmax over fp32 logit rows (lowest index on ties), optional fp16 copy
// ---------------------------------------------------------------------------
namespace w4 {
__global__ void __launch_bounds__(256) argmax_rows_kernel(const float* __restrict__ logits, int V, int32_t* tokens,
                                                          __half* logits16, int tag) {
  W4_TRACE_SCOPE(tag);
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  __shared__ unsigned long long best[8];
  const int b = blockIdx.x;
  const float* row = logits + (size_t)b * V;
  unsigned long long k = 0;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float v = row[i];
    if (logits16) logits16[(size_t)b * V + i] = __float2half_rn(v);
    if (v == v) {  // skip NaN
      uint32_t bits = __float_as_uint(v);
      uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
      const unsigned long long key = ((unsigned long long)ord << 32) | (0xFFFFFFFFu - (uint32_t)i);
      k = max(k, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
  if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = k;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int w = 0; w < 8; ++w) m = max(m, best[w]);
    tokens[b] = m ? (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull)) : -1;
  }
}

int launch_argmax_rows(const float* logits, int B, int V, int32_t* tokens, __half* logits16, cudaStream_t s,
                       int tag) {
  cudaError_t e = launch_pdl(argmax_rows_kernel, dim3(B), dim3(256), 0, s, logits, V, tokens, logits16, tag);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "argmax launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}
}  // namespace w4

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
using namespace w4;

extern "C" size_t w4a16_gemm_workspace_size(int M, int K, int N, int silu) {
  (void)M;
  if (K < 64 || N < 1) return 0;
  return tc_workspace_bytes(N, tc_default_ksplit(N, K), silu != 0);
}

static int tc_common_checks(const uint16_t* x, int M, int K, int N, const uint16_t* y, const void* ws, size_t wsb,
                            int N_silu, int* ksplit) {
  W4_CHECK_ARG(x && y, "w4a16_gemm: null x or y");
  W4_CHECK_ARG(M >= 1 && K >= 1 && N >= 1, "w4a16_gemm: sizes must be positive");
  W4_CHECK_SHAPE(M <= 32, "w4a16_gemm: M=%d > 32", M);
  W4_CHECK_SHAPE(K % 128 == 0, "w4a16_gemm: K=%d must be a multiple of 128", K);
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(y, 128, "y");
  W4_CHECK_ALIGN(ws, 128, "workspace");
  *ksplit = 1;
  if (ws != nullptr) {
    const int ks = tc_default_ksplit(N, K);
    if (wsb >= tc_workspace_bytes(N, ks, N_silu != 0)) *ksplit = ks;
  }
  return W4A16_OK;
}

static void tc_ws(TcArgs& a, void* ws) {
  if (a.ksplit > 1) tc_workspace_layout(a, ws);
}

extern "C" int w4a16_gemm(const uint16_t* x, int M, int K, const uint32_t* qweight, const uint16_t* scales, int N,
                          const uint16_t* bias, const uint16_t* residual, uint16_t* y, void* workspace,
                          size_t workspace_bytes, w4a16_stream_t stream) {
  int ks = 1;
  int rc = tc_common_checks(x, M, K, N, y, workspace, workspace_bytes, 0, &ks);
  if (rc) return rc;
  W4_CHECK_ARG(qweight && scales, "w4a16_gemm: null weights");
  W4_CHECK_ALIGN(qweight, 128, "qweight");
  W4_CHECK_ALIGN(scales, 128, "scales");
  W4_CHECK_ALIGN(bias, 128, "bias");
  W4_CHECK_ALIGN(residual, 128, "residual");
  TcArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.residual = reinterpret_cast<const __half*>(residual);
  a.y = reinterpret_cast<__half*>(y);
  a.seg[0] = {qweight, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(bias), N};
  a.nseg = 1;
  a.M = M;
  a.K = K;
  a.N = N;
  a.ldy = N;
  a.ksplit = ks;
  tc_ws(a, workspace);
  return launch_gemm_tc(a, true, false, (cudaStream_t)stream);
}

extern "C" int w4a16_gemm_silu_mul(const uint16_t* x, int M, int K, const uint32_t* qweight_gate,
                                   const uint16_t* scales_gate, const uint32_t* qweight_up, const uint16_t* scales_up,
                                   int N, uint16_t* y, void* workspace, size_t workspace_bytes,
                                   w4a16_stream_t stream) {
  int ks = 1;
  int rc = tc_common_checks(x, M, K, N, y, workspace, workspace_bytes, 1, &ks);
  if (rc) return rc;
  W4_CHECK_ARG(qweight_gate && scales_gate && qweight_up && scales_up, "w4a16_gemm_silu_mul: null weights");
  W4_CHECK_ALIGN(qweight_gate, 128, "qweight_gate");
  W4_CHECK_ALIGN(qweight_up, 128, "qweight_up");
  W4_CHECK_ALIGN(scales_gate, 128, "scales_gate");
  W4_CHECK_ALIGN(scales_up, 128, "scales_up");
  TcArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.y = reinterpret_cast<__half*>(y);
  a.seg[0] = {qweight_gate, reinterpret_cast<const __half*>(scales_gate), nullptr, N};
  a.seg[1] = {qweight_up, reinterpret_cast<const __half*>(scales_up), nullptr, N};
  a.nseg = 2;
  a.M = M;
  a.K = K;
  a.N = N;
  a.ldy = N;
  a.ksplit = ks;
  tc_ws(a, workspace);
  return launch_gemm_tc(a, true, true, (cudaStream_t)stream);
}

extern "C" int lm_head_logits_batched(const uint16_t* x, int B, int H, const uint16_t* lm_head, int vocab,
                                      float* logits, w4a16_stream_t stream) {
  W4_CHECK_ARG(x && lm_head && logits, "lm_head_logits_batched: null pointer");
  W4_CHECK_ARG(B >= 1 && H >= 1 && vocab >= 1, "lm_head_logits_batched: sizes must be positive");
  W4_CHECK_SHAPE(B <= 32, "lm_head_logits_batched: B=%d > 32", B);
  W4_CHECK_SHAPE(H % 128 == 0, "lm_head_logits_batched: H=%d must be a multiple of 128", H);
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(lm_head, 128, "lm_head");
  W4_CHECK_ALIGN(logits, 128, "logits");
  TcArgs a = {};
  a.x = reinterpret_cast<const __half*>(x);
  a.y32 = logits;
  a.w16 = reinterpret_cast<const __half*>(lm_head);
  a.nseg = 0;
  a.M = B;
  a.K = H;
  a.N = vocab;
  a.ldy = vocab;
  a.ksplit = 1;
  return launch_gemm_tc(a, false, false, (cudaStream_t)stream);
}

extern "C" int argmax_rows(const float* logits, int B, int vocab, int32_t* tokens_out, uint16_t* logits16,
                           w4a16_stream_t stream) {
  W4_CHECK_ARG(logits && tokens_out, "argmax_rows: null pointer");
  W4_CHECK_ARG(B >= 1 && vocab >= 1, "argmax_rows: sizes must be positive");
  return launch_argmax_rows(logits, B, vocab, tokens_out, reinterpret_cast<__half*>(logits16), (cudaStream_t)stream,
                            0);
}
