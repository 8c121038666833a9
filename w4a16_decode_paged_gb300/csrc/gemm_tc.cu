// gemm_tc.cu -- W4A16 GEMM for a batch of rows (decode batches of up to 32
// sequences; the wider row blocks of a prompt) on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// With a decode batch of 32 the q/k/v, o, gate/up and down projections
// become real dense contractions, y[m][n] = sum_k x[m][k] * w[n][k]
// ("Архитектурные решения и оптимизации" of the aikraft.ru article fixes the
// symmetric group-wise INT4 weights with group 128; the pages' "maximize
// batch sizes" motivates the batched form).  Swap-AB: the MMA's A operand is a
// 128-row weight tile, its B operand the NC activation rows (32, or 64 / 128
// for a prompt), so D[n][m] (128 lanes x NC columns, fp32) lives in tensor
// memory.
//
// The weights are streamed once, so the kernel is a bandwidth pipe with
// specialised warps that meet only at mbarriers: a producer warp fills a
// ring of 64-k stages with one bulk-tensor (TMA) copy per operand (the packed
// int4 rows; the activation tile with the 128-byte swizzle the MMA's
// shared-memory descriptor reads), or per-lane 16-byte copies where a weight
// tile would straddle two segments; expander warps turn each row's codes into
// exact fp16 integers (q in [-8, 7]) and store them with tcgen05.st into one
// of NAB tensor-memory A buffers (the MMA reads A from tensor memory, so the
// expanded codes never touch shared memory); one warp issues four kind::f16
// MMAs (K = 16) per weight matrix and stage and commits them to the barriers
// that free the ring slot (and with it the A buffer) and, per group, the
// accumulator buffer; reader warps take the group sums out.
//
// Precision: the MMAs see exact codes and exact fp16 activations (products
// exact, fp32 sums).  Each 128-wide scale group accumulates into its own
// tensor-memory buffer (two alternate); the readers read a group's sums with
// tcgen05.ld as soon as the tensor core has finished the group and add them
// times the row's fp32 scale, so the only roundings are fp32 sums and the
// final fp16 store.
//
// Small-N projections split K across CTAs (split length chosen so the work
// items fill whole waves of CTAs): each split parks its fp32 tile in the
// workspace and the last split of a tile (atomic ticket) sums them and runs
// the epilogue.  Dense fp16 weights (the batched lm_head) are copied into the
// ring in the swizzled layout and used by the MMA as they are.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace w4 {

constexpr int TC_M = 128;      // weight rows per tile (MMA M)
constexpr int TC_N = 32;       // batch columns (MMA N) of the decode-batch shape
constexpr int TC_K = 128;      // K per stage: one scale group
constexpr int TC_KH = 64;      // K of one 128-byte swizzled half of a stage's fp16 tiles
constexpr int TC_ACOLS = 64;   // tensor-memory columns of one A buffer (128 rows x 128 k fp16)
constexpr int TC_EXP_WARPS = 4;                  // warps that expand int4 codes into tensor memory
constexpr int TC_READERS = 256;                  // threads that read the group sums and run the epilogue
constexpr int TC_THREADS_WS = 64 + 32 * TC_EXP_WARPS + TC_READERS;  // + producer warp + MMA warp
constexpr int TC_A_BYTES = TC_M * TC_K * 2;  // 32 KB fp16 A tile per matrix per stage (two halves)
constexpr unsigned long long TC_TIMEOUT_NS = 2000000000ull;

constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// NC: batch columns per tile (the MMA's N).  32 for decode batches; 128
// (one weight matrix) or 64 (gate and up together) for the wide row blocks
// of a prompt, where each weight tile is then read once per NC rows.
// PIPES: pipelines per CTA.  The occupancy calculator allows one CTA of this
// kernel per SM whatever its registers and shared memory, and at NC = 32 one
// MMA warp's issue loop bounds the kernel, so the int4 NC = 32 shapes run two
// complete pipelines (producer, MMA warp, expanders, readers, ring, half the
// tensor memory) per CTA: gate|up with pipeline p on matrix p of every tile
// (COOP, the readers meet in shared memory for SiLU(gate) x up), the other
// projections with the pipelines on alternate work items (IND).
template <bool INT4, bool SILU, int NC>
struct TcShape {
  static constexpr int NA = SILU ? 2 : 1;                                   // weight matrices per tile
  static constexpr int PIPES = (INT4 && NC == 32) ? 2 : 1;
  static constexpr bool COOP = SILU && PIPES == 2;
  static constexpr bool IND = !SILU && PIPES == 2;
  static constexpr int NAP = PIPES == 2 ? 1 : NA;                           // matrices per pipeline
  static constexpr int THREADS = PIPES * TC_THREADS_WS;
  static constexpr uint32_t A_TX = INT4 ? TC_M * (TC_K / 2) : TC_A_BYTES;   // A bytes per matrix per stage
  static constexpr uint32_t A_RAW = NAP * A_TX;                             // A bytes per ring slot
  static constexpr uint32_t B_HALF = NC * TC_KH * 2;                        // one swizzled half of B
  static constexpr uint32_t B_BYTES = NC * TC_K * 2;                        // activation tile per stage
  static constexpr uint32_t SLOT = A_RAW + B_BYTES;
  static constexpr int CPT = NC / 2;                                        // columns per reader thread
  // A buffers in tensor memory (int4): how far code expansion runs ahead of
  // the MMAs, as many as fit (2 to 4) beside a pipeline's 2 accumulators (8
  // measured no faster than 4); each pipeline has 512 / PIPES columns.
  static constexpr int TM_BUDGET = 512 / PIPES;
  static constexpr int NAB_FIT = (TM_BUDGET - 2 * NAP * NC) / (NAP * TC_ACOLS);
  static constexpr int NAB = NAB_FIT < 2 ? 2 : (NAB_FIT > 4 ? 4 : NAB_FIT);
  // tensor memory of a pipeline: 2 accumulators x NAP x NC columns, and
  // (int4) NAB A buffers x NAP x 64 columns of exact codes, rounded up to a
  // power of two
  static constexpr uint32_t TM_P = pow2_at_least(INT4 ? 2 * NAP * NC + NAB * NAP * TC_ACOLS : 2 * NAP * NC);
  static constexpr uint32_t TMEM_COLS = PIPES * TM_P;
  // ring stages per pipeline: as many as the shared memory holds (4 to 12),
  // the weights of that many stages in flight per CTA hide the memory latency
  static constexpr int SMEM_BUDGET = 200 * 1024;
  static constexpr int S_FIT = (int)(SMEM_BUDGET / (PIPES * SLOT));
  static constexpr int S = S_FIT < 4 ? 4 : (S_FIT > 12 ? 12 : S_FIT);
  static_assert(A_RAW % 1024 == 0 && B_HALF % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
  // COOP: the up sums of a tile, fp32 [NC][128], from pipeline 1's readers
  static constexpr uint32_t XCH = COOP ? (uint32_t)NC * TC_M * 4 : 0u;
  static constexpr size_t SMEM = (size_t)PIPES * S * SLOT + XCH + 1024;
  static_assert(NC % 32 == 0 && NC <= 128, "NC: 32, 64 or 128 columns");
  static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");
};

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


// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: a
// stage's rows of 64 fp16 are 128 bytes each, 8-row atoms of 1024 bytes apart
// (SBO); 16-byte chunk c of row r sits at chunk c ^ (r % 8) of the row, so
// the eight rows of a core matrix fall on different banks.  The 16-k slice kk
// of the stage starts 32 kk bytes into the atom (the swizzle applies to the
// absolute address; every stage tile is 1024-byte aligned).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor: kind::f16, fp32 accumulate, fp16 A and B, both
// K-major, N = NC, M = 128.
template <int NC>
constexpr uint32_t tc_idesc() {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(NC >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24);
}

// byte offset of (row, 8-wide k group w) of a 64-wide stage in the swizzled layout
__device__ __forceinline__ uint32_t tc_off(int row, int w) { return (uint32_t)(row * 128 + ((w ^ (row & 7)) << 4)); }

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

// The 8 codes of one packed word (nibble i = element i, offset binary
// u = q + 8) as exact fp16 integers q0..q7 in k order.  A nibble placed in
// the low mantissa bits of 1024 gives 1024 + u; one placed four bits higher
// gives 1024 + 16 u, scaled back by 1/16 -- both exact in fp16.
__device__ __forceinline__ uint4 codes_word(uint32_t w) {
  constexpr uint32_t MAGIC = 0x64006400u;      // half2{1024, 1024}
  constexpr uint32_t OFF = 0x64086408u;        // half2{1032, 1032}
  constexpr uint32_t SIXTEENTH = 0x2C002C00u;  // half2{1/16, 1/16}
  constexpr uint32_t M72 = 0xD480D480u;        // half2{-72, -72}
  const uint32_t w8 = w >> 8;
  const uint32_t q04 = hsub2(and_or(w, 0x000F000Fu, MAGIC), OFF);
  const uint32_t q15 = hfma2_u32(and_or(w, 0x00F000F0u, MAGIC), SIXTEENTH, M72);
  const uint32_t q26 = hsub2(and_or(w8, 0x000F000Fu, MAGIC), OFF);
  const uint32_t q37 = hfma2_u32(and_or(w8, 0x00F000F0u, MAGIC), SIXTEENTH, M72);
  uint4 o;
  o.x = prmt(q04, q15, 0x5410);  // q0 q1
  o.y = prmt(q26, q37, 0x5410);  // q2 q3
  o.z = prmt(q04, q15, 0x7632);  // q4 q5
  o.w = prmt(q26, q37, 0x7632);  // q6 q7
  return o;
}

// Bounded mbarrier wait that also gives up as soon as another role of the
// CTA has given up (*fail set); a wait that runs out sets *fail.
__device__ __forceinline__ bool tcw_wait(uint64_t* bar, uint32_t parity, volatile int* fail,
                                         unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = tc_now();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*fail) return false;
    if (tc_now() - t0 > limit) {
      *fail = 1;
      return false;
    }
  }
}

#ifdef W4A16_TRACE
// Trace builds: per-stage event times of CTA 0 (pipeline 0) of the last
// launch, in SM clock cycles (one SM, so the roles' clocks agree;
// w4a16_trace_tc_timeline):
//   0 producer issued the stage's copies      5 MMA warp at the loop top
//   1 expander: A buffer free                 6 MMA: operands ready
//   2 expander: the stage's copies landed     7 MMA: accumulator buffer free
//   3 expander: codes stored                  8 MMA: fence done
//   4 expander: stage released                9 MMA: MMAs issued
//  10 MMA: commits issued, 11 reader: before the group wait, 12 group done
//  seen, 13 buffer read and released; row 14 by event, once per launch:
//  0 entry, 1 set up, 2 producer past the dependency wait, 3 MMA warp past
//  it, 4 readers' epilogue start, 5 partial stored and ticket taken, 6 split
//  sums added, 7 epilogue end, 8 exit
constexpr int TC_TL_EVENTS = 15, TC_TL_STAGES = 512;
__device__ unsigned long long g_tc_timeline[TC_TL_EVENTS][TC_TL_STAGES];
#define TC_TL(ev, s)                                                              \
  do {                                                                             \
    if (blockIdx.x == 0 && pipe == 0 && (s) < TC_TL_STAGES) g_tc_timeline[ev][s] = clock64(); \
  } while (0)
#define TC_CE(e) TC_TL(14, e)
#else
#define TC_TL(ev, s) \
  do {               \
  } while (0)
#define TC_CE(e) \
  do {           \
  } while (0)
#endif

// One 2-D bulk-tensor (TMA) copy of the box at (c0 innermost, c1) of `map`
// into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Warp roles within a pipeline (14 warps; pipeline p is warps 14p ..
// 14p + 13): warp 0 lane 0 issues the bulk-tensor copies (producer), warp
// 1 lane 0 issues the MMAs, warps 2..5 (the expanders, 128 threads, one
// weight row each) expand the int4 codes of their row into tensor-memory A
// buffers, up to NAB stages ahead of the tensor core, and warps 6..13 (the
// readers, 256 threads: a row and half of the batch columns each) read each
// stage's sums from tensor memory as soon as the tensor core has finished
// the stage and run the epilogue.  A stage is 128 k, one scale group: eight
// MMAs per weight matrix between one barrier wait, one fence and one commit
// of the MMA warp, whose loop is what bounds the kernel at small N.  Stage s
// of a pipeline's work uses its ring slot s % TS, A buffer s % NAB and
// accumulator buffer s % 2.  The roles only meet at the pipeline's mbarriers:
//   full[slot]   the slot's bulk-tensor copies landed            (1 + tx bytes)
//   empty[slot]  expanders done with the raw A, MMAs done        (128 + 1; dense: 1);
//                its phase for stage s also tells the expanders that A
//                buffer s % NAB is free again at stage s + NAB, and the
//                readers that the stage's sums are in tensor memory
//   afull[b]     stage s = b (mod NAB) may start: expanders wrote A buffer b,
//                and readers read accumulator buffer s % 2 of stage s - 2
//                (for s < 2 they arrive at the start)          (128 + 256)
//   gempty[b]    dense only: readers read accumulator buffer b  (256)
template <bool INT4, bool SILU, int NC>
__global__ void __launch_bounds__(TcShape<INT4, SILU, NC>::THREADS, 1)
    w4pg_tc_batch(const __grid_constant__ TcArgs a) {
  using SH = TcShape<INT4, SILU, NC>;
  constexpr int NA = SH::NA;
  constexpr int NAP = SH::NAP;
  constexpr int PIPES = SH::PIPES;
  constexpr bool COOP = SH::COOP;
  constexpr bool IND = SH::IND;
  constexpr int CPT = SH::CPT;
  // The array is declared with the alignment every build guarantees (16
  // bytes): the 1024-byte alignment of the ring (needed by the 128-byte
  // swizzle) is made at run time, as an offset into the array so that the
  // compiler keeps shared-memory loads for it.  (Declaring 1024 here lets
  // the compiler take the offset to be 0, which relocatable builds do not
  // honour.)
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* ring0 = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // [PIPES][TS][A raw | B]
  constexpr int NAB = SH::NAB;
  constexpr int TS = SH::S;  // ring stages per pipeline
  static_assert(NAB < TS, "an A buffer is reused before its ring slot");
  __shared__ __align__(8) uint64_t full_[PIPES][TS], empty_[PIPES][TS], afull_[PIPES][NAB], gempty_[PIPES][2],
      drain_[PIPES];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_last_[PIPES], s_rfail_[PIPES];
  __shared__ volatile int s_fail;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int pipe = PIPES == 2 ? warp / 14 : 0;
  const int lw = warp - 14 * pipe;  // warp within the pipeline
  unsigned char* ring = ring0 + pipe * TS * SH::SLOT;
  float* xch = reinterpret_cast<float*>(ring0 + PIPES * TS * SH::SLOT);  // COOP exchange [NC][128]
  uint64_t* const full = full_[pipe];
  uint64_t* const empty = empty_[pipe];
  uint64_t* const afull = afull_[pipe];
  uint64_t* const gempty = gempty_[pipe];
  uint64_t* const drainp = &drain_[pipe];
  int& s_last = s_last_[pipe];
  int& s_rfail = s_rfail_[pipe];
  const int K = a.K, N = a.N;
  const int nst = K / TC_K, ps = a.per_split, ks = a.ksplit;
  const int ntiles = (N + TC_M - 1) / TC_M;
  const int nwork = ntiles * ks;
  const unsigned long long wl = a.wait_limit_ns;
  W4_TRACE_SCOPE(a.tag);
  if (tid == 0) TC_CE(0);

  constexpr uint32_t TMEM_COLS = SH::TMEM_COLS;
  // a pipeline's columns, from its base: [0, 2 NAP NC) accumulators; then
  // (int4) A buffer ab, matrix g at 2 NAP NC + (ab NAP + g) TC_ACOLS
  constexpr uint32_t TM_A = 2 * NAP * NC;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32) {
    for (int p = 0; p < PIPES; ++p) {
      for (int i = 0; i < TS; ++i) {
        mbar_init(&full_[p][i], 1);
        mbar_init(&empty_[p][i], (INT4 ? 128 : 0) + 1);
      }
      for (int i = 0; i < NAB; ++i) mbar_init(&afull_[p][i], 128 + TC_READERS);
      for (int i = 0; i < 2; ++i) mbar_init(&gempty_[p][i], TC_READERS);
      mbar_init(&drain_[p], 1);
    }
    s_fail = 0;
    fence_mbar_init();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot + (uint32_t)pipe * SH::TM_P;  // this pipeline's columns
  if (tid == 0) TC_CE(1);

  // (work item, stage) cursor over this CTA's work, shared by all roles
  struct Cursor {
    int work, st, end, begin;
  };
  // IND: the pipelines take alternate work items
  const int wstep = IND ? 2 * (int)gridDim.x : (int)gridDim.x;
  const int wfirst = IND ? 2 * (int)blockIdx.x + pipe : (int)blockIdx.x;
  auto c_init = [&](Cursor& c) {
    c.work = wfirst;
    if (c.work < nwork) {
      c.begin = c.st = (c.work % ks) * ps;
      c.end = min(nst, c.begin + ps);
    }
  };
  auto c_next = [&](Cursor& c) {  // returns true when a new work item starts
    if (++c.st < c.end) return false;
    c.work += wstep;
    if (c.work < nwork) {
      c.begin = c.st = (c.work % ks) * ps;
      c.end = min(nst, c.begin + ps);
    }
    return true;
  };

  if (lw == 0) {
    // =========================== producer ===================================
    // Lane 0 copies a stage's weight tiles (int4: 128 rows x 64 bytes of
    // codes; dense: two swizzled 64-k halves) and its activation tile (two
    // swizzled halves); the slot's barrier expects their bytes.
    Cursor cur;
    c_init(cur);
    int tm_map[NAP], tm_row = 0;  // the item's weight map per matrix and its first row in it
    auto item_tma = [&]() {
      const int r0 = (cur.work / ks) * TC_M;
      tm_row = r0;
      if (SILU || !INT4) {
#pragma unroll
        for (int g = 0; g < NAP; ++g) tm_map[g] = COOP ? pipe : g;
      } else {
        int si = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (si < a.nseg - 1 && tm_row >= a.seg[si].rows) { tm_row -= a.seg[si].rows; ++si; }
        tm_map[0] = si;
      }
    };
    auto tma_a = [&](int slot, int st) {
      unsigned char* sa = ring + slot * SH::SLOT;
#pragma unroll
      for (int g = 0; g < NAP; ++g) {
        if (INT4) {
          tma_load_2d(sa + g * SH::A_TX, &a.tm_w[tm_map[g]], st * (TC_K / 8), tm_row, &full[slot]);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sa + h * (TC_A_BYTES / 2), &a.tm_w[tm_map[g]], st * TC_K + h * TC_KH, tm_row, &full[slot]);
        }
      }
    };
    auto tma_b = [&](int slot, int st) {
      unsigned char* sb = ring + slot * SH::SLOT + SH::A_RAW;
#pragma unroll
      for (int h = 0; h < 2; ++h) tma_load_2d(sb + h * SH::B_HALF, &a.tm_x, st * TC_K + h * TC_KH, 0, &full[slot]);
    };
    if (cur.work < nwork) item_tma();
    // prologue: the weights of the first stages before the dependency wait
    int pro_st[TS];
    int npro = 0;
    {
      Cursor c2 = cur;
      for (int i = 0; i < TS && c2.work < nwork; ++i) {
        if (i > 0 && c2.st == c2.begin) break;  // a new item inside the prologue: stop (its rows differ)
        pro_st[i] = c2.st;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[i], SH::A_RAW + SH::B_BYTES);
          tma_a(i, c2.st);
        }
        ++npro;
        c_next(c2);
      }
    }
    pdl_wait_then_trigger();
    W4_TRACE_WAITED();
    if (lane == 0) TC_CE(2);
    if (lane == 0)
      for (int i = 0; i < npro; ++i) tma_b(i, pro_st[i]);
    for (int i = 0; i < npro; ++i)
      if (c_next(cur) && cur.work < nwork) item_tma();
    for (uint32_t s = npro; cur.work < nwork; ++s) {
      const int slot = s % TS;
      if (s >= TS && !tcw_wait(&empty[slot], ((s / TS) - 1) & 1, &s_fail, wl)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[slot], SH::A_RAW + SH::B_BYTES);
        tma_a(slot, cur.st);
        tma_b(slot, cur.st);
        TC_TL(0, s);
      }
      __syncwarp();
      if (c_next(cur) && cur.work < nwork) item_tma();
    }
  } else if (lw == 1) {
    // =========================== MMA issuer =================================
    // The whole warp runs the loop (waits: warp-uniform values); lane 0
    // issues the MMAs and the commits.
    pdl_wait_then_trigger();
    if (lane == 0) TC_CE(3);
    Cursor cur;
    c_init(cur);
    uint32_t s = 0;
    for (; cur.work < nwork; ++s) {
      const int slot = s % TS, ab = s % NAB, gb = s & 1;
      if (lane == 0) TC_TL(5, s);
      // int4: the expanders saw the slot's copies land before they filled A
      // buffer ab, so its barrier (acquired here) covers the B tile too, and
      // the readers' arrivals on it free the accumulator buffer
      bool ok = INT4 ? tcw_wait(&afull[ab], (s / NAB) & 1, &s_fail, wl) : tcw_wait(&full[slot], (s / TS) & 1, &s_fail, wl);
      if (lane == 0) TC_TL(6, s);
      if (!INT4 && s >= 2 && ok) ok = tcw_wait(&gempty[gb], ((s - 2) >> 1) & 1, &s_fail, wl);
      if (lane == 0) TC_TL(7, s);
      if (!__all_sync(0xffffffffu, ok)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (lane == 0) TC_TL(8, s);
      unsigned char* sl = ring + slot * SH::SLOT;
      const uint32_t dbase = tmem + gb * (NAP * NC);
      if (lane == 0) {
        const uint64_t bd0 = tc_desc(smem_u32(sl + SH::A_RAW));
        const uint64_t bd1 = tc_desc(smem_u32(sl + SH::A_RAW + SH::B_HALF));
#pragma unroll
        for (int g = 0; g < NAP; ++g) {
#pragma unroll
          for (int kk = 0; kk < TC_K / 16; ++kk) {
            // 16-k slice kk: half kk / 4 of the swizzled B tile, 32 bytes per slice
            const uint64_t bd = (kk < 4 ? bd0 : bd1) + (uint64_t)(((kk & 3) * 32) >> 4);
            const uint32_t accum = kk > 0 ? 1u : 0u;
            if (INT4) {
              // A (128 x 16 exact codes) from tensor memory: 8 columns per 16 k
              const uint32_t at = tmem + TM_A + (uint32_t)((ab * NAP + g) * TC_ACOLS + kk * 8);
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dbase + (uint32_t)(g * NC)),
                  "r"(at), "l"(bd), "r"(tc_idesc<NC>()), "r"(accum)
                  : "memory");
            } else {
              const uint64_t ad =
                  tc_desc(smem_u32(sl + (kk < 4 ? 0 : TC_A_BYTES / 2))) + (uint64_t)(((kk & 3) * 32) >> 4);
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dbase + (uint32_t)(g * NC)),
                  "l"(ad), "l"(bd), "r"(tc_idesc<NC>()), "r"(accum)
                  : "memory");
            }
          }
        }
        TC_TL(9, s);
        // the ring slot (producer), through it A buffer ab (expanders wait on
        // the slot of the stage NAB back) and the stage's sums (readers)
        tc_commit(&empty[slot]);
        TC_TL(10, s);
      }
      __syncwarp();
      c_next(cur);
    }
    // before tensor memory is freed no MMA may be in flight: one more
    // commit tracks every MMA this thread issued, and its wait ignores an
    // abort elsewhere in the CTA (the MMAs finish on their own; the wait
    // keeps the normal bound)
    if (s > 0) {
      if (lane == 0) tc_commit(drainp);
      __syncwarp();
      (void)tc_wait(drainp, 0);
    }
  } else if (lw < 2 + TC_EXP_WARPS) {
    // =========================== expanders ==================================
    // Each thread expands its weight row's 128 codes per stage (per matrix)
    // into A buffer s % NAB, up to NAB stages ahead of the tensor core.
    pdl_wait_then_trigger();
    if (INT4) {
      const int row_l = 32 * (warp & 3) + lane;  // tensor-memory lanes of this warp's quadrant
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + TM_A;
      // With more than two A buffers the tensor-memory stores of a stage
      // complete while the expanders wait for the next stage, and the stage
      // is released one iteration later; with two, that wait is on the MMAs
      // of the stage before, so the stage is released at once.
      constexpr bool LAZY = NAB > 2;
      auto release = [&](uint32_t ps_) {
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(&afull[ps_ % NAB]);
        mbar_arrive(&empty[ps_ % TS]);
        if (lw == 2 && lane == 0) TC_TL(4, ps_);
      };
      Cursor cur;
      c_init(cur);
      bool pend = false;
      uint32_t s = 0;
      for (; cur.work < nwork; ++s) {
        const int slot = s % TS, ab = s % NAB;
        // the A buffer's previous MMAs are done, the slot's copies landed
        // (the MMA's commit to that stage's ring slot also covers A buffer ab)
        if (s >= NAB && !tcw_wait(&empty[(s - NAB) % TS], ((s - NAB) / TS) & 1, &s_fail, wl)) break;
        if (lw == 2 && lane == 0) TC_TL(1, s);
        if (!tcw_wait(&full[slot], (s / TS) & 1, &s_fail, wl)) break;
        if (lw == 2 && lane == 0) TC_TL(2, s);
        const unsigned char* sl = ring + slot * SH::SLOT;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (LAZY && pend) release(s - 1);
        // exact codes of this row's 128 k per matrix, 64 k (32 columns of
        // fp16 pairs in k order) at a time
#pragma unroll
        for (int g = 0; g < NAP; ++g) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const unsigned char* src = sl + (g * TC_M + row_l) * (TC_K / 2) + h * 32;
            const uint4 r0 = *reinterpret_cast<const uint4*>(src);
            const uint4 r1 = *reinterpret_cast<const uint4*>(src + 16);
            uint4 c[8];
            c[0] = codes_word(r0.x);
            c[1] = codes_word(r0.y);
            c[2] = codes_word(r0.z);
            c[3] = codes_word(r0.w);
            c[4] = codes_word(r1.x);
            c[5] = codes_word(r1.y);
            c[6] = codes_word(r1.z);
            c[7] = codes_word(r1.w);
            const uint32_t ta = lane_base + (uint32_t)((ab * NAP + g) * TC_ACOLS + h * 32);
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
                "r"(c[0].x), "r"(c[0].y), "r"(c[0].z), "r"(c[0].w), "r"(c[1].x), "r"(c[1].y), "r"(c[1].z), "r"(c[1].w),
                "r"(c[2].x), "r"(c[2].y), "r"(c[2].z), "r"(c[2].w), "r"(c[3].x), "r"(c[3].y), "r"(c[3].z), "r"(c[3].w),
                "r"(c[4].x), "r"(c[4].y), "r"(c[4].z), "r"(c[4].w), "r"(c[5].x), "r"(c[5].y), "r"(c[5].z), "r"(c[5].w),
                "r"(c[6].x), "r"(c[6].y), "r"(c[6].z), "r"(c[6].w), "r"(c[7].x), "r"(c[7].y), "r"(c[7].z), "r"(c[7].w)
                : "memory");
          }
        }
        if (lw == 2 && lane == 0) TC_TL(3, s);
        if (!LAZY) release(s);
        pend = true;
        c_next(cur);
      }
      if (LAZY && pend && cur.work >= nwork) release(s - 1);
    }
  } else {
    // =========================== accumulators ===============================
    // Stage by stage (one scale group each, in the order the tensor core
    // finishes them): tcgen05.ld of this row's CPT columns of the stage's
    // buffer, times the group's scale into fp32 registers; at the end of a
    // work item the epilogue.  They run up to one stage behind the tensor core.
    pdl_wait_then_trigger();
    const int r = tid - TC_THREADS_WS * pipe - 64 - 32 * TC_EXP_WARPS;   // 0..255
    const int half = r >> 7;                      // batch columns CPT h .. CPT h + CPT - 1
    const int row_l = 32 * (warp & 3) + lane;     // tensor-memory lanes of this warp's quadrant
    const int M = a.M;
    Cursor cur;
    c_init(cur);
    // stages of this CTA's work: the readers free the accumulator buffer of
    // stage s + 2 after reading stage s, and those of stages 0 and 1 now
    uint32_t nstages = 0;
    for (int w = wfirst; w < nwork; w += wstep) nstages += (uint32_t)(min(nst, (w % ks) * ps + ps) - (w % ks) * ps);
    // the readers' own barrier (one per pipeline; 3 joins both pipelines' readers)
    auto rsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + pipe), "n"(TC_READERS) : "memory"); };
    if (INT4) {
      if (nstages > 0) mbar_arrive(&afull[0]);
      if (nstages > 1) mbar_arrive(&afull[1 % NAB]);
    }
    const __half* sp[NAP];
    bool rok = false;
    __half sreg[NAP];  // the scales of the group being read
    float acc[NA][CPT];
#pragma unroll
    for (int g = 0; g < NA; ++g)
#pragma unroll
      for (int j = 0; j < CPT; ++j) acc[g][j] = 0.f;

    // the scales of tile `tile`, row row_l
    auto scale_rows = [&](int tile) {
      const int row = tile * TC_M + row_l;
      rok = row < N;
      const int rr = rok ? row : 0;
      if (SILU) {
#pragma unroll
        for (int g = 0; g < NAP; ++g) sp[g] = a.seg[COOP ? pipe : g].s + (size_t)rr * (K / 128);
      } else if (INT4) {
        int q = rr, si = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (si < a.nseg - 1 && q >= a.seg[si].rows) { q -= a.seg[si].rows; ++si; }
        sp[0] = a.seg[si].s + (size_t)q * (K / 128);
      }
    };

    // add tensor-memory stage `st_i` (this row, CPT columns) times the scales
    auto tm_read = [&](uint32_t st_i) {
      if (r == 0) TC_TL(11, st_i);
      const bool ok = __all_sync(0xffffffffu, tcw_wait(&empty[st_i % TS], (st_i / TS) & 1, &s_fail, wl));
      if (r == 0) TC_TL(12, st_i);
      if (ok) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int g = 0; g < NAP; ++g) {
          const float sc = INT4 ? __half2float(sreg[g]) : 1.0f;
#pragma unroll
          for (int c0 = 0; c0 < CPT; c0 += 16) {
            uint32_t v[16];
            const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (st_i & 1) * (NAP * NC) +
                                   (uint32_t)(g * NC + half * CPT + c0);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[g][c0 + j] = fmaf(__uint_as_float(v[j]), sc, acc[g][c0 + j]);
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      }
      if (!INT4) mbar_arrive(&gempty[st_i & 1]);
      else if (st_i + 2 < nstages) mbar_arrive(&afull[(st_i + 2) % NAB]);
      if (r == 0) TC_TL(13, st_i);
    };

    auto epilogue = [&](int work) {
      const int tile = work / ks, split = work % ks;
      const int row = tile * TC_M + row_l;
      bool finish = true;
      if (r == 0) TC_CE(4);
      if (ks > 1) {
        float* wsp = a.ws + ((size_t)tile * ks + split) * (size_t)(NA * NC * TC_M);
#pragma unroll
        for (int g = 0; g < NA; ++g)
#pragma unroll
          for (int j = 0; j < CPT; ++j) wsp[(g * NC + half * CPT + j) * TC_M + row_l] = acc[g][j];
        __threadfence();
        rsync();
        if (r == 0) s_last = (atomicAdd(&a.counters[tile], 1u) == (unsigned int)(ks - 1));
        rsync();
        if (r == 0) TC_CE(5);
        finish = s_last;
        if (finish) {
          __threadfence();
#pragma unroll
          for (int g = 0; g < NA; ++g)
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[g][j] = 0.f;
          for (int spl = 0; spl < ks; ++spl) {
            const float* wp = a.ws + ((size_t)tile * ks + spl) * (size_t)(NA * NC * TC_M);
#pragma unroll
            for (int g = 0; g < NA; ++g)
#pragma unroll
              for (int j = 0; j < CPT; ++j) acc[g][j] += __ldcg(&wp[(g * NC + half * CPT + j) * TC_M + row_l]);
          }
          if (r == 0) a.counters[tile] = 0u;  // ready for the next call
          if (r == 0) TC_CE(6);
        }
      }
      if (!finish || row >= N) return;
      if (a.y32 != nullptr) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int m = half * CPT + j;
          if (m < M) a.y32[(size_t)m * a.ldy + row] = acc[0][j];
        }
      } else if (SILU) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int m = half * CPT + j;
          if (m < M) {
            const float gv = __half2float(__float2half_rn(acc[0][j]));
            const float u = __half2float(__float2half_rn(acc[NA - 1][j]));
            a.y[(size_t)m * a.ldy + row] = __float2half_rn(gv / (1.0f + expf(-gv)) * u);
          }
        }
      } else {
        float bv = 0.f;
        if (INT4) {
          int rr = row, si = 0;
#pragma unroll
          for (int k = 0; k < 2; ++k)
            if (si < a.nseg - 1 && rr >= a.seg[si].rows) { rr -= a.seg[si].rows; ++si; }
          if (a.seg[si].bias) bv = __half2float(a.seg[si].bias[rr]);
        }
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int m = half * CPT + j;
          if (m < M) {
            float v = acc[0][j] + bv;
            if (a.residual) v += __half2float(a.residual[(size_t)m * a.ldy + row]);
            a.y[(size_t)m * a.ldy + row] = __float2half_rn(v);
          }
        }
      }
    };

    uint32_t grp = 0;  // stages read so far (all items): buffer grp & 1
    while (cur.work < nwork) {
      if (INT4) scale_rows(cur.work / ks);
      const int g0 = cur.begin, ng = cur.end - cur.begin;  // one scale group per stage
      // scales of the next two groups in flight (requested two groups ahead)
      __half snext[NAP], snext2[NAP];
#pragma unroll
      for (int g = 0; g < NAP; ++g) {
        snext[g] = (INT4 && rok) ? sp[g][g0] : __float2half(0.f);
        snext2[g] = (INT4 && rok && ng > 1) ? sp[g][g0 + 1] : __float2half(0.f);
      }
      for (int gi = 0; gi < ng; ++gi, ++grp) {
#pragma unroll
        for (int g = 0; g < NAP; ++g) {
          sreg[g] = snext[g];
          snext[g] = snext2[g];
          if (INT4 && rok && gi + 2 < ng) snext2[g] = sp[g][g0 + gi + 2];
        }
        tm_read(grp);
      }
      if (COOP) {
        // pipeline 1's up sums to pipeline 0's readers, which run the epilogue
        if (pipe == 1) {
#pragma unroll
          for (int j = 0; j < CPT; ++j) xch[(half * CPT + j) * TC_M + row_l] = acc[0][j];
        }
        asm volatile("bar.sync 3, %0;" ::"n"(2 * TC_READERS) : "memory");
        if (pipe == 0) {
#pragma unroll
          for (int j = 0; j < CPT; ++j) acc[NA - 1][j] = xch[(half * CPT + j) * TC_M + row_l];
        }
        asm volatile("bar.sync 3, %0;" ::"n"(2 * TC_READERS) : "memory");
      }
      if (!COOP || pipe == 0) epilogue(cur.work);
      if (r == 0) TC_CE(7);
#pragma unroll
      for (int g = 0; g < NA; ++g)
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[g][j] = 0.f;
      if (r == 0) s_rfail = s_fail;
      rsync();
      // both COOP pipelines run every item (their exchange barriers must meet);
      // after a failure their waits give up at once
      if (s_rfail && !COOP) break;
      cur.work += wstep;
      if (cur.work < nwork) {
        cur.begin = cur.st = (cur.work % ks) * ps;
        cur.end = min(nst, cur.begin + ps);
      }
    }
  }
  __syncthreads();
  if (tid == 0) TC_CE(8);
  if (s_fail && tid == 0 && a.err_flag) atomicOr(a.err_flag, 2);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_slot), "r"(TMEM_COLS) : "memory");
}

int tc_cols(int M, bool int4, bool silu) {
  if (M <= TC_N || !int4) return TC_N;
  return silu ? 64 : 128;
}

int tc_max_rows(bool int4, bool silu) { return int4 ? (silu ? 64 : 128) : TC_N; }

size_t tc_workspace_bytes(int N, int ksplit, bool silu, int nc) {
  const int ntiles = (N + TC_M - 1) / TC_M;
  const size_t na = silu ? 2 : 1;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return TC_TICKET_BYTES + up((size_t)ntiles * ksplit * na * nc * TC_M * 4);
}

void tc_workspace_layout(TcArgs& a, void* ws) {
  a.counters = static_cast<unsigned int*>(ws);
  a.ws = reinterpret_cast<float*>(static_cast<char*>(ws) + TC_TICKET_BYTES);
}

template <bool INT4, bool SILU, int NC>
static int tc_ctas_per_sm() {
  using SH = TcShape<INT4, SILU, NC>;
  static PerDeviceOnce once;
  static int cached[64] = {};
  once_per_device(once, [] {
    auto kern = w4pg_tc_batch<INT4, SILU, NC>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SH::SMEM);
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, SH::THREADS, SH::SMEM) != cudaSuccess || bps < 1)
      bps = 1;
    // tensor memory: 512 columns per SM
    cached[device_index() & 63] = std::max(1, std::min(bps, (int)(512 / SH::TMEM_COLS)));
  });
  return cached[device_index() & 63];
}

static int tc_slots(bool int4, bool silu, int nc) {
  int per;
  if (!int4) per = tc_ctas_per_sm<false, false, TC_N>();
  else if (nc == TC_N) per = silu ? tc_ctas_per_sm<true, true, TC_N>() : tc_ctas_per_sm<true, false, TC_N>() * 2;
  else per = silu ? tc_ctas_per_sm<true, true, 64>() : tc_ctas_per_sm<true, false, 128>();
  return per * num_sms();  // work items in flight (the two pipelines of an IND CTA take one each)
}

// Split of K: the split length (in stages, each a scale group) that
// minimises waves x (stages per item + a per-item overhead of ~2 stages)
// over the CTAs that fit on the GPU.
void tc_plan(int N, int K, bool int4, bool silu, bool allow_split, int* ksplit, int* per_split, int nc) {
  const int ntiles = (N + TC_M - 1) / TC_M;
  const int nst = K / TC_K;
  const int slots = tc_slots(int4, silu, nc);
  int best_ps = nst, best_ks = 1;
  long best = -1;
  for (int p = nst; p >= 1; --p) {
    const int k = (nst + p - 1) / p;
    if (k > 1 && (!allow_split || (size_t)ntiles * 4 > TC_TICKET_BYTES)) continue;
    const long items = (long)ntiles * k;
    const long waves = (items + slots - 1) / slots;
    const long cost = waves * (p + 2);
    if (best < 0 || cost < best) {
      best = cost;
      best_ps = p;
      best_ks = k;
    }
  }
  *ksplit = best_ks;
  *per_split = best_ps;
}

// Bound of the persistent decode kernel's grid-barrier waits (the test hook
// below changes it).  The tensor-core GEMM always keeps its own 2 s bound:
// when one of its roles gives up, the others still run to the end of their
// work item against shared-memory and tensor-memory buffers the tensor core
// may be using, so its abort is only a last resort, not something to trigger.
static std::atomic<unsigned long long> g_wait_limit_ns{TC_TIMEOUT_NS};
unsigned long long tc_wait_limit_ns() { return g_wait_limit_ns.load(); }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null if the driver does not provide it.
static PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over rows of `inner` elements, `row_bytes` apart; boxes of
// box_inner x box_rows (rows past the end read as zeros)
static bool tma_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto enc = tma_encoder();
  if (enc == nullptr || base == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the launch's operands: activations and dense weights in
// swizzled 64-k halves, int4 codes in 128-row x 64-byte boxes.  False when
// the driver gives no encoder or an operand does not fit the boxes (a
// 128-row weight tile across two segments).
static bool tc_tensor_maps(TcArgs& a, bool int4, bool silu, int nc) {
  bool ok = tma_map_2d(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.M,
                       (uint64_t)a.K * 2, TC_KH, (uint32_t)nc, CU_TENSOR_MAP_SWIZZLE_128B);
  if (int4) {
    const int nm = silu ? 2 : a.nseg;
    for (int i = 0; i + 1 < nm && !silu; ++i) ok = ok && a.seg[i].rows % TC_M == 0;
    for (int i = 0; i < nm && ok; ++i)
      ok = tma_map_2d(&a.tm_w[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.seg[i].qw, (uint64_t)a.K / 8,
                      (uint64_t)a.seg[i].rows, (uint64_t)a.K / 2, TC_K / 8, TC_M, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    ok = ok && tma_map_2d(&a.tm_w[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.w16, (uint64_t)a.K, (uint64_t)a.N,
                          (uint64_t)a.K * 2, TC_KH, TC_M, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  return ok;
}

#ifdef W4A16_TRACE
// trace builds: occupancy of each GEMM shape, 16 ints per shape (raw CTAs per
// SM from the occupancy calculator, its error code, tensor-memory columns,
// dynamic shared memory bytes, registers per thread, static shared memory,
// CTAs per SM without dynamic shared memory, shared memory per SM, registers
// and threads per SM, the kernel's thread limit, CTAs per SM at 320 and 224
// threads, local memory) for <int4,silu,nc> = <1,0,32>, <1,1,32>,
// <1,0,128>, <1,1,64>, <0,0,32>
template <bool INT4, bool SILU, int NC>
static void tc_occ(int* o) {
  using SH = TcShape<INT4, SILU, NC>;
  auto kern = w4pg_tc_batch<INT4, SILU, NC>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SH::SMEM);
  int bps = -1;
  o[1] = (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, SH::THREADS, SH::SMEM);
  o[0] = bps;
  o[2] = (int)SH::TMEM_COLS;
  o[3] = (int)SH::SMEM;
  cudaFuncAttributes fa = {};
  cudaFuncGetAttributes(&fa, kern);
  o[4] = fa.numRegs;
  o[5] = (int)fa.sharedSizeBytes;
  int b0 = -1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, kern, SH::THREADS, 0);
  o[6] = b0;
  int smpm = 0;
  cudaDeviceGetAttribute(&smpm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, 0);
  o[7] = smpm;
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxRegistersPerMultiprocessor, 0);
  o[8] = v;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxThreadsPerMultiProcessor, 0);
  o[9] = v;
  o[10] = fa.maxThreadsPerBlock;
  int b1 = -1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, kern, 320, 0);
  o[11] = b1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, kern, 224, 0);
  o[12] = b1;
  o[13] = (int)fa.localSizeBytes;
}
extern "C" W4A16_API int w4a16_trace_tc_occupancy(int* out) {
  tc_occ<true, false, 32>(out);
  tc_occ<true, true, 32>(out + 16);
  tc_occ<true, false, 128>(out + 32);
  tc_occ<true, true, 64>(out + 48);
  tc_occ<false, false, 32>(out + 64);
  return 0;
}

// trace builds: copy CTA 0's per-stage event times of the last GEMM launch
extern "C" W4A16_API int w4a16_trace_tc_timeline(unsigned long long* host_out, int n) {
  const size_t bytes = std::min((size_t)n, (size_t)TC_TL_EVENTS * TC_TL_STAGES) * sizeof(unsigned long long);
  return cudaMemcpyFromSymbol(host_out, g_tc_timeline, bytes) == cudaSuccess ? 0 : 4;
}
#endif

int launch_gemm_tc(const TcArgs& a_in, bool int4, bool silu, cudaStream_t s) {
  TcArgs a = a_in;
  a.wait_limit_ns = TC_TIMEOUT_NS;
  const int maxm = tc_max_rows(int4, silu);
  if (a.M < 1 || a.M > maxm) return set_error(W4A16_ERR_SHAPE, "gemm_tc: M=%d outside 1..%d", a.M, maxm);
  const int nc = tc_cols(a.M, int4, silu);
  // a stage is one 128-wide group (the int4 scale group), dense weights too
  if (a.K % 128 != 0) return set_error(W4A16_ERR_SHAPE, "gemm_tc: K=%d not a multiple of 128", a.K);
  if (!tc_tensor_maps(a, int4, silu, nc))
    return set_error(W4A16_ERR_SHAPE, "gemm_tc: no tensor maps for the operands (weight segments must be "
                     "multiples of 128 rows, rows 16-byte aligned)");
  if (a.ksplit < 1) return set_error(W4A16_ERR_INVALID_ARG, "gemm_tc: ksplit < 1");
  const int nst = a.K / TC_K;
  if (a.per_split <= 0) a.per_split = (nst + a.ksplit - 1) / a.ksplit;
  if ((long)a.per_split * (a.ksplit - 1) >= nst || (long)a.per_split * a.ksplit < nst)
    return set_error(W4A16_ERR_INVALID_ARG, "gemm_tc: split of %d stages x %d does not tile %d stages", a.per_split,
                     a.ksplit, nst);
  const int ntiles = (a.N + TC_M - 1) / TC_M;
  const int nwork = ntiles * a.ksplit;
  auto go = [&](auto kern, auto shape, int per_sm) -> int {
    using SH = decltype(shape);
    const int items_per_cta = SH::IND ? 2 : 1;
    const int blocks = std::max(1, std::min((nwork + items_per_cta - 1) / items_per_cta, per_sm * num_sms()));
    cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(SH::THREADS), SH::SMEM, s, a);
    if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "gemm_tc launch: %s", cudaGetErrorString(e));
    return W4A16_OK;
  };
  if (!int4) return go(w4pg_tc_batch<false, false, TC_N>, TcShape<false, false, TC_N>{},
                       tc_ctas_per_sm<false, false, TC_N>());
  if (nc == TC_N) {
    if (silu) return go(w4pg_tc_batch<true, true, TC_N>, TcShape<true, true, TC_N>{}, tc_ctas_per_sm<true, true, TC_N>());
    return go(w4pg_tc_batch<true, false, TC_N>, TcShape<true, false, TC_N>{}, tc_ctas_per_sm<true, false, TC_N>());
  }
  if (silu) return go(w4pg_tc_batch<true, true, 64>, TcShape<true, true, 64>{}, tc_ctas_per_sm<true, true, 64>());
  return go(w4pg_tc_batch<true, false, 128>, TcShape<true, false, 128>{}, tc_ctas_per_sm<true, false, 128>());
}

}  // namespace w4

// ---------------------------------------------------------------------------
// argmax over fp32 logit rows (lowest index on ties), optional fp16 copy
// ---------------------------------------------------------------------------
namespace w4 {
// One cluster of AM_CL CTAs per row: each CTA takes a contiguous slice of
// the row (eight loads in flight per thread), the slice maxima meet in the
// shared memory of CTA 0 of the cluster.  Keys order by value, then by the
// lower index.
constexpr int AM_CL = 8;
constexpr int AM_U = 8;
__device__ __forceinline__ void st_dsmem_u64(unsigned long long* p, int rank, unsigned long long v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}
__global__ void __cluster_dims__(AM_CL, 1, 1) __launch_bounds__(256)
    w4pg_argmax_rows(const float* __restrict__ logits, int V, int32_t* tokens, __half* logits16, int tag) {
  W4_TRACE_SCOPE(tag);
  pdl_wait_then_trigger();
  W4_TRACE_WAITED();
  __shared__ unsigned long long best[8];
  __shared__ unsigned long long cl_best[AM_CL];
  const int b = blockIdx.y, rank = blockIdx.x;
  const int per = (V + AM_CL - 1) / AM_CL;
  const int lo = rank * per, hi = min(V, lo + per);
  const float* row = logits + (size_t)b * V;
  unsigned long long k = 0;
  for (int i0 = lo + threadIdx.x; i0 < hi; i0 += 256 * AM_U) {
    float v[AM_U];
#pragma unroll
    for (int u = 0; u < AM_U; ++u) {
      const int i = i0 + u * 256;
      v[u] = i < hi ? row[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < AM_U; ++u) {
      const int i = i0 + u * 256;
      if (i < hi) {
        if (logits16) logits16[(size_t)b * V + i] = __float2half_rn(v[u]);
        if (v[u] == v[u]) {  // skip NaN
          const uint32_t bits = __float_as_uint(v[u]);
          const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
          k = max(k, ((unsigned long long)ord << 32) | (0xFFFFFFFFu - (uint32_t)i));
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
  if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = k;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int w = 0; w < 8; ++w) m = max(m, best[w]);
    st_dsmem_u64(&cl_best[rank], 0, m);
  }
  cluster_sync();  // every slice maximum is in CTA 0's shared memory
  if (rank == 0 && threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int r = 0; r < AM_CL; ++r) m = max(m, cl_best[r]);
    tokens[b] = m ? (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull)) : -1;
  }
}

int launch_argmax_rows(const float* logits, int B, int V, int32_t* tokens, __half* logits16, cudaStream_t s,
                       int tag) {
  cudaError_t e = launch_pdl(w4pg_argmax_rows, dim3(AM_CL, B), dim3(256), 0, s, logits, V, tokens, logits16, tag);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "argmax launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}
}  // namespace w4

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
using namespace w4;

extern "C" unsigned long long w4a16_debug_set_wait_limit_ns(unsigned long long ns) {
  return g_wait_limit_ns.exchange(ns);
}

extern "C" size_t w4a16_gemm_workspace_size(int M, int K, int N, int silu) {
  if (K < 128 || N < 1 || M < 1) return 0;
  const int nc = tc_cols(M, true, silu != 0);
  int ks = 1, ps = 0;
  tc_plan(N, K, true, silu != 0, true, &ks, &ps, nc);
  return tc_workspace_bytes(N, ks, silu != 0, nc);
}

static int tc_common_checks(const uint16_t* x, int M, int K, int N, const uint16_t* y, const void* ws, size_t wsb,
                            int N_silu, int* ksplit, int* per_split) {
  W4_CHECK_ARG(x && y, "w4a16_gemm: null x or y");
  W4_CHECK_ARG(M >= 1 && K >= 1 && N >= 1, "w4a16_gemm: sizes must be positive");
  const int maxm = tc_max_rows(true, N_silu != 0);
  W4_CHECK_SHAPE(M <= maxm, "w4a16_gemm: M=%d > %d", M, maxm);
  W4_CHECK_SHAPE(K % 128 == 0, "w4a16_gemm: K=%d must be a multiple of 128", K);
  W4_CHECK_ALIGN(x, 128, "x");
  W4_CHECK_ALIGN(y, 128, "y");
  W4_CHECK_ALIGN(ws, 128, "workspace");
  const int nc = tc_cols(M, true, N_silu != 0);
  tc_plan(N, K, true, N_silu != 0, ws != nullptr, ksplit, per_split, nc);
  if (*ksplit > 1 && wsb < tc_workspace_bytes(N, *ksplit, N_silu != 0, nc))
    tc_plan(N, K, true, N_silu != 0, false, ksplit, per_split, nc);
  return W4A16_OK;
}

static void tc_ws(TcArgs& a, void* ws) {
  if (a.ksplit > 1) tc_workspace_layout(a, ws);
}

extern "C" int w4a16_gemm(const uint16_t* x, int M, int K, const uint32_t* qweight, const uint16_t* scales, int N,
                          const uint16_t* bias, const uint16_t* residual, uint16_t* y, void* workspace,
                          size_t workspace_bytes, w4a16_stream_t stream) {
  int ks = 1, ps = 0;
  int rc = tc_common_checks(x, M, K, N, y, workspace, workspace_bytes, 0, &ks, &ps);
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
  a.per_split = ps;
  tc_ws(a, workspace);
  return launch_gemm_tc(a, true, false, (cudaStream_t)stream);
}

extern "C" int w4a16_gemm_silu_mul(const uint16_t* x, int M, int K, const uint32_t* qweight_gate,
                                   const uint16_t* scales_gate, const uint32_t* qweight_up, const uint16_t* scales_up,
                                   int N, uint16_t* y, void* workspace, size_t workspace_bytes,
                                   w4a16_stream_t stream) {
  int ks = 1, ps = 0;
  int rc = tc_common_checks(x, M, K, N, y, workspace, workspace_bytes, 1, &ks, &ps);
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
  a.per_split = ps;
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
  W4_CHECK_SHAPE(B <= 65535, "argmax_rows: B=%d > 65535", B);
  return launch_argmax_rows(logits, B, vocab, tokens_out, reinterpret_cast<__half*>(logits16), (cudaStream_t)stream,
                            0);
}
