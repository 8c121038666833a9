// common.cuh -- shared device/host helpers for the sm_103a decode kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "w4a16.h"

namespace w4 {

// ---------------------------------------------------------------------------
// Host-side status plumbing.  Every entry point returns a status code and
// leaves a thread-local message for w4a16_last_error().
// ---------------------------------------------------------------------------
int set_error(int code, const char* fmt, ...);
int check_launch(const char* what);
bool aligned(const void* p, size_t a);
int num_sms();
int device_index();

// One-time set-up per device (kernel attributes such as the dynamic shared
// memory limit are per device): f() runs once for each device ordinal that
// reaches it, under a lock, before any caller on that device proceeds.
struct PerDeviceOnce {
  std::mutex mu;
  unsigned long long done = 0;  // bit d: device d is set up (ordinals < 64)
};
template <class F>
inline void once_per_device(PerDeviceOnce& o, F f) {
  const unsigned long long bit = 1ull << (device_index() & 63);
  std::lock_guard<std::mutex> lk(o.mu);
  if (!(o.done & bit)) {
    f();
    o.done |= bit;
  }
}

#define W4_CHECK_ARG(cond, ...)                                   \
  do {                                                            \
    if (!(cond)) return ::w4::set_error(W4A16_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define W4_CHECK_SHAPE(cond, ...)                                 \
  do {                                                            \
    if (!(cond)) return ::w4::set_error(W4A16_ERR_SHAPE, __VA_ARGS__); \
  } while (0)
#define W4_CHECK_ALIGN(p, a, name)                                \
  do {                                                            \
    if ((p) != nullptr && !::w4::aligned((p), (a)))               \
      return ::w4::set_error(W4A16_ERR_ALIGNMENT, "%s must be %d-byte aligned", name, (int)(a)); \
  } while (0)

// Launch with programmatic dependent launch (PDL) enabled, so the next
// kernel in the stream may start its prologue while this one drains.
template <typename Kern, typename... Args>
inline cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// Device helpers (inline PTX for sm_100+ features).
// ---------------------------------------------------------------------------

// PDL: let dependents launch / wait for the grids this one depends on.
//
// Ordering rule kept by every kernel in this library: a kernel triggers its
// dependents (launch_dependents) only after its own griddepcontrol.wait has
// returned.  So when a kernel starts, its predecessor has passed its wait,
// which means every grid before the predecessor has completed.  Before its
// own wait a kernel may therefore read (through L2) anything written only by
// grids older than its predecessor -- weights, the block table, the context
// lengths written at the start of the step, KV pages of earlier positions --
// but nothing its predecessor writes, and it writes nothing.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_then_trigger() {
  pdl_wait();
  pdl_launch_dependents();
}

// 128-bit streaming load that bypasses L1 (weights are read exactly once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Packed fp16 subtraction a - b (exact for the small integers used here).
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per-thread async copy of 16 bytes global -> shared (bypasses L1).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
// 16-byte cp.async that writes zeros when `valid` is false (src not read).
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
// 4-byte cp.async (through L1) that writes zeros when `valid` is false.
__device__ __forceinline__ void cp_async4_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// acc += lo(a)*lo(b) + hi(a)*hi(b) with fp16 operands and fp32 accumulation
// (mixed-precision FMA, exact products).  Two chained FMAs into one sum.
__device__ __forceinline__ void fma2_f16_f32(float& acc, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\t"
      "mov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
}

// Two independent accumulators: acc0 += lo*lo, acc1 += hi*hi.
__device__ __forceinline__ void fma2_f16_f32_split(float& acc0, float& acc1, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\t"
      "mov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(a), "r"(b));
}

// Packed fp32 FMA (two lanes per instruction): d = a*b + c elementwise.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier helpers.  All waits are bounded: a wait
// that runs out sets *timed_out and returns false instead of spinning.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~max_iters polls (each try_wait itself
// suspends for a hardware-defined interval).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t max_iters) {
  for (uint32_t i = 0; i < max_iters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// Thread-block cluster helpers (distributed shared memory).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ unsigned int cluster_ctarank() {
  unsigned int r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Store four floats at the same shared-memory offset in CTA `rank` of the
// cluster (ordered before a later barrier.cluster.arrive.release).
__device__ __forceinline__ void st_dsmem4(float* p, int rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_dsmem2(float* p, int rank, float2 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(v.x), "f"(v.y) : "memory");
}
// Load a float from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_dsmem(const float* p, int rank) {
  // Not volatile: the loads are ordered after the cluster barrier (which is
  // volatile with a memory clobber) and may overlap one another.
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

// ---------------------------------------------------------------------------
// Optional kernel timeline (builds with -DW4A16_TRACE only).  Thread 0 of
// every CTA records the global timer at entry, when griddepcontrol.wait
// returns, and at exit, with the launch's tag (its index in the step).
// ---------------------------------------------------------------------------
struct TraceRec {
  unsigned long long t_entry, t_wait, t_exit, mark[3];
  unsigned int tag, cta, smid, pad;
};
static_assert(sizeof(TraceRec) == 64, "trace record layout is part of the trace API");
#ifdef W4A16_TRACE
extern __device__ TraceRec* g_trace_buf;
extern __device__ unsigned int g_trace_cap;
extern __device__ unsigned int g_trace_n;
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
struct TraceScope {
  unsigned long long t0, tw, m[3];
  unsigned int tag;
  __device__ TraceScope(unsigned int tg) : t0(trace_now()), tw(0), m{0, 0, 0}, tag(tg) {}
  __device__ void waited() { tw = trace_now(); }
  __device__ void mark(int k) { m[k] = trace_now(); }
  __device__ void set_mark(int k, unsigned long long v) { m[k] = v; }
  __device__ ~TraceScope() {
    if (threadIdx.x == 0 && g_trace_buf != nullptr) {
      const unsigned int i = atomicAdd(&g_trace_n, 1u);
      if (i < g_trace_cap) {
        unsigned int sm;
        asm volatile("mov.u32 %0, %smid;" : "=r"(sm));
        g_trace_buf[i] = TraceRec{t0, tw, trace_now(), {m[0], m[1], m[2]}, tag, (unsigned int)blockIdx.x, sm, 0u};
      }
    }
  }
};
#define W4_TRACE_SCOPE(tag) ::w4::TraceScope w4_trace_scope_(tag)
#define W4_TRACE_WAITED() w4_trace_scope_.waited()
#define W4_TRACE_MARK(k) w4_trace_scope_.mark(k)
#define W4_TRACE_SET_MARK(k, v) w4_trace_scope_.set_mark(k, v)
#else
#define W4_TRACE_SCOPE(tag) \
  do {                     \
  } while (0)
#define W4_TRACE_WAITED() \
  do {                    \
  } while (0)
#define W4_TRACE_MARK(k) \
  do {                   \
  } while (0)
#define W4_TRACE_SET_MARK(k, v) \
  do {                          \
  } while (0)
#endif

}  // namespace w4
