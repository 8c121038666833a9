/*
 * w4a16.h -- C ABI of the sm_103a W4A16 + paged-GQA single-token decode library.
 *
 * The operations follow the "annotated-llm-runtime" decode path as described on
 *   [RU] aikraft.ru, "How to build your own LLM runtime from scratch",
 *        section "Архитектурные решения и оптимизации" (28 layers, hidden 3584,
 *        28 heads with 7:1 GQA, symmetric group-wise INT4 weights with group 128,
 *        RMSNorm and lm_head in FP16, 16-token KV pages whose per-head slice is
 *        4 KiB), and
 *   [EN] explore.n1n.ai, "Building a Custom LLM Inference Runtime on H100",
 *        sections "2. The KV Cache and PagedAttention", "3. CUDA Graph Capture",
 *        "Bug 1: The KV Cache Indexing 'Off-By-One'", "Bug 2: Tensor Core
 *        Alignment", "Bug 3: CUDA Graph Stream Synchronization" and
 *        "Implementation Guide: Step-by-Step" (static pre-allocation).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - fp16 tensors are passed as `uint16_t*` holding IEEE binary16 bit patterns.
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, and must be
 *    128-byte aligned ([EN] "Bug 2": the runtime enforces 128-byte alignment);
 *    a misaligned pointer returns W4A16_ERR_ALIGNMENT.  Row pitches of the
 *    packed tensors follow from the shapes (no padding).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work: none allocates, synchronises or copies through the host, so
 *    all of them may be recorded into a CUDA graph ([EN] "Bug 3").
 *  - Kernels are launched with programmatic dependent launch.  A kernel of
 *    this library may start while the previous kernel of this library on the
 *    same stream is still running.  It may read its weights (packed weights,
 *    scales, biases, RMSNorm gamma, lm_head rows) before waiting for that
 *    kernel, and waits before it reads activations, KV pools, block tables or
 *    lengths.  So weights must not be produced by the call of this library
 *    immediately before on the same stream; a copy, another library's kernel
 *    or an earlier call in between orders them as usual.
 *  - Return value: W4A16_OK or an error code; w4a16_last_error() gives the
 *    message of the last failure on the calling thread.  Shape and pointer
 *    checks happen on the host before anything is enqueued.  Conditions only
 *    the device can see (a block-table entry outside the pool, a token id
 *    outside the vocabulary) are reported through an optional device
 *    `err_flag` word: the offending access is skipped, bit 0 of *err_flag is
 *    set, and nothing traps.
 *
 * Storage formats
 * ---------------
 *  - Packed INT4 weight of an [N][K] matrix: uint32 qweight[N][K/8]; element k
 *    of row n is nibble (k % 8) of word k/8, lowest nibble first, stored
 *    offset-binary u = q + 8 so q = u - 8 is in [-8, 7].  Scales: fp16
 *    scales[N][K/128], one per 128 consecutive k.  Dequantised weight =
 *    q * scale (symmetric, no zero point).  K must be a multiple of 128.
 *  - Paged KV pool (one K pool and one V pool per layer): fp16
 *    [num_pages][Hkv][16][D]; the (page, kv head) slice is 16*D*2 bytes
 *    (4 KiB at D = 128).  block_table is int32 [B][max_blocks]; token t of
 *    sequence b lives in page block_table[b][t / 16], slot t % 16.  Entries
 *    past a sequence's last page are never read.
 *  - context_lens (int32 [B], device) counts tokens AFTER the current token is
 *    appended: the new token sits at position context_lens[b] - 1, and
 *    attention covers positions [0, context_lens[b]).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

typedef struct CUstream_st* w4a16_stream_t; /* same type as cudaStream_t */

enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad flag */
  W4A16_ERR_ALIGNMENT = 2,   /* a pointer is not 128-byte aligned */
  W4A16_ERR_SHAPE = 3,       /* K % 128 != 0, D != 128, Hq % Hkv != 0, ... */
  W4A16_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  W4A16_ERR_CAPTURE = 5,     /* call not allowed while the stream is capturing */
  W4A16_ERR_DEVICE_BOUNDS = 6, /* device reported an out-of-range index */
  W4A16_ERR_TIMEOUT = 7,     /* a bounded device wait gave up */
  W4A16_ERR_NO_PAGES = 8     /* the page allocator has fewer free pages than asked for */
};

/* Message of the last failed call on this thread ("" if none). */
W4A16_API const char* w4a16_last_error(void);

/* Library ABI version (major * 100 + minor). */
W4A16_API int w4a16_version(void);

/* ------------------------------------------------------------------------
 * w4a16_gemv -- y = x . dequant(W)^T (+ bias) (+ residual), fp32 accumulate.
 * [RU] "Архитектурные решения и оптимизации": q/k/v/o and gate/up/down are
 * symmetric group-wise INT4 (group 128) with FP16 activations.
 *   x        fp16 [M][K]              input activations
 *   qweight  uint32 [N][K/8]          packed INT4 weight (format above)
 *   scales   fp16 [N][K/128]          group scales
 *   bias     fp16 [N] or NULL
 *   residual fp16 [M][N] or NULL      added before the single fp16 rounding
 *   y        fp16 [M][N]              output (must not alias x)
 * Shapes: 1 <= M <= 32, K % 128 == 0, N >= 1.  M <= 4 runs on the CUDA
 * cores (rows whose activations exceed 49152 elements together go in
 * launches of floor(49152 / K) rows, each streaming the weights); larger M
 * on the tensor cores (see w4a16_gemm).
 * ------------------------------------------------------------------------ */
W4A16_API int w4a16_gemv(const uint16_t* x, int M, int K, const uint32_t* qweight, const uint16_t* scales,
               int N, const uint16_t* bias, const uint16_t* residual, uint16_t* y,
               w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * w4a16_gemm -- the same product for a batch of rows on the tensor cores
 * (tcgen05 MMAs, fp32 accumulation in tensor memory): a decode batch
 * (1 <= M <= 32), or the wider row block of a prompt (M <= 128;
 * w4a16_gemm_silu_mul M <= 64), where every 128-row weight tile is read
 * once for all M rows.  The
 * MMAs take the exact integer codes q; each 128-wide scale group is summed
 * in tensor memory and multiplied by its fp32 scale on the way out, so the
 * only roundings are fp32 accumulation and the final fp16 store.
 * Projections with few 128-row tiles split K across CTAs when a workspace of
 * w4a16_gemm_workspace_size() bytes is given (zeroed once before first use;
 * every call leaves its counters zero; the counters occupy the first 8 KiB
 * whatever the shape, so one workspace serves calls of different shapes in
 * turn); with workspace == NULL they run without the split.  Calls sharing
 * a workspace must not overlap on the GPU.
 * w4a16_gemv routes 5 <= M <= 32 here (without the split).
 * ------------------------------------------------------------------------ */
W4A16_API int w4a16_gemm(const uint16_t* x, int M, int K, const uint32_t* qweight,
                         const uint16_t* scales, int N, const uint16_t* bias,
                         const uint16_t* residual, uint16_t* y, void* workspace,
                         size_t workspace_bytes, w4a16_stream_t stream);
/* Gated MLP front half for a batch: y = silu(G . x) * (U . x), gate and up
 * rounded to fp16 before the SiLU. */
W4A16_API int w4a16_gemm_silu_mul(const uint16_t* x, int M, int K, const uint32_t* qweight_gate,
                                  const uint16_t* scales_gate, const uint32_t* qweight_up,
                                  const uint16_t* scales_up, int N, uint16_t* y, void* workspace,
                                  size_t workspace_bytes, w4a16_stream_t stream);
W4A16_API size_t w4a16_gemm_workspace_size(int M, int K, int N, int silu);

/* Test hook for the failure path of the persistent decode kernel
 * (W4A16_PATH_PERSISTENT below).  Its grid-barrier waits are bounded
 * (default 2 s of the GPU's global timer); a wait that runs out sets bit 1
 * of the model's error word and an abort flag, every CTA leaves at its next
 * barrier once its own copies have landed, and w4a16_model_check_errors
 * reports W4A16_ERR_TIMEOUT and resets the kernel's counters.  This sets the
 * bound for launches enqueued from now on (a captured graph keeps the bound
 * it was captured with) and returns the previous one; 0 makes the first
 * barrier that is not already complete give up at once, which exercises
 * that path without any stuck barrier.  The tensor-core GEMM's own mbarrier
 * waits keep their fixed 2 s bound.  Not for production use. */
W4A16_API unsigned long long w4a16_debug_set_wait_limit_ns(unsigned long long ns);

/* Batched FP16 lm_head on the tensor cores: logits fp32 [B][vocab] = x . W^T,
 * B <= 32, H % 128 == 0; and the row-wise argmax (lowest index on ties, NaN
 * skipped, -1 for a row of NaN) with an optional fp16 copy of the logits,
 * B <= 65535. */
W4A16_API int lm_head_logits_batched(const uint16_t* x, int B, int H, const uint16_t* lm_head,
                                     int vocab, float* logits, w4a16_stream_t stream);
W4A16_API int argmax_rows(const float* logits, int B, int vocab, int32_t* tokens_out,
                          uint16_t* logits16, w4a16_stream_t stream);

/* w4a16_gemv with the RMSNorm of x fused in front (the input norm of the
 * q/k/v projection): y = dequant(W) . (x / sqrt(mean(x^2) + eps) * gamma)
 * (+ bias).  The normalised x is rounded to fp16 before the product.
 *   gamma fp16 [K]. */
W4A16_API int w4a16_gemv_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                       const uint32_t* qweight, const uint16_t* scales, int N,
                       const uint16_t* bias, uint16_t* y, w4a16_stream_t stream);

/* Gated MLP front half: y = silu(G . xn) * (U . xn), xn = RMSNorm(x) if gamma
 * is non-NULL else x.  G and U are packed INT4 [N][K/8] with scales
 * [N][K/128]; y fp16 [M][N].  silu(g) = g / (1 + exp(-g)). */
W4A16_API int w4a16_gemv_silu_mul(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                        const uint32_t* qweight_gate, const uint16_t* scales_gate,
                        const uint32_t* qweight_up, const uint16_t* scales_up, int N, uint16_t* y,
                        w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * rmsnorm -- y[m] = x[m] / sqrt(mean_k x[m][k]^2 + eps) * gamma, fp32 math,
 * one fp16 rounding.  [RU]: RMSNorm kept in FP16.  x, y fp16 [M][H];
 * gamma fp16 [H].  y may alias x.
 * ------------------------------------------------------------------------ */
W4A16_API int rmsnorm(const uint16_t* x, const uint16_t* gamma, uint16_t* y, int M, int H, float eps,
            w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * kv_append_rope -- rotate q and k by RoPE at position p = context_lens[b]-1
 * and append k, v to the paged pools ([EN] "2. The KV Cache and
 * PagedAttention", "Bug 1"; RoPE itself is not on the pages: rotate-half
 * pairs (i, i + D/2), inverse frequency theta^(-2i/D) rounded to fp32,
 * angle = fp32 product p * inv_freq).
 *   q        fp16 [B][Hq][D], rotated in place
 *   k, v     fp16 [B][Hkv][D]; k is rotated on its way into the pool
 *   row_stride  elements between sequence b and b+1 in q, k and v
 *               (0 = packed, i.e. Hq*D for q and Hkv*D for k and v; a
 *               non-zero value applies to all three, e.g. the row pitch
 *               of a fused q|k|v buffer)
 *   k_pool, v_pool fp16 [num_pages][Hkv][16][D]; exactly one slot per
 *               (b, kv head) is written, nothing else changes
 *   err_flag int32 device word or NULL: bit 0 set if a block-table entry
 *            is outside [0, num_pages) (that sequence is skipped).
 * D must be 128 and Hq % Hkv == 0.
 * ------------------------------------------------------------------------ */
W4A16_API int kv_append_rope(uint16_t* q, const uint16_t* k, const uint16_t* v, int row_stride, uint16_t* k_pool,
                   uint16_t* v_pool, int num_pages, const int32_t* block_table, int max_blocks,
                   const int32_t* context_lens, int B, int Hq, int Hkv, int D, float theta,
                   int32_t* err_flag, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * paged_gqa_decode -- out[b][h] = sum_t softmax_t(q[b][h] . k_t * sm_scale) v_t
 * over t < context_lens[b], k_t/v_t gathered through the block table, query
 * head h reading kv head h / (Hq/Hkv) ([RU] 7:1 GQA; [EN] "2. The KV Cache
 * and PagedAttention").  Tokens are split into partitions of
 * partition_tokens (a multiple of 16); each partition's (max, sum, weighted
 * V) partials go to `workspace` and are merged with the online-softmax
 * combine by the last partition to finish (no extra launch).
 *   q   fp16 [B][Hq][D] with row pitch q_stride elements (0 = Hq*D)
 *   out fp16 [B][Hq][D] (packed)
 *   max_context   upper bound on every context_lens[b] (sizes the grid); a
 *                 longer context sets bit 0 of err_flag (its tokens past the
 *                 grid's partitions are not attended to)
 *   workspace     device scratch of paged_gqa_decode_workspace_size() bytes;
 *                 its counter words must be zero before the first use and
 *                 every call leaves them zero again (w4a16_workspace_clear
 *                 zeroes it once).  The counters sit in the first 16 KiB
 *                 whatever the sizes, so one workspace serves calls of
 *                 different shapes in turn (B*Hkv <= 4096 when split);
 *                 calls that run concurrently on the GPU need separate
 *                 workspaces.
 *   err_flag      as for kv_append_rope (bad pages are skipped).
 * D must be 128, Hq % Hkv == 0, Hq/Hkv <= 8.  context_lens[b] == 0 yields
 * zeros.
 * ------------------------------------------------------------------------ */
W4A16_API int paged_gqa_decode(const uint16_t* q, int q_stride, const uint16_t* k_pool,
                     const uint16_t* v_pool, int num_pages, const int32_t* block_table,
                     int max_blocks, const int32_t* context_lens, int max_context, int B, int Hq,
                     int Hkv, int D, float sm_scale, int partition_tokens, void* workspace,
                     size_t workspace_bytes, uint16_t* out, int32_t* err_flag,
                     w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * paged_gqa_decode_rope_append -- kv_append_rope followed by
 * paged_gqa_decode, as one kernel (the form the decode step runs).
 *   qkv  fp16 rows of pitch qkv_stride: q [Hq][D] | k_new [Hkv][D] |
 *        v_new [Hkv][D] per sequence (the q|k|v GEMV output); read only --
 *        the rotated q is used in place, not written back.
 *   theta  RoPE base; the new token's position is context_lens[b] - 1.
 * k_new (rotated) and v_new are written to their slot in the pools, as
 * kv_append_rope does; the other arguments are as for paged_gqa_decode.
 * ------------------------------------------------------------------------ */
W4A16_API int paged_gqa_decode_rope_append(const uint16_t* qkv, int qkv_stride, uint16_t* k_pool,
                                           uint16_t* v_pool, int num_pages,
                                           const int32_t* block_table, int max_blocks,
                                           const int32_t* context_lens, int max_context, int B,
                                           int Hq, int Hkv, int D, float theta, float sm_scale,
                                           int partition_tokens, void* workspace,
                                           size_t workspace_bytes, uint16_t* out, int32_t* err_flag,
                                           w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) KV pages ([EN] "1. Weight Packing and FP8 Utilization": FP8
 * halves the bytes of fp16 and needs scaling factors; E4M3 is the format it
 * names).  A pool holds codes uint8 [num_pages][Hkv][16][D] (E4M3: sign, 4
 * exponent bits with bias 7, 3 fraction bits, no infinities, largest 448)
 * beside fp32 row scales [num_pages][Hkv][16]: value = code * scale.  A row
 * is quantised when appended: amax = largest magnitude of its fp16 values
 * (k after RoPE), inv = 448 / amax and scale = amax / 448 in fp32, code =
 * E4M3(x * inv) with the product in fp32, round to nearest even (an all-zero
 * row: scale 0, codes 0).  Per page and kv head: 2 x 2 KiB of codes and
 * 2 x 64 B of scales instead of 2 x 4 KiB.
 *   kv_append_rope_fp8     kv_append_rope into FP8 pools.
 *   paged_gqa_decode_fp8   paged_gqa_decode over FP8 pools (q fp16; scores
 *                          and P V in fp32 on the dequantised values).
 *   paged_gqa_decode_rope_append_fp8  the fused form (qkv rows as for
 *                          paged_gqa_decode_rope_append).
 * Pools and scales must be 128-byte aligned; the other arguments, the
 * workspace and the error flag are as for the fp16 calls.
 * ------------------------------------------------------------------------ */
W4A16_API int kv_append_rope_fp8(uint16_t* q, const uint16_t* k, const uint16_t* v, int row_stride,
                                 uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
                                 int num_pages, const int32_t* block_table, int max_blocks,
                                 const int32_t* context_lens, int B, int Hq, int Hkv, int D, float theta,
                                 int32_t* err_flag, w4a16_stream_t stream);
W4A16_API int paged_gqa_decode_fp8(const uint16_t* q, int q_stride, const uint8_t* k_pool,
                                   const uint8_t* v_pool, const float* k_scale, const float* v_scale,
                                   int num_pages, const int32_t* block_table, int max_blocks,
                                   const int32_t* context_lens, int max_context, int B, int Hq, int Hkv,
                                   int D, float sm_scale, int partition_tokens, void* workspace,
                                   size_t workspace_bytes, uint16_t* out, int32_t* err_flag,
                                   w4a16_stream_t stream);
W4A16_API int paged_gqa_decode_rope_append_fp8(const uint16_t* qkv, int qkv_stride, uint8_t* k_pool,
                                               uint8_t* v_pool, float* k_scale, float* v_scale,
                                               int num_pages, const int32_t* block_table, int max_blocks,
                                               const int32_t* context_lens, int max_context, int B,
                                               int Hq, int Hkv, int D, float theta, float sm_scale,
                                               int partition_tokens, void* workspace,
                                               size_t workspace_bytes, uint16_t* out, int32_t* err_flag,
                                               w4a16_stream_t stream);

/* Bytes of workspace paged_gqa_decode needs for these sizes. */
W4A16_API size_t paged_gqa_decode_workspace_size(int B, int Hq, int Hkv, int max_context,
                                       int partition_tokens, int D);

/* Partition size the library picks when partition_tokens == 0 is passed to
 * paged_gqa_decode (a multiple of 16): 128 up to 1024 tokens of context,
 * else 256 when B * Hkv >= 64, else 512. */
W4A16_API int paged_gqa_decode_default_partition(int B, int Hkv, int max_context);

/* ------------------------------------------------------------------------
 * paged_gqa_decode_noalloc -- the same attention as paged_gqa_decode, for
 * callers that cannot allocate device memory: a plugin handed only input
 * and output pointers by a host framework that owns the device's memory
 * pool, or code running while allocation is forbidden (inside a global-mode
 * stream capture, where cudaMalloc is illegal).  Nothing is allocated: the
 * split-K partials and ticket counters live in one static device array of
 * W4A16_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds
 * until the process exits.  The pages describe no such call; it has no
 * counterpart there.
 *   Arguments as for paged_gqa_decode, minus the workspace.
 *   Sizes whose partials need more than W4A16_NOALLOC_SCRATCH_BYTES return
 *   W4A16_ERR_SHAPE (need = paged_gqa_decode_workspace_size()).
 *   The first call on each device looks the array's device address up (with
 *   that device current); make that first call before any stream capture.
 *   Every call zeroes the counters it uses on `stream` before launching.
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other threads) race and must be serialised by the caller.
 * ------------------------------------------------------------------------ */
#define W4A16_NOALLOC_SCRATCH_BYTES (4u << 20)
W4A16_API int paged_gqa_decode_noalloc(const uint16_t* q, int q_stride, const uint16_t* k_pool,
                                       const uint16_t* v_pool, int num_pages,
                                       const int32_t* block_table, int max_blocks,
                                       const int32_t* context_lens, int max_context, int B, int Hq,
                                       int Hkv, int D, float sm_scale, int partition_tokens,
                                       uint16_t* out, int32_t* err_flag, w4a16_stream_t stream);

/* Zero a workspace once before first use (enqueued on `stream`). */
W4A16_API int w4a16_workspace_clear(void* workspace, size_t bytes, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * Embedding row gather: x[b] = embed[tokens[b]], embed fp16 [vocab][H].
 * Not on the pages (plain decoder front end).  A token outside [0, vocab)
 * sets bit 0 of err_flag and yields a zero row.
 * ------------------------------------------------------------------------ */
W4A16_API int embedding_gather(const uint16_t* embed, int vocab, int H, const int32_t* tokens, int B,
                     uint16_t* x, int32_t* err_flag, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * lm_head_argmax -- logits = W . x (FP16 weight [vocab][H], fp32 accumulate)
 * and token = argmax (lowest index on ties), per sequence.  [RU]: lm_head
 * kept in FP16; the argmax is the greedy decode rule.
 *   x          fp16 [B][H]
 *   logits     fp16 [B][vocab] or NULL
 *   tokens_out int32 [B]
 *   workspace  lm_head_argmax_workspace_size() bytes; counter words zero
 *              before first use, left zero by every call.
 * ------------------------------------------------------------------------ */
W4A16_API int lm_head_argmax(const uint16_t* x, int B, int H, const uint16_t* lm_head, int vocab,
                   uint16_t* logits, int32_t* tokens_out, void* workspace, size_t workspace_bytes,
                   w4a16_stream_t stream);
W4A16_API size_t lm_head_argmax_workspace_size(int B, int vocab);

/* ------------------------------------------------------------------------
 * Whole model (Qwen2-shaped decoder).  [EN] "Implementation Guide": static
 * pre-allocation and a CUDA-graph-captured decode step; [RU] "Ключевые
 * метрики производительности": the graph-captured steady-state decode.
 * ------------------------------------------------------------------------ */
typedef struct {
  int hidden, n_q_heads, n_kv_heads, head_dim, inter, n_layers, vocab;
  float eps, theta;
  int num_pages;        /* pages in each layer's K (and V) pool */
  int partition_tokens; /* split-K partition for attention; 0 = library choice */
} w4a16_model_config;

typedef struct {
  const uint16_t *ln1, *ln2;                          /* fp16 [hidden] */
  const uint32_t *wq, *wk, *wv, *wo, *wg, *wu, *wd;   /* packed INT4 */
  const uint16_t *sq, *sk, *sv, *so, *sg, *su, *sd;   /* fp16 group scales */
  const uint16_t *bq, *bk, *bv;                       /* fp16 biases or NULL */
  uint16_t *k_pool, *v_pool;                          /* this layer's pools */
  /* FP8 (E4M3) KV pages instead of k_pool / v_pool (every layer or none;
   * k_pool / v_pool then NULL): codes uint8 [num_pages][Hkv][16][D] and fp32
   * row scales [num_pages][Hkv][16], as paged_gqa_decode_fp8 takes them.
   * The decode step and w4a16_prefill then append quantised rows and attend
   * over the codes; the persistent decode path is not built for them. */
  uint8_t *k8, *v8;
  float *k_scale, *v_scale;
} w4a16_layer_weights;

typedef struct {
  const uint16_t* embed;      /* fp16 [vocab][hidden] */
  const uint16_t* final_norm; /* fp16 [hidden] */
  const uint16_t* lm_head;    /* fp16 [vocab][hidden] */
  const w4a16_layer_weights* layers; /* HOST array [n_layers], copied */
} w4a16_model_weights;

typedef struct w4a16_model w4a16_model;

/* Builds the model handle.  The only call that allocates: one device arena
 * for activations and workspaces sized for max_batch (1..32) sequences of up
 * to max_context tokens.  Weight and pool pointers are borrowed (caller keeps
 * them alive).  A decode_step that takes a sequence past max_context tokens
 * sets bit 0 of the model's error word (W4A16_ERR_DEVICE_BOUNDS from
 * w4a16_model_check_errors). */
W4A16_API int w4a16_model_create(const w4a16_model_config* cfg, const w4a16_model_weights* w, int max_batch,
                       int max_context, w4a16_model** out);
W4A16_API void w4a16_model_destroy(w4a16_model* m);

/* Device word the model's kernels report out-of-range indices into. */
W4A16_API int32_t* w4a16_model_err_flag(w4a16_model* m);

/* Synchronise `stream`, read and clear the model's device error word:
 * returns W4A16_ERR_DEVICE_BOUNDS if a kernel skipped an out-of-range page or
 * token, W4A16_ERR_TIMEOUT if a bounded wait gave up, else W4A16_OK.  After
 * a timeout the step's outputs are not valid; the call also clears the
 * split-K tickets of the model's workspaces, so the next step runs clean.
 * This call blocks and copies to the host, so it must not be used while the
 * stream is capturing. */
W4A16_API int w4a16_model_check_errors(w4a16_model* m, w4a16_stream_t stream);

/* Copy the final hidden states (before the final RMSNorm) that the last
 * decode_step left in the model's arena into dst fp16 [B][hidden]
 * (enqueued on `stream`; capture-safe). */
W4A16_API int w4a16_model_hidden(w4a16_model* m, uint16_t* dst, int B, w4a16_stream_t stream);

/* Copy one of the activation buffers the last layer (or decode step) left
 * in the model's arena into dst fp16 [B][width] (enqueued on `stream`):
 *   W4A16_ACT_HIDDEN  the step's hidden state x            width hidden
 *   W4A16_ACT_QKV     q | k | v projections (+bias)        width (Hq+2Hkv)*D
 *   W4A16_ACT_ATTN    attention output, before o           width Hq*D
 *   W4A16_ACT_RESID   x + o projection (post-attention)    width hidden
 *   W4A16_ACT_MLP     silu(gate) * up                      width inter
 * For checking each kernel of a layer on its own inputs. */
enum {
  W4A16_ACT_HIDDEN = 0,
  W4A16_ACT_QKV = 1,
  W4A16_ACT_ATTN = 2,
  W4A16_ACT_RESID = 3,
  W4A16_ACT_MLP = 4
};
W4A16_API int w4a16_model_activation(w4a16_model* m, int which, uint16_t* dst, int B, w4a16_stream_t stream);

/* One decoder layer on hidden states x fp16 [B][hidden] (in place), with
 * context_lens already counting the appended token. */
W4A16_API int w4a16_model_layer(w4a16_model* m, int layer, uint16_t* x, const int32_t* block_table,
                      int max_blocks, const int32_t* context_lens, int B, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * decode_step -- one greedy decode step for B sequences:
 *   context_lens[b] += 1 (on the device; the new token goes to position
 *   context_lens[b] - 1), x = embed[tokens_in], n_layers decoder layers
 *   (RMSNorm -> q/k/v GEMV + bias -> RoPE + KV append -> paged GQA
 *   attention -> o GEMV + residual -> RMSNorm -> gate/up GEMV + SiLU-mul ->
 *   down GEMV + residual), final RMSNorm, lm_head, argmax -> tokens_out.
 *   B <= 4 runs the CUDA-core GEMVs with the RMSNorms fused in front and
 *   the lm_head GEMV with a fused argmax (at B = 3, 4 gate/up, and down
 *   at K = 18944, take the tensor-core GEMM, gate/up after its own
 *   RMSNorm); 4 < B <= max_batch runs each
 *   RMSNorm on its own, the projections and the lm_head as tensor-core
 *   GEMMs (fp32 logits in the model's arena) and a row-wise argmax.
 *   tokens_in, tokens_out  int32 [B] device (may be the same buffer)
 *   block_table            int32 [B][max_blocks]; pages for the new
 *                          position must already be assigned
 *   logits                 fp16 [B][vocab] or NULL
 *   use_graph              1: capture the step into a CUDA graph on first
 *                          use for this argument set and replay it after;
 *                          0: launch the kernels directly.
 * Every pointer must stay the same across replays of one graph (the graph
 * is keyed on them); the data they point to may change between calls.
 * ------------------------------------------------------------------------ */
W4A16_API int decode_step(w4a16_model* m, const int32_t* tokens_in, int32_t* tokens_out,
                const int32_t* block_table, int max_blocks, int32_t* context_lens, int B,
                uint16_t* logits, int use_graph, w4a16_stream_t stream);

/* Number of kernels one decode_step launches for B sequences (graph or not). */
W4A16_API int decode_step_kernel_count(w4a16_model* m, int B);

/* ------------------------------------------------------------------------
 * w4a16_prefill -- the prompt of one sequence in one pass ([RU] "Ключевые
 * метрики производительности": TTFT for a 512-token prompt).
 *   tokens         int32 [T] device, the prompt (T >= 1)
 *   block_table    int32 [1][max_blocks] device; pages for positions
 *                  [context_lens[0], context_lens[0] + T) already assigned
 *   context_lens   int32 [1] device: tokens cached before the prompt (0 for
 *                  a new sequence); advanced by T on the device
 *   token_out      int32 [1] device: greedy next token after the prompt
 *   logits         fp16 [vocab] or NULL: the last prompt token's logits
 *   workspace      w4a16_prefill_workspace_size(m, T, max_blocks) bytes,
 *                  256-byte aligned (activations of the T rows)
 * Per layer: RMSNorm, q|k|v (tensor-core GEMM over the T rows, bias), RoPE
 * and the append of all T positions to the pages, causal paged attention
 * (token t sees positions <= context_lens[0] + t), o + residual, RMSNorm,
 * gate|up + SiLU-mul, down + residual; then final RMSNorm, lm_head and
 * argmax for the last token.  Same arithmetic as T decode steps (fp16
 * roundings at the same points; sums in other orders).  Enqueue only.
 * ------------------------------------------------------------------------ */
W4A16_API size_t w4a16_prefill_workspace_size(w4a16_model* m, int T, int max_blocks);
W4A16_API int w4a16_prefill(w4a16_model* m, const int32_t* tokens, int T, const int32_t* block_table,
                            int max_blocks, int32_t* context_lens, int32_t* token_out, uint16_t* logits,
                            void* workspace, size_t workspace_bytes, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * How decode_step runs a step ([EN] "3. CUDA Graph Capture"; [RU]
 * "Ключевые метрики производительности": the per-token cost that is not
 * bandwidth is kernel launches).
 *   W4A16_PATH_KERNELS     one kernel per operation (5 per layer for B <= 4),
 *                          chained with programmatic dependent launch;
 *   W4A16_PATH_PERSISTENT  one cooperative kernel for the whole step: every
 *                          SM runs one CTA that walks all layers' phases with
 *                          a grid-wide barrier between them, streaming the
 *                          next phase's weights (and the attention's KV pages)
 *                          into shared memory before each barrier.  It covers
 *                          one sequence (B == 1) of a model with head_dim 128,
 *                          Hq == 7 Hkv, inter <= 18944, an even vocabulary and
 *                          max_context <= 4096; it needs all SMs (cooperative
 *                          launch), and its barrier waits are bounded (a wait
 *                          that runs out reports W4A16_ERR_TIMEOUT through
 *                          w4a16_model_check_errors, which also resets it);
 *   W4A16_PATH_AUTO        (default) the path measured faster on GB300 for
 *                          the shapes the persistent kernel covers (see
 *                          w4a16_model_decode_path); else the kernels.
 * Both paths compute the same step; sums are ordered differently, so
 * outputs agree to fp16 rounding, not bit for bit.  Graphs captured by
 * decode_step are keyed on the path.  set returns W4A16_ERR_SHAPE when the
 * persistent path is asked for a model it does not cover;
 * w4a16_model_decode_path reports the path decode_step takes for B
 * sequences (W4A16_PATH_KERNELS or W4A16_PATH_PERSISTENT).
 * ------------------------------------------------------------------------ */
enum { W4A16_PATH_AUTO = 0, W4A16_PATH_KERNELS = 1, W4A16_PATH_PERSISTENT = 2 };
W4A16_API int w4a16_model_set_decode_path(w4a16_model* m, int path);
W4A16_API int w4a16_model_decode_path(w4a16_model* m, int B);

/* ------------------------------------------------------------------------
 * Host page allocator ([EN] "2. The KV Cache and PagedAttention": the KV
 * cache managed like virtual memory, fixed-size pages handed out as
 * sequences grow).  Host-side bookkeeping only, thread-safe; it never
 * touches device memory.  Pages are the indices of a pool's first dimension.
 *   create        pages [0, num_pages) all free; handed out lowest first.
 *   alloc         n pages into pages[0..n): all or nothing (W4A16_ERR_NO_PAGES
 *                 leaves the allocator unchanged).
 *   free          returns pages; a page outside the pool, one not handed out,
 *                 or one named twice returns W4A16_ERR_INVALID_ARG and frees
 *                 nothing.
 *   free_count    pages free now (-1 for a NULL allocator).
 *   seq_reserve   makes a host block-table row cover len tokens: entries
 *                 [0, ceil(len/16)) that are -1 get pages (all or nothing);
 *                 W4A16_ERR_SHAPE if that exceeds max_blocks.
 *   seq_release   frees every entry >= 0 of the row and sets it to -1.
 * ------------------------------------------------------------------------ */
typedef struct w4a16_page_allocator w4a16_page_allocator;
W4A16_API int w4a16_page_allocator_create(int num_pages, w4a16_page_allocator** out);
W4A16_API void w4a16_page_allocator_destroy(w4a16_page_allocator* a);
W4A16_API int w4a16_page_alloc(w4a16_page_allocator* a, int n, int32_t* pages);
W4A16_API int w4a16_page_free(w4a16_page_allocator* a, const int32_t* pages, int n);
W4A16_API int w4a16_page_free_count(w4a16_page_allocator* a);
W4A16_API int w4a16_seq_reserve(w4a16_page_allocator* a, int32_t* row, int max_blocks, int len);
W4A16_API int w4a16_seq_release(w4a16_page_allocator* a, int32_t* row, int max_blocks);

/* ------------------------------------------------------------------------
 * Continuous batching over decode_step ([EN] "2. The KV Cache and
 * PagedAttention", "Why Build from Scratch?" item 3: maximise batch sizes).
 * The batcher owns a page allocator over the model's pools (num_pages must
 * not exceed the model's), the host block tables and small device buffers
 * (allocated at create; steps allocate nothing on the device).
 *   submit   queues a sequence: its prompt (host int32, >= 1 token) is fed
 *            one token per step, then up to max_new_tokens greedy tokens
 *            are generated; prompt_len + max_new_tokens - 1 <= max_context,
 *            and the sequence alone must fit the pool (else
 *            W4A16_ERR_NO_PAGES).  Returns its id.
 *   step     admits queued sequences into free slots (max_batch), gives
 *            every active sequence the page of its next position (a page per
 *            16 tokens; with the pool empty the most recently admitted
 *            sequence is preempted -- pages freed, restarted from its prompt
 *            later, same greedy result), uploads tokens, lengths and block
 *            tables, runs decode_step for the B active sequences (one
 *            captured graph per B), reads the new tokens back (synchronises
 *            `stream`), and retires finished sequences, freeing their pages.
 *            *n_active: sequences in the step (0: nothing to do).
 *   poll     a sequence's generated tokens so far (up to cap copied),
 *            their count and whether it finished.
 *   stats    steps run, preemptions, queued and active sequences, free pages.
 * ------------------------------------------------------------------------ */
typedef struct w4a16_batcher w4a16_batcher;
W4A16_API int w4a16_batcher_create(w4a16_model* model, int num_pages, int max_batch, int max_blocks,
                                   int max_context, w4a16_batcher** out);
W4A16_API void w4a16_batcher_destroy(w4a16_batcher* b);
W4A16_API int w4a16_batcher_submit(w4a16_batcher* b, const int32_t* prompt, int prompt_len, int max_new_tokens,
                                   int* seq_id);
W4A16_API int w4a16_batcher_step(w4a16_batcher* b, w4a16_stream_t stream, int* n_active);
W4A16_API int w4a16_batcher_poll(w4a16_batcher* b, int seq_id, int32_t* tokens, int cap, int* n_tokens,
                                 int* done);
W4A16_API int w4a16_batcher_stats(w4a16_batcher* b, long* steps, long* preemptions, int* waiting, int* active,
                                  int* free_pages);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
