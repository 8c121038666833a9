// kernels.h -- internal launch interfaces shared by the C-ABI files and the
// model runtime (not part of the public ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's driver entry point)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4 {

// One weight matrix (or a row range of the logical output) of a GEMV.
struct GemvSeg {
  const uint32_t* qw;   // packed int4 [rows][K/8]
  const __half* s;      // scales [rows][K/128]
  const __half* bias;   // [rows] or null
  int rows;
};

struct GemvArgs {
  const __half* x;         // [M][K]
  const __half* gamma;     // optional fused RMSNorm weight [K]
  const __half* residual;  // optional [M][N]
  __half* y;               // [M][N]
  GemvSeg seg[3];          // rows of seg 0, then seg 1, ... (SiLU mode: gate, up)
  int nseg;
  int M, K, N;
  float eps;
  int tag;                 // launch index (kernel timeline builds only)
};

int launch_gemv(const GemvArgs& a, bool silu, cudaStream_t s);
int gemv_cuda_core_supported(int M, int K);

// Tensor-core (tcgen05) GEMM: decode batches of up to 32 sequences, and the
// wider row blocks of a prompt (up to tc_max_rows rows per call).
struct TcArgs {
  const __half* x;         // [M][K] activations
  const __half* residual;  // [M][ldy] or null
  __half* y;               // [M][ldy] fp16 output (unless y32)
  float* y32;              // [M][ldy] fp32 output or null (dense lm_head logits)
  GemvSeg seg[3];          // int4 weights (SiLU: gate, up)
  int nseg;
  const __half* w16;       // dense fp16 weights [N][K] (lm_head)
  float* ws;               // split-K partial tiles
  unsigned int* counters;  // split-K tickets, one per 128-row tile (zero before first use)
  int32_t* err_flag;
  int M, K, N, ldy, ksplit, tag;
  int per_split;           // stages (128 k, one scale group) per split; 0: ceil(stages / ksplit)
  unsigned long long wait_limit_ns;  // bound of every mbarrier wait (set by the launcher)
  // Bulk-tensor (TMA) copies, set by the launcher: tm_w[i] the weights of
  // segment i (int4: u32 [rows][K/8], 16 x 128 boxes; dense fp16: [N][K],
  // 64 x 128 boxes, 128-byte swizzle), tm_x the activations [M][K] (64 x NC
  // boxes, 128-byte swizzle).
  CUtensorMap tm_w[3];
  CUtensorMap tm_x;
};
// Bound of the persistent decode kernel's grid-barrier waits, read at each
// launch (w4a16_debug_set_wait_limit_ns changes it; 0 = give up at the first
// barrier that is not already complete).
unsigned long long tc_wait_limit_ns();
int launch_gemm_tc(const TcArgs& a, bool int4, bool silu, cudaStream_t s);

// Split-K workspaces (tensor-core GEMM and attention) start with a fixed
// block of tickets, zero between calls, followed by the partial results.
// The tickets' place does not depend on the call's shape, so one zeroed
// workspace can serve calls of different shapes in turn.
constexpr size_t TC_TICKET_BYTES = 8192;    // one ticket per 128-row tile: up to 2048 tiles
constexpr size_t ATT_TICKET_BYTES = 16384;  // one ticket per (sequence, kv head): up to 4096
// batch columns per tile for M rows (32, or 64 / 128 for wider int4 blocks)
int tc_cols(int M, bool int4, bool silu);
int tc_max_rows(bool int4, bool silu);  // 128 int4, 64 int4 gate|up, 32 dense
size_t tc_workspace_bytes(int N, int ksplit, bool silu, int nc = 32);
// split of K (ksplit splits of per_split stages) that fills whole waves of CTAs
void tc_plan(int N, int K, bool int4, bool silu, bool allow_split, int* ksplit, int* per_split, int nc = 32);
void tc_workspace_layout(TcArgs& a, void* ws);  // sets a.counters / a.ws (a.ksplit > 1)
int launch_argmax_rows(const float* logits, int B, int V, int32_t* tokens, __half* logits16, cudaStream_t s,
                       int tag);

// Paged attention (+ fused split-K combine, optionally fused RoPE + append).
struct AttnArgs {
  const __half* q;          // [B][Hq][D] with row pitch q_stride (fused: q | k_new | v_new rows)
  __half* k_pool;           // [pages][Hkv][16][D] (written only by the fused variant)
  __half* v_pool;
  const int32_t* block_table;
  const int32_t* context_lens;
  __half* out;              // [B][Hq][D]
  float* ws_o;              // [B][Hq][P][D]
  float* ws_ml;             // [B][Hq][P][2]
  unsigned int* counters;   // [B][Hkv]
  int32_t* err_flag;
  int q_stride, num_pages, max_blocks, B, Hq, Hkv, P, part_tokens;
  float scale_log2;         // sm_scale * log2(e)
  int fuse_rope_append;     // 1: rotate q and k_new at len-1, append k_new/v_new, then attend
  int use_cluster;          // set by the launcher: partitions merged in a thread-block cluster
  float inv_freq[64];       // RoPE inverse frequencies (fused variant)
  int tag;                  // launch index (kernel timeline builds only)
  // FP8 (E4M3) pages instead of k_pool / v_pool: codes [pages][Hkv][16][D]
  // and fp32 row scales [pages][Hkv][16] (value = code * scale)
  int kv8;
  uint8_t* k8;
  uint8_t* v8;
  float* ks;
  float* vs;
};
int launch_paged_attention(const AttnArgs& a, cudaStream_t s);
// Causal prompt attention: rows 0..B-1 of q are tokens of one sequence at
// positions context_lens[i] - 1, its pages in row 0 of block_table; out [B][Hq][D].
int launch_prefill_attention(const AttnArgs& a, cudaStream_t s);
constexpr int ATT_MAX_PARTITIONS = 1024;
size_t attention_workspace_bytes(int B, int Hq, int Hkv, int P);
void attention_workspace_layout(AttnArgs& a, void* ws, int B, int Hq, int P);  // sets ws_o, ws_ml, counters

// RoPE + KV append.
struct RopeArgs {
  __half* q;                // [B][Hq][D] pitch stride
  __half* k;                // [B][Hkv][D] pitch stride (rotated in place too)
  const __half* v;
  __half* k_pool;
  __half* v_pool;
  const int32_t* block_table;
  const int32_t* context_lens;
  int32_t* err_flag;
  int stride_q, stride_kv, num_pages, max_blocks, B, Hq, Hkv;
  float inv_freq[64];       // fp32 inverse frequencies, D = 128
  // FP8 pools (non-null k8 selects them): codes and fp32 row scales
  uint8_t* k8;
  uint8_t* v8;
  float* ks;
  float* vs;
};
int launch_rope_append(const RopeArgs& a, cudaStream_t s);
void rope_inv_freq_table(float theta, int D, float* out);

int launch_rmsnorm(const __half* x, const __half* gamma, __half* y, int M, int H, float eps, cudaStream_t s,
                   int tag = 0);
// lens_to_advance (nullable): context_lens[b] += 1; a length above max_len sets bit 0 of err_flag
int launch_embedding(const __half* embed, int vocab, int H, const int32_t* tokens, int B, __half* x,
                     int32_t* err_flag, int32_t* lens_to_advance, int max_len, cudaStream_t s, int tag = 0);

int launch_prefill_rows(const int32_t* bt_row, int max_blocks, const int32_t* len0, int T, int32_t* bt_rep,
                        int32_t* lens, cudaStream_t s);
int launch_advance_len(int32_t* len, int T, int max_len, int32_t* err_flag, cudaStream_t s);

struct LmHeadArgs {
  const __half* x;      // [B][H]
  const __half* w;      // [vocab][H]
  __half* logits;       // [B][vocab] or null
  int32_t* tokens_out;  // [B]
  unsigned long long* partial;  // [B][blocks] packed (key, index)
  unsigned int* counters;       // [B]
  int B, H, vocab;
  const __half* gamma;  // optional fused final RMSNorm
  float eps;
  int tag;              // launch index (kernel timeline builds only)
};
int launch_lm_head_argmax(const LmHeadArgs& a, cudaStream_t s);
size_t lm_head_workspace_bytes(int B, int vocab);

}  // namespace w4
