// persistent.h -- internal interface of the persistent decode kernel (not
// part of the public ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4 {

// One decoder layer's device pointers, as the persistent kernel reads them
// (a device array of these lives in the model's arena).
struct PkLayer {
  const uint32_t *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const __half *sq, *sk, *sv, *so, *sg, *su, *sd;
  const __half *bq, *bk, *bv, *ln1, *ln2;
  __half *k_pool, *v_pool;
};

// Control words of the persistent kernel (a small zeroed block of the arena).
enum { PK_CTL_BAR = 0, PK_CTL_STEP = 1, PK_CTL_ABORT = 2, PK_CTL_LM_TICKET = 3, PK_CTL_WORDS = 64 };

struct PkArgs {
  const PkLayer* layers;  // device array [n_layers]
  int n_layers;
  const __half* embed;
  const __half* final_norm;
  const __half* lm_head;
  const int32_t* tokens_in;
  int32_t* tokens_out;
  const int32_t* block_table;  // [1][max_blocks]
  int max_blocks;
  int32_t* context_lens;       // [1]
  __half* logits;              // [vocab] or null
  __half *x, *qkv, *att, *h, *mlp;  // activations (arena)
  float* att_part;             // [Hkv][P][G][128 + 2] partial attention states
  unsigned* att_tickets;       // [Hkv], zero between uses
  unsigned long long* lm_keys; // [grid] per-CTA argmax keys
  unsigned* ctl;               // PK_CTL_* words
  int32_t* err_flag;
  int H, Hq, Hkv, I, vocab, num_pages, max_context, P;
  float eps, scale_log2;
  unsigned long long wait_limit_ns;
  float inv_freq[64];
};

// Tokens per attention partition of the persistent kernel (4 pages).
constexpr int PK_PARTITION_TOKENS = 64;
// Largest context the persistent path takes (its attention merges up to 64
// partitions per kv head).
constexpr int PK_MAX_CONTEXT = 64 * PK_PARTITION_TOKENS;

// Shapes the persistent kernel is built for: one sequence, head_dim 128,
// 7 query heads per kv head, hidden, inter and every projection width a
// multiple of 128 (inter <= 18944), Hq/Hkv == 7.
bool persistent_supported(int hidden, int n_q_heads, int n_kv_heads, int head_dim, int inter, int n_layers,
                          int max_context);
// Bytes of arena the persistent path needs beyond the kernel path's buffers.
size_t persistent_workspace_bytes(int n_kv_heads, int max_context, int n_layers);
int launch_persistent(const PkArgs& a, cudaStream_t s);

}  // namespace w4
