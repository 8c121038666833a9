// runtime.cu -- the whole-model decode step: static arena, layer sequence,
// CUDA-graph capture and replay.
//
// "Building a Custom LLM Inference Runtime on H100" (explore.n1n.ai) names
// the pieces: pre-allocate the KV cache and activation buffers so nothing
// calls cudaMalloc while decoding ("Implementation Guide", step 2), capture
// the kernel sequence into a CUDA graph to remove per-launch CPU overhead
// ("3. CUDA Graph Capture"), and keep every asynchronous operation ordered
// inside the capture ("Bug 3").  The aikraft.ru article ("Ключевые метрики
// производительности") reports the graph-captured decode as the steady state.
//
// One decode step = embedding (+ device-side context_lens advance), then per
// layer: [RMSNorm + q|k|v GEMV + bias] -> [RoPE + KV append + paged GQA
// attention + split-K combine] -> [o GEMV + residual] -> [RMSNorm + gate|up
// GEMV + SiLU-mul] -> [down GEMV + residual], then [final RMSNorm + lm_head +
// argmax].  Every kernel is launched with programmatic dependent launch, so
// a GEMV streams its first weights, and the attention its KV pages, while
// the predecessor finishes.
//
// A decode batch of more than 4 sequences is a dense contraction: each
// projection becomes [RMSNorm] + a tensor-core GEMM (exact int4 codes into
// tcgen05 MMAs, K split across CTAs), and the lm_head a tensor-core GEMM to
// fp32 logits followed by a row-wise argmax.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "persistent.h"

namespace w4 {
int default_partition(int B, int Hkv, int max_context);
}

using namespace w4;

struct GraphKey {
  int B, max_blocks, persistent;
  const void *tin, *tout, *bt, *lens, *logits;
  bool operator<(const GraphKey& o) const {
    return std::tie(B, max_blocks, persistent, tin, tout, bt, lens, logits) <
           std::tie(o.B, o.max_blocks, o.persistent, o.tin, o.tout, o.bt, o.lens, o.logits);
  }
};

struct w4a16_model {
  w4a16_model_config cfg;
  std::vector<w4a16_layer_weights> layers;
  const __half *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
  int max_batch = 0, max_context = 0, part_tokens = 0, P = 0;
  bool kv8 = false;  // the layers' KV pools are FP8 (E4M3) codes + row scales
  char* arena = nullptr;
  size_t arena_bytes = 0;
  __half *x = nullptr, *qkv = nullptr, *att = nullptr, *h = nullptr, *mlp = nullptr;
  void* attn_ws = nullptr;
  size_t attn_ws_bytes = 0;
  void* lm_ws = nullptr;
  size_t lm_ws_bytes = 0;
  __half* xn = nullptr;      // normalised activations of the batched path [max_batch][max K]
  float* logits32 = nullptr; // batched lm_head logits [max_batch][vocab] (max_batch > 4)
  void* tc_ws = nullptr;     // split-K partial tiles + tickets of the tensor-core GEMMs
  size_t tc_ws_bytes = 0;
  int32_t* err_flag = nullptr;
  float inv_freq[64];
  // persistent decode kernel (one sequence): layer table, attention partials
  // and tickets, per-CTA argmax keys, control words (barrier counter, step
  // counter, abort flag, lm_head ticket)
  bool pk_ok = false;
  int decode_path = W4A16_PATH_AUTO;
  int pk_P = 0;
  PkLayer* pk_layers = nullptr;
  float* pk_att_part = nullptr;
  unsigned* pk_att_tickets = nullptr;
  unsigned long long* pk_lm_keys = nullptr;
  unsigned* pk_ctl = nullptr;
  size_t pk_att_tickets_bytes = 0;
  cudaStream_t cap_stream = nullptr;
  std::mutex mu;
  std::map<GraphKey, cudaGraphExec_t> graphs;
};

static size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Largest batch whose projections all take the CUDA-core GEMV with the
// RMSNorm fused in front, and whose lm_head takes the fused GEMV + argmax.
static constexpr int GEMV_MAX_BATCH = 4;
static bool batched_path(const w4a16_model* m, int B) {
  return B > GEMV_MAX_BATCH || !gemv_cuda_core_supported(B, m->cfg.hidden);
}
// From 3 rows on, gate|up (the largest projection) takes the tensor-core GEMM
// after an RMSNorm of its own: at M = 3 / 4 the CUDA-core GEMV does 3-4 FMAs
// per weight (39.7 / 45.9 us for 2 x 18944 rows at K = 3584, against 26.7 us
// for the GEMM).  q|k|v and o stay on the GEMV (13 us against 14).
static constexpr int SILU_TC_MIN_ROWS = 3;

extern "C" int w4a16_model_create(const w4a16_model_config* cfg, const w4a16_model_weights* w, int max_batch,
                                  int max_context, w4a16_model** out) {
  W4_CHECK_ARG(cfg && w && out, "model_create: null argument");
  *out = nullptr;
  const w4a16_model_config& c = *cfg;
  W4_CHECK_ARG(c.hidden > 0 && c.n_q_heads > 0 && c.n_kv_heads > 0 && c.inter > 0 && c.n_layers >= 0,
               "model_create: bad sizes");
  W4_CHECK_SHAPE(c.head_dim == 128, "model_create: head_dim must be 128");
  W4_CHECK_SHAPE(c.hidden % 128 == 0 && c.inter % 128 == 0 && (c.n_q_heads * c.head_dim) % 128 == 0,
                 "model_create: hidden, inter and Hq*D must be multiples of 128");
  W4_CHECK_SHAPE(c.n_q_heads % c.n_kv_heads == 0, "model_create: Hq %% Hkv != 0");
  W4_CHECK_ARG(max_batch >= 1 && max_context >= 1 && c.num_pages >= 1, "model_create: bad limits");
  W4_CHECK_ARG(c.n_layers == 0 || w->layers != nullptr, "model_create: null layer array");
  W4_CHECK_SHAPE(c.partition_tokens % 16 == 0 && c.partition_tokens >= 0, "model_create: partition_tokens");
  const int maxK = std::max(std::max(c.hidden, c.inter), c.n_q_heads * c.head_dim);
  W4_CHECK_SHAPE(max_batch <= 32, "model_create: max_batch=%d > 32 (one tensor-core tile of sequences)", max_batch);

  w4a16_model* m = new w4a16_model();
  m->cfg = c;
  m->layers.assign(w->layers, w->layers + c.n_layers);
  m->kv8 = c.n_layers > 0 && m->layers[0].k8 != nullptr;
  for (int l = 0; l < c.n_layers; ++l) {
    const w4a16_layer_weights& L = m->layers[l];
    const bool pools = m->kv8 ? (L.k8 && L.v8 && L.k_scale && L.v_scale) : (L.k_pool && L.v_pool && !L.k8);
    if (!(L.ln1 && L.ln2 && L.wq && L.wk && L.wv && L.wo && L.wg && L.wu && L.wd && L.sq && L.sk && L.sv && L.so &&
          L.sg && L.su && L.sd && pools)) {
      delete m;
      return set_error(W4A16_ERR_INVALID_ARG,
                       "model_create: layer %d has a null weight or pool (FP8 pools: every layer or none)", l);
    }
    const void* ptrs[] = {L.ln1, L.ln2, L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, L.sq, L.sk, L.sv, L.so, L.sg,
                          L.su,  L.sd,  L.bq, L.bk, L.bv, L.k_pool, L.v_pool, L.k8, L.v8, L.k_scale, L.v_scale};
    for (const void* p : ptrs) {
      if (p && !aligned(p, 128)) {
        delete m;
        return set_error(W4A16_ERR_ALIGNMENT, "model_create: layer %d has a weight not 128-byte aligned", l);
      }
    }
  }
  for (const void* p : {static_cast<const void*>(w->embed), static_cast<const void*>(w->final_norm),
                        static_cast<const void*>(w->lm_head)}) {
    if (p && !aligned(p, 128)) {
      delete m;
      return set_error(W4A16_ERR_ALIGNMENT, "model_create: embedding, final norm or lm_head not 128-byte aligned");
    }
  }
  m->embed = reinterpret_cast<const __half*>(w->embed);
  m->final_norm = reinterpret_cast<const __half*>(w->final_norm);
  m->lm_head = reinterpret_cast<const __half*>(w->lm_head);
  m->max_batch = max_batch;
  m->max_context = max_context;
  m->part_tokens = c.partition_tokens > 0 ? c.partition_tokens : default_partition(max_batch, c.n_kv_heads, max_context);
  m->P = (max_context + m->part_tokens - 1) / m->part_tokens;
  rope_inv_freq_table(c.theta, c.head_dim, m->inv_freq);

  const int D = c.head_dim;
  const size_t nqkv = (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * D;
  size_t off = 0;
  const size_t o_x = off; off += up256((size_t)max_batch * c.hidden * 2);
  const size_t o_qkv = off; off += up256((size_t)max_batch * nqkv * 2);
  const size_t o_att = off; off += up256((size_t)max_batch * c.n_q_heads * D * 2);
  const size_t o_h = off; off += up256((size_t)max_batch * c.hidden * 2);
  const size_t o_mlp = off; off += up256((size_t)max_batch * c.inter * 2);
  m->attn_ws_bytes = attention_workspace_bytes(max_batch, c.n_q_heads, c.n_kv_heads, m->P);
  const size_t o_aws = off; off += up256(m->attn_ws_bytes);
  m->lm_ws_bytes = lm_head_workspace_bytes(max_batch, c.vocab);
  const size_t o_lws = off; off += up256(m->lm_ws_bytes);
  const size_t o_xn = off; off += up256((size_t)max_batch * maxK * 2);
  const size_t o_l32 = off; off += max_batch > GEMV_MAX_BATCH ? up256((size_t)max_batch * c.vocab * 4) : 0;
  {
    auto need = [&](int N, int K, bool silu) {
      int ks = 1, ps = 0;
      tc_plan(N, K, true, silu, true, &ks, &ps);
      m->tc_ws_bytes = std::max(m->tc_ws_bytes, tc_workspace_bytes(N, ks, silu));
    };
    need((int)nqkv, c.hidden, false);
    need(c.hidden, c.n_q_heads * D, false);
    need(c.inter, c.hidden, true);
    need(c.hidden, c.inter, false);
  }
  const size_t o_tws = off; off += up256(m->tc_ws_bytes);
  const size_t o_err = off; off += 256;
  // the persistent path: one sequence, the Qwen2-style 7:1 GQA shapes, contexts
  // its attention merge covers
  m->pk_ok = persistent_supported(c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.inter, c.n_layers, max_context) &&
             c.vocab >= 2 && c.vocab % 2 == 0 && !m->kv8;
  size_t o_pk = off;
  if (m->pk_ok) {
    m->pk_P = (max_context + PK_PARTITION_TOKENS - 1) / PK_PARTITION_TOKENS;
    off += up256(persistent_workspace_bytes(c.n_kv_heads, max_context, c.n_layers));
  }
  m->arena_bytes = off;
  cudaError_t e = cudaMalloc(&m->arena, off);
  if (e != cudaSuccess) {
    delete m;
    return set_error(W4A16_ERR_CUDA, "model_create: arena of %zu bytes: %s", off, cudaGetErrorString(e));
  }
  cudaMemset(m->arena, 0, off);
  m->x = reinterpret_cast<__half*>(m->arena + o_x);
  m->qkv = reinterpret_cast<__half*>(m->arena + o_qkv);
  m->att = reinterpret_cast<__half*>(m->arena + o_att);
  m->h = reinterpret_cast<__half*>(m->arena + o_h);
  m->mlp = reinterpret_cast<__half*>(m->arena + o_mlp);
  m->attn_ws = m->arena + o_aws;
  m->lm_ws = m->arena + o_lws;
  m->xn = reinterpret_cast<__half*>(m->arena + o_xn);
  m->logits32 = max_batch > GEMV_MAX_BATCH ? reinterpret_cast<float*>(m->arena + o_l32) : nullptr;
  m->tc_ws = m->arena + o_tws;
  m->err_flag = reinterpret_cast<int32_t*>(m->arena + o_err);
  if (m->pk_ok) {
    char* p = m->arena + o_pk;
    m->pk_layers = reinterpret_cast<PkLayer*>(p);
    p += up256((size_t)c.n_layers * sizeof(PkLayer));
    m->pk_att_part = reinterpret_cast<float*>(p);
    p += up256((size_t)c.n_kv_heads * m->pk_P * 7 * (c.head_dim + 4) * 4);  // 16-byte aligned records
    m->pk_att_tickets = reinterpret_cast<unsigned*>(p);
    m->pk_att_tickets_bytes = up256((size_t)c.n_kv_heads * 4);
    p += m->pk_att_tickets_bytes;
    m->pk_lm_keys = reinterpret_cast<unsigned long long*>(p);
    p += up256((size_t)1024 * 8);
    m->pk_ctl = reinterpret_cast<unsigned*>(p);
    std::vector<PkLayer> tab(c.n_layers);
    auto hp = [](const uint16_t* q) { return reinterpret_cast<const __half*>(q); };
    for (int l = 0; l < c.n_layers; ++l) {
      const w4a16_layer_weights& L = m->layers[l];
      tab[l] = PkLayer{L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, hp(L.sq), hp(L.sk), hp(L.sv), hp(L.so), hp(L.sg),
                       hp(L.su), hp(L.sd), hp(L.bq), hp(L.bk), hp(L.bv), hp(L.ln1), hp(L.ln2),
                       reinterpret_cast<__half*>(L.k_pool), reinterpret_cast<__half*>(L.v_pool)};
    }
    e = cudaMemcpy(m->pk_layers, tab.data(), tab.size() * sizeof(PkLayer), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      cudaFree(m->arena);
      delete m;
      return set_error(W4A16_ERR_CUDA, "model_create: layer table: %s", cudaGetErrorString(e));
    }
  }
  e = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(m->arena);
    delete m;
    return set_error(W4A16_ERR_CUDA, "model_create: %s", cudaGetErrorString(e));
  }
  *out = m;
  return W4A16_OK;
}

extern "C" void w4a16_model_destroy(w4a16_model* m) {
  if (!m) return;
  for (auto& kv : m->graphs) cudaGraphExecDestroy(kv.second);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  if (m->arena) cudaFree(m->arena);
  delete m;
}

extern "C" int32_t* w4a16_model_err_flag(w4a16_model* m) { return m ? m->err_flag : nullptr; }

extern "C" int w4a16_model_hidden(w4a16_model* m, uint16_t* dst, int B, w4a16_stream_t stream) {
  W4_CHECK_ARG(m && dst, "model_hidden: null argument");
  W4_CHECK_ARG(B >= 1 && B <= m->max_batch, "model_hidden: B=%d", B);
  cudaError_t e = cudaMemcpyAsync(dst, m->x, (size_t)B * m->cfg.hidden * 2, cudaMemcpyDeviceToDevice,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "model_hidden: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

extern "C" int w4a16_model_activation(w4a16_model* m, int which, uint16_t* dst, int B, w4a16_stream_t stream) {
  W4_CHECK_ARG(m && dst, "model_activation: null argument");
  W4_CHECK_ARG(B >= 1 && B <= m->max_batch, "model_activation: B=%d", B);
  const w4a16_model_config& c = m->cfg;
  const __half* src = nullptr;
  size_t width = 0;
  switch (which) {
    case W4A16_ACT_HIDDEN: src = m->x; width = c.hidden; break;
    case W4A16_ACT_QKV: src = m->qkv; width = (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim; break;
    case W4A16_ACT_ATTN: src = m->att; width = (size_t)c.n_q_heads * c.head_dim; break;
    case W4A16_ACT_RESID: src = m->h; width = c.hidden; break;
    case W4A16_ACT_MLP: src = m->mlp; width = c.inter; break;
    default: return set_error(W4A16_ERR_INVALID_ARG, "model_activation: unknown buffer %d", which);
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)B * width * 2, cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "model_activation: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

extern "C" int w4a16_model_check_errors(w4a16_model* m, w4a16_stream_t stream) {
  W4_CHECK_ARG(m, "model_check_errors: null model");
  cudaStream_t s = (cudaStream_t)stream;
  cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cst) == cudaSuccess && cst != cudaStreamCaptureStatusNone)
    return set_error(W4A16_ERR_CAPTURE, "model_check_errors: stream is capturing");
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, m->err_flag, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(m->err_flag, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "model_check_errors: %s", cudaGetErrorString(e));
  if (host & 2) {
    // a CTA that gave up left its split-K tiles unfinished: their tickets
    // may be part-counted, so every ticket block is cleared before the next step
    e = cudaMemsetAsync(m->tc_ws, 0, std::min(m->tc_ws_bytes, TC_TICKET_BYTES), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->attn_ws, 0, std::min(m->attn_ws_bytes, ATT_TICKET_BYTES), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->lm_ws, 0, m->lm_ws_bytes, s);
    // the persistent kernel's barrier and step counters restart together
    if (e == cudaSuccess && m->pk_ok) e = cudaMemsetAsync(m->pk_ctl, 0, PK_CTL_WORDS * 4, s);
    if (e == cudaSuccess && m->pk_ok) e = cudaMemsetAsync(m->pk_att_tickets, 0, m->pk_att_tickets_bytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "model_check_errors: %s", cudaGetErrorString(e));
    return set_error(W4A16_ERR_TIMEOUT, "a bounded device wait gave up (flag 0x%x)", host);
  }
  if (host & 1) return set_error(W4A16_ERR_DEVICE_BOUNDS, "a kernel skipped an out-of-range index (flag 0x%x)", host);
  return W4A16_OK;
}

// One projection.  Small batches take the CUDA-core GEMV (RMSNorm fused in
// front); otherwise the RMSNorm (if any) runs on its own into m->xn and the
// tensor-core GEMM follows with K split across CTAs.  Returns the number of
// tags used through *tag.
static int project(w4a16_model* m, GemvArgs g, bool silu, cudaStream_t s, int* tag) {
  if (gemv_cuda_core_supported(g.M, g.K) && !(g.gamma && batched_path(m, g.M)) &&
      !(silu && g.M >= SILU_TC_MIN_ROWS)) {
    g.tag = (*tag)++;
    return launch_gemv(g, silu, s);
  }
  int rc;
  if (g.gamma) {
    if ((rc = launch_rmsnorm(g.x, g.gamma, m->xn, g.M, g.K, g.eps, s, (*tag)++))) return rc;
    g.x = m->xn;
  }
  TcArgs t = {};
  t.x = g.x;
  t.residual = g.residual;
  t.y = g.y;
  for (int i = 0; i < 3; ++i) t.seg[i] = g.seg[i];
  t.nseg = g.nseg;
  t.err_flag = m->err_flag;
  t.M = g.M;
  t.K = g.K;
  t.N = g.N;
  t.ldy = g.N;
  tc_plan(g.N, g.K, true, silu, true, &t.ksplit, &t.per_split);
  if (t.ksplit > 1 && tc_workspace_bytes(g.N, t.ksplit, silu) > m->tc_ws_bytes)
    tc_plan(g.N, g.K, true, silu, false, &t.ksplit, &t.per_split);
  if (t.ksplit > 1) tc_workspace_layout(t, m->tc_ws);
  t.tag = (*tag)++;
  return launch_gemm_tc(t, true, silu, s);
}

static int run_layer(w4a16_model* m, int l, __half* x, const int32_t* bt, int max_blocks, const int32_t* lens, int B,
                     cudaStream_t s, int tag0 = 0) {
  const w4a16_model_config& c = m->cfg;
  const w4a16_layer_weights& L = m->layers[l];
  const int D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, H = c.hidden, I = c.inter;
  const int nqkv = (Hq + 2 * Hkv) * D;
  auto hp = [](const uint16_t* p) { return reinterpret_cast<const __half*>(p); };
  int rc;

  GemvArgs g = {};
  g.x = x;
  g.gamma = hp(L.ln1);
  g.eps = c.eps;
  g.y = m->qkv;
  g.seg[0] = {L.wq, hp(L.sq), hp(L.bq), Hq * D};
  g.seg[1] = {L.wk, hp(L.sk), hp(L.bk), Hkv * D};
  g.seg[2] = {L.wv, hp(L.sv), hp(L.bv), Hkv * D};
  g.nseg = 3;
  g.M = B;
  g.K = H;
  g.N = nqkv;
  int tag = tag0;
  if ((rc = project(m, g, false, s, &tag))) return rc;

  // RoPE of q and the new k, the KV append and the paged attention are one
  // kernel: it prefetches this partition's pages while the q|k|v GEMV runs.
  AttnArgs a = {};
  a.q = m->qkv;
  a.q_stride = nqkv;
  a.k_pool = reinterpret_cast<__half*>(L.k_pool);
  a.v_pool = reinterpret_cast<__half*>(L.v_pool);
  if (m->kv8) {
    a.kv8 = 1;
    a.k8 = L.k8;
    a.v8 = L.v8;
    a.ks = L.k_scale;
    a.vs = L.v_scale;
  }
  a.block_table = bt;
  a.context_lens = lens;
  a.out = m->att;
  attention_workspace_layout(a, m->attn_ws, m->max_batch, Hq, m->P);
  a.err_flag = m->err_flag;
  a.num_pages = c.num_pages;
  a.max_blocks = max_blocks;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = m->P;
  a.part_tokens = m->part_tokens;
  a.scale_log2 = (1.0f / sqrtf((float)D)) * 1.4426950408889634f;
  a.fuse_rope_append = 1;
  std::memcpy(a.inv_freq, m->inv_freq, sizeof(a.inv_freq));
  a.tag = tag++;
  if ((rc = launch_paged_attention(a, s))) return rc;

  GemvArgs o = {};
  o.x = m->att;
  o.residual = x;
  o.y = m->h;
  o.seg[0] = {L.wo, hp(L.so), nullptr, H};
  o.nseg = 1;
  o.M = B;
  o.K = Hq * D;
  o.N = H;
  if ((rc = project(m, o, false, s, &tag))) return rc;

  GemvArgs gu = {};
  gu.x = m->h;
  gu.gamma = hp(L.ln2);
  gu.eps = c.eps;
  gu.y = m->mlp;
  gu.seg[0] = {L.wg, hp(L.sg), nullptr, I};
  gu.seg[1] = {L.wu, hp(L.su), nullptr, I};
  gu.nseg = 2;
  gu.M = B;
  gu.K = H;
  gu.N = I;
  if ((rc = project(m, gu, true, s, &tag))) return rc;

  GemvArgs dn = {};
  dn.x = m->mlp;
  dn.residual = m->h;
  dn.y = x;
  dn.seg[0] = {L.wd, hp(L.sd), nullptr, H};
  dn.nseg = 1;
  dn.M = B;
  dn.K = I;
  dn.N = H;
  return project(m, dn, false, s, &tag);
}

// ---------------------------------------------------------------------------
// Prefill: the T prompt tokens of one sequence in one pass (the "TTFT (512
// tokens)" row of the aikraft.ru article's "Ключевые метрики
// производительности").  Each projection is a tensor-core GEMM over the T
// rows (row blocks of up to 128); RoPE + append write all T positions into
// the sequence's pages; the attention gives row i the keys at positions
// 0 .. len0 + i (causal attention over the prompt and any tokens cached
// before it), 16 rows per CTA sharing every page they read.
// ---------------------------------------------------------------------------
struct PrefillWs {
  __half *x, *xn, *qkv, *att, *h, *mlp;
  int32_t *bt_rep, *lens;
  void* tc;         // split-K workspace of the tensor-core GEMMs (tickets first)
  size_t tc_bytes;
};

// rows per tensor-core GEMM launch of the prompt, and that launch's split-K
// workspace need (the largest over the layer's projections)
static size_t prefill_tc_bytes(const w4a16_model_config& c, int T) {
  const int D = c.head_dim;
  const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * D;
  const struct { int N, K; bool silu; } proj[4] = {
      {nqkv, c.hidden, false}, {c.hidden, c.n_q_heads * D, false}, {c.inter, c.hidden, true}, {c.hidden, c.inter, false}};
  size_t need = TC_TICKET_BYTES;
  for (const auto& p : proj) {
    const int rows = std::min(T, tc_max_rows(true, p.silu));
    const int nc = tc_cols(rows, true, p.silu);
    int ks = 1, ps = 0;
    tc_plan(p.N, p.K, true, p.silu, true, &ks, &ps, nc);
    if (ks > 1) need = std::max(need, tc_workspace_bytes(p.N, ks, p.silu, nc));
  }
  return need;
}

static size_t prefill_layout(const w4a16_model* m, int T, int max_blocks, char* base, PrefillWs* w) {
  const w4a16_model_config& c = m->cfg;
  const size_t D = c.head_dim, nqkv = (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * D;
  const size_t maxK = std::max(std::max((size_t)c.hidden, (size_t)c.inter), (size_t)c.n_q_heads * D);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes);
    return base ? base + o : nullptr;
  };
  char* px = take((size_t)T * c.hidden * 2);
  char* pxn = take((size_t)T * maxK * 2);
  char* pqkv = take((size_t)T * nqkv * 2);
  char* patt = take((size_t)T * c.n_q_heads * D * 2);
  char* ph = take((size_t)T * c.hidden * 2);
  char* pmlp = take((size_t)T * c.inter * 2);
  char* pbt = take((size_t)T * max_blocks * 4);
  char* pl = take((size_t)T * 4);
  const size_t tcb = prefill_tc_bytes(c, T);
  char* ptc = take(tcb);
  if (w) {
    w->x = reinterpret_cast<__half*>(px);
    w->xn = reinterpret_cast<__half*>(pxn);
    w->qkv = reinterpret_cast<__half*>(pqkv);
    w->att = reinterpret_cast<__half*>(patt);
    w->h = reinterpret_cast<__half*>(ph);
    w->mlp = reinterpret_cast<__half*>(pmlp);
    w->bt_rep = reinterpret_cast<int32_t*>(pbt);
    w->lens = reinterpret_cast<int32_t*>(pl);
    w->tc = ptc;
    w->tc_bytes = tcb;
  }
  return off;
}

extern "C" size_t w4a16_prefill_workspace_size(w4a16_model* m, int T, int max_blocks) {
  if (!m || T < 1 || max_blocks < 1) return 0;
  return prefill_layout(m, T, max_blocks, nullptr, nullptr);
}

// y[T][N] = x[T][K] . W^T (+bias, +residual; SiLU-mul for gate|up) on the
// tensor cores in row blocks of up to 128 (64 for gate|up, whose two weight
// matrices share the tile's tensor memory), so each weight tile is read once
// per block
static int gemm_rows(w4a16_model* m, const PrefillWs& w, const __half* x, int T, int K, const GemvSeg* segs, int nseg,
                     int N, const __half* residual, __half* y, bool silu, cudaStream_t s) {
  const int rows = tc_max_rows(true, silu);
  for (int r0 = 0; r0 < T; r0 += rows) {
    TcArgs t = {};
    t.x = x + (size_t)r0 * K;
    t.residual = residual ? residual + (size_t)r0 * N : nullptr;
    t.y = y + (size_t)r0 * N;
    for (int i = 0; i < nseg; ++i) t.seg[i] = segs[i];
    t.nseg = nseg;
    t.err_flag = m->err_flag;
    t.M = std::min(rows, T - r0);
    t.K = K;
    t.N = N;
    t.ldy = N;
    const int nc = tc_cols(t.M, true, silu);
    tc_plan(N, K, true, silu, true, &t.ksplit, &t.per_split, nc);
    if (t.ksplit > 1 && tc_workspace_bytes(N, t.ksplit, silu, nc) > w.tc_bytes)
      tc_plan(N, K, true, silu, false, &t.ksplit, &t.per_split, nc);
    if (t.ksplit > 1) tc_workspace_layout(t, w.tc);
    const int rc = launch_gemm_tc(t, true, silu, s);
    if (rc) return rc;
  }
  return W4A16_OK;
}

extern "C" int w4a16_prefill(w4a16_model* m, const int32_t* tokens, int T, const int32_t* block_table,
                             int max_blocks, int32_t* context_lens, int32_t* token_out, uint16_t* logits,
                             void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  W4_CHECK_ARG(m && tokens && block_table && context_lens && token_out && workspace, "prefill: null argument");
  W4_CHECK_ARG(m->embed && m->final_norm && m->lm_head && m->cfg.vocab > 0, "prefill: model has no lm_head");
  W4_CHECK_ARG(T >= 1 && max_blocks >= 1, "prefill: T=%d max_blocks=%d", T, max_blocks);
  W4_CHECK_SHAPE(T <= m->max_context, "prefill: %d tokens > max_context %d", T, m->max_context);
  W4_CHECK_ALIGN(workspace, 256, "workspace");
  W4_CHECK_ALIGN(logits, 128, "logits");
  const size_t need = prefill_layout(m, T, max_blocks, nullptr, nullptr);
  W4_CHECK_ARG(workspace_bytes >= need, "prefill: workspace of %zu bytes needed", need);
  const w4a16_model_config& c = m->cfg;
  const int D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, H = c.hidden, I = c.inter;
  const int nqkv = (Hq + 2 * Hkv) * D;
  cudaStream_t s = (cudaStream_t)stream;
  PrefillWs w;
  prefill_layout(m, T, max_blocks, static_cast<char*>(workspace), &w);
  auto hp = [](const uint16_t* p) { return reinterpret_cast<const __half*>(p); };
  int rc;
  // split-K tickets of the GEMMs start at zero (each call leaves them zero)
  if (cudaMemsetAsync(w.tc, 0, TC_TICKET_BYTES, s) != cudaSuccess)
    return set_error(W4A16_ERR_CUDA, "prefill: workspace memset failed");
  if ((rc = launch_embedding(m->embed, c.vocab, H, tokens, T, w.x, m->err_flag, nullptr, 0, s))) return rc;
  if ((rc = launch_prefill_rows(block_table, max_blocks, context_lens, T, w.bt_rep, w.lens, s))) return rc;
  for (int l = 0; l < c.n_layers; ++l) {
    const w4a16_layer_weights& L = m->layers[l];
    if ((rc = launch_rmsnorm(w.x, hp(L.ln1), w.xn, T, H, c.eps, s))) return rc;
    const GemvSeg qkv[3] = {{L.wq, hp(L.sq), hp(L.bq), Hq * D}, {L.wk, hp(L.sk), hp(L.bk), Hkv * D},
                            {L.wv, hp(L.sv), hp(L.bv), Hkv * D}};
    if ((rc = gemm_rows(m, w, w.xn, T, H, qkv, 3, nqkv, nullptr, w.qkv, false, s))) return rc;
    RopeArgs ra = {};
    ra.q = w.qkv;
    ra.k = w.qkv + (size_t)Hq * D;
    ra.v = w.qkv + (size_t)(Hq + Hkv) * D;
    ra.k_pool = reinterpret_cast<__half*>(L.k_pool);
    ra.v_pool = reinterpret_cast<__half*>(L.v_pool);
    if (m->kv8) {  // FP8 pages: quantised rows appended
      ra.k8 = L.k8;
      ra.v8 = L.v8;
      ra.ks = L.k_scale;
      ra.vs = L.v_scale;
    }
    ra.block_table = w.bt_rep;
    ra.context_lens = w.lens;
    ra.err_flag = m->err_flag;
    ra.stride_q = nqkv;
    ra.stride_kv = nqkv;
    ra.num_pages = c.num_pages;
    ra.max_blocks = max_blocks;
    ra.B = T;
    ra.Hq = Hq;
    ra.Hkv = Hkv;
    std::memcpy(ra.inv_freq, m->inv_freq, sizeof(ra.inv_freq));
    if ((rc = launch_rope_append(ra, s))) return rc;
    AttnArgs a = {};
    a.q = w.qkv;
    a.q_stride = nqkv;
    a.k_pool = ra.k_pool;
    a.v_pool = ra.v_pool;
    if (m->kv8) {
      a.kv8 = 1;
      a.k8 = L.k8;
      a.v8 = L.v8;
      a.ks = L.k_scale;
      a.vs = L.v_scale;
    }
    a.block_table = w.bt_rep;
    a.context_lens = w.lens;
    a.out = w.att;
    a.err_flag = m->err_flag;
    a.num_pages = c.num_pages;
    a.max_blocks = max_blocks;
    a.B = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.scale_log2 = (1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    if ((rc = launch_prefill_attention(a, s))) return rc;
    const GemvSeg o[1] = {{L.wo, hp(L.so), nullptr, H}};
    if ((rc = gemm_rows(m, w, w.att, T, Hq * D, o, 1, H, w.x, w.h, false, s))) return rc;
    if ((rc = launch_rmsnorm(w.h, hp(L.ln2), w.xn, T, H, c.eps, s))) return rc;
    const GemvSeg gu[2] = {{L.wg, hp(L.sg), nullptr, I}, {L.wu, hp(L.su), nullptr, I}};
    if ((rc = gemm_rows(m, w, w.xn, T, H, gu, 2, I, nullptr, w.mlp, true, s))) return rc;
    const GemvSeg dn[1] = {{L.wd, hp(L.sd), nullptr, H}};
    if ((rc = gemm_rows(m, w, w.mlp, T, I, dn, 1, H, w.h, w.x, false, s))) return rc;
  }
  // the last prompt token's logits and greedy next token
  LmHeadArgs la = {};
  la.x = w.x + (size_t)(T - 1) * H;
  la.w = m->lm_head;
  la.gamma = m->final_norm;
  la.eps = c.eps;
  la.logits = reinterpret_cast<__half*>(logits);
  la.tokens_out = token_out;
  la.partial = reinterpret_cast<unsigned long long*>(m->lm_ws);
  la.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(m->lm_ws) + (size_t)4 * 4096 * 8);
  la.B = 1;
  la.H = H;
  la.vocab = c.vocab;
  if ((rc = launch_lm_head_argmax(la, s))) return rc;
  return launch_advance_len(context_lens, T, m->max_context, m->err_flag, s);
}

// kernels one layer launches at batch B
static int layer_kernel_count(const w4a16_model* m, int B) {
  return batched_path(m, B) ? 7 : (B >= SILU_TC_MIN_ROWS ? 6 : 5);
}

extern "C" int w4a16_model_layer(w4a16_model* m, int layer, uint16_t* x, const int32_t* block_table, int max_blocks,
                                 const int32_t* context_lens, int B, w4a16_stream_t stream) {
  W4_CHECK_ARG(m && x && block_table && context_lens, "model_layer: null argument");
  W4_CHECK_ARG(layer >= 0 && layer < m->cfg.n_layers, "model_layer: layer %d out of range", layer);
  W4_CHECK_ARG(B >= 1 && B <= m->max_batch && max_blocks >= 1, "model_layer: B=%d (max %d)", B, m->max_batch);
  W4_CHECK_ALIGN(x, 128, "x");
  return run_layer(m, layer, reinterpret_cast<__half*>(x), block_table, max_blocks, context_lens, B,
                   (cudaStream_t)stream);
}

static int enqueue_step(w4a16_model* m, const int32_t* tin, int32_t* tout, const int32_t* bt, int max_blocks,
                        int32_t* lens, int B, uint16_t* logits, cudaStream_t s) {
  const w4a16_model_config& c = m->cfg;
  int rc = launch_embedding(m->embed, c.vocab, c.hidden, tin, B, m->x, m->err_flag, lens, m->max_context, s, 0);
  if (rc) return rc;
  const int per_layer = layer_kernel_count(m, B);
  for (int l = 0; l < c.n_layers; ++l)
    if ((rc = run_layer(m, l, m->x, bt, max_blocks, lens, B, s, 1 + per_layer * l))) return rc;
  const int tag = 1 + per_layer * c.n_layers;
  if (batched_path(m, B)) {
    // final RMSNorm, lm_head on the tensor cores (fp32 logits), argmax
    if ((rc = launch_rmsnorm(m->x, m->final_norm, m->xn, B, c.hidden, c.eps, s, tag))) return rc;
    TcArgs t = {};
    t.x = m->xn;
    t.y32 = m->logits32;
    t.w16 = m->lm_head;
    t.err_flag = m->err_flag;
    t.M = B;
    t.K = c.hidden;
    t.N = c.vocab;
    t.ldy = c.vocab;
    t.ksplit = 1;
    t.tag = tag + 1;
    if ((rc = launch_gemm_tc(t, false, false, s))) return rc;
    return launch_argmax_rows(m->logits32, B, c.vocab, tout, reinterpret_cast<__half*>(logits), s, tag + 2);
  }
  LmHeadArgs a = {};
  a.x = m->x;
  a.w = m->lm_head;
  a.gamma = m->final_norm;
  a.eps = c.eps;
  a.logits = reinterpret_cast<__half*>(logits);
  a.tokens_out = tout;
  a.partial = reinterpret_cast<unsigned long long*>(m->lm_ws);
  a.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(m->lm_ws) + (size_t)4 * 4096 * 8);
  a.B = B;
  a.H = c.hidden;
  a.vocab = c.vocab;
  a.tag = tag;
  return launch_lm_head_argmax(a, s);
}

// decode_step takes the persistent kernel for this batch size: when asked
// for, or by default where it is the faster path (see PK_IS_DEFAULT)
static constexpr bool PK_IS_DEFAULT = false;
static bool use_persistent(const w4a16_model* m, int B) {
  if (!m->pk_ok || B != 1) return false;
  return m->decode_path == W4A16_PATH_PERSISTENT || (m->decode_path == W4A16_PATH_AUTO && PK_IS_DEFAULT);
}

static int enqueue_persistent(w4a16_model* m, const int32_t* tin, int32_t* tout, const int32_t* bt, int max_blocks,
                              int32_t* lens, uint16_t* logits, cudaStream_t s) {
  const w4a16_model_config& c = m->cfg;
  PkArgs a = {};
  a.layers = m->pk_layers;
  a.n_layers = c.n_layers;
  a.embed = m->embed;
  a.final_norm = m->final_norm;
  a.lm_head = m->lm_head;
  a.tokens_in = tin;
  a.tokens_out = tout;
  a.block_table = bt;
  a.max_blocks = max_blocks;
  a.context_lens = lens;
  a.logits = reinterpret_cast<__half*>(logits);
  a.x = m->x;
  a.qkv = m->qkv;
  a.att = m->att;
  a.h = m->h;
  a.mlp = m->mlp;
  a.att_part = m->pk_att_part;
  a.att_tickets = m->pk_att_tickets;
  a.lm_keys = m->pk_lm_keys;
  a.ctl = m->pk_ctl;
  a.err_flag = m->err_flag;
  a.H = c.hidden;
  a.Hq = c.n_q_heads;
  a.Hkv = c.n_kv_heads;
  a.I = c.inter;
  a.vocab = c.vocab;
  a.num_pages = c.num_pages;
  a.max_context = m->max_context;
  a.P = m->pk_P;
  a.eps = c.eps;
  a.scale_log2 = (1.0f / sqrtf((float)c.head_dim)) * 1.4426950408889634f;
  a.wait_limit_ns = tc_wait_limit_ns();
  std::memcpy(a.inv_freq, m->inv_freq, sizeof(a.inv_freq));
  return launch_persistent(a, s);
}

extern "C" int decode_step_kernel_count(w4a16_model* m, int B) {
  if (!m) return 0;
  if (use_persistent(m, B)) return 1;
  return 1 + layer_kernel_count(m, B) * m->cfg.n_layers + (batched_path(m, B) ? 3 : 1);
}

extern "C" int w4a16_model_set_decode_path(w4a16_model* m, int path) {
  W4_CHECK_ARG(m, "model_set_decode_path: null model");
  W4_CHECK_ARG(path == W4A16_PATH_AUTO || path == W4A16_PATH_KERNELS || path == W4A16_PATH_PERSISTENT,
               "model_set_decode_path: unknown path %d", path);
  if (path == W4A16_PATH_PERSISTENT && !m->pk_ok)
    return set_error(W4A16_ERR_SHAPE, "model_set_decode_path: the persistent kernel does not cover this model "
                                      "(one sequence, head_dim 128, Hq = 7 Hkv, max_context <= %d, fp16 KV pools)",
                     PK_MAX_CONTEXT);
  std::lock_guard<std::mutex> lk(m->mu);
  m->decode_path = path;
  return W4A16_OK;
}

extern "C" int w4a16_model_decode_path(w4a16_model* m, int B) {
  if (!m) return -1;
  return use_persistent(m, B) ? W4A16_PATH_PERSISTENT : W4A16_PATH_KERNELS;
}

extern "C" int decode_step(w4a16_model* m, const int32_t* tokens_in, int32_t* tokens_out, const int32_t* block_table,
                           int max_blocks, int32_t* context_lens, int B, uint16_t* logits, int use_graph,
                           w4a16_stream_t stream) {
  W4_CHECK_ARG(m && tokens_in && tokens_out && block_table && context_lens, "decode_step: null argument");
  W4_CHECK_ARG(m->embed && m->final_norm && m->lm_head && m->cfg.vocab > 0, "decode_step: model has no lm_head");
  W4_CHECK_ARG(B >= 1 && B <= m->max_batch && max_blocks >= 1, "decode_step: B=%d (max %d)", B, m->max_batch);
  W4_CHECK_ALIGN(logits, 128, "logits");
  cudaStream_t s = (cudaStream_t)stream;
  const bool pk = use_persistent(m, B);
  auto enqueue = [&](cudaStream_t st) {
    return pk ? enqueue_persistent(m, tokens_in, tokens_out, block_table, max_blocks, context_lens, logits, st)
              : enqueue_step(m, tokens_in, tokens_out, block_table, max_blocks, context_lens, B, logits, st);
  };
  if (!use_graph) return enqueue(s);

  cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
  if (s != nullptr && cudaStreamIsCapturing(s, &cst) == cudaSuccess && cst == cudaStreamCaptureStatusActive) {
    // The caller is capturing already: record the kernels into their graph.
    return enqueue(s);
  }
  GraphKey key{B, max_blocks, pk ? 1 : 0, tokens_in, tokens_out, block_table, context_lens, logits};
  cudaGraphExec_t exec = nullptr;
  {
    std::lock_guard<std::mutex> lk(m->mu);
    auto it = m->graphs.find(key);
    if (it != m->graphs.end()) exec = it->second;
  }
  if (!exec) {
    // Capture on the model's private stream (the legacy default stream cannot
    // capture); nothing but kernel launches is recorded.
    cudaError_t e = cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) return set_error(W4A16_ERR_CAPTURE, "decode_step: begin capture: %s", cudaGetErrorString(e));
    int rc = enqueue(m->cap_stream);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(m->cap_stream, &graph);
    if (rc != W4A16_OK) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (e != cudaSuccess) return set_error(W4A16_ERR_CAPTURE, "decode_step: end capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "decode_step: instantiate: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(m->mu);
    m->graphs[key] = exec;
  }
  cudaError_t e = cudaGraphLaunch(exec, s);
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "decode_step: graph launch: %s", cudaGetErrorString(e));
  return W4A16_OK;
}

#ifdef W4A16_TRACE
namespace w4 {
extern __device__ TraceRec* g_trace_buf;
extern __device__ unsigned int g_trace_cap;
extern __device__ unsigned int g_trace_n;
}
// Kernel timeline (trace builds only): start recording into a device buffer
// of `cap` records of 64 bytes; w4a16_trace_count returns how many were
// written (synchronises the device).
extern "C" W4A16_API int w4a16_trace_start(void* dev_buf, unsigned int cap) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyToSymbol(w4::g_trace_buf, &dev_buf, sizeof(void*));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(w4::g_trace_cap, &cap, sizeof(cap));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(w4::g_trace_n, &zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? W4A16_OK : set_error(W4A16_ERR_CUDA, "trace_start: %s", cudaGetErrorString(e));
}
extern "C" W4A16_API unsigned int w4a16_trace_count(void) {
  unsigned int n = 0;
  cudaDeviceSynchronize();
  cudaMemcpyFromSymbol(&n, w4::g_trace_n, sizeof(n));
  return n;
}
#endif
