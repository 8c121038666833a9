// batcher.cu -- host page allocator and continuous batching over decode_step.
//
// "Building a Custom LLM Inference Runtime on H100" (explore.n1n.ai), "2. The
// KV Cache and PagedAttention", treats the KV cache like virtual memory:
// fixed-size pages handed out as sequences grow, so that sequences need no
// contiguous reservation and the batch can be as large as memory allows
// ("Why Build from Scratch?": maximise batch sizes).  This file is the host
// side of that: a free list over a pool's pages, block-table rows that grow
// one page every 16 tokens, and a scheduler that keeps a decode batch full
// -- sequences join as others finish, their pages go back to the free list,
// and each step runs the model for the sequences now active (decode_step
// captures one CUDA graph per batch size, so batch sizes are graph buckets).
//
// A sequence's prompt is fed through decode steps one token at a time
// (outputs discarded until its last prompt token, whose output is the first
// generated token).  When a step needs a page and the pool is empty, the
// most recently admitted sequence is preempted: its pages are freed and it
// goes back to the front of the queue to start again from its prompt (greedy
// decoding makes the restarted sequence produce the same tokens).
#include <algorithm>
#include <deque>
#include <map>
#include <mutex>
#include <vector>

#include "common.cuh"

// ---------------------------------------------------------------------------
// Page allocator
// ---------------------------------------------------------------------------
struct w4a16_page_allocator {
  int num_pages = 0;
  std::vector<int32_t> free_list;  // stack; the next page handed out is free_list.back()
  std::vector<uint8_t> used;       // 1 while a page is handed out
  std::mutex mu;
};

extern "C" int w4a16_page_allocator_create(int num_pages, w4a16_page_allocator** out) {
  W4_CHECK_ARG(out != nullptr, "page_allocator_create: null out");
  *out = nullptr;
  W4_CHECK_ARG(num_pages >= 1, "page_allocator_create: num_pages=%d", num_pages);
  auto* a = new w4a16_page_allocator();
  a->num_pages = num_pages;
  a->free_list.resize(num_pages);
  for (int i = 0; i < num_pages; ++i) a->free_list[i] = num_pages - 1 - i;  // page 0 first
  a->used.assign(num_pages, 0);
  *out = a;
  return W4A16_OK;
}

extern "C" void w4a16_page_allocator_destroy(w4a16_page_allocator* a) { delete a; }

extern "C" int w4a16_page_free_count(w4a16_page_allocator* a) {
  if (!a) return -1;
  std::lock_guard<std::mutex> lk(a->mu);
  return (int)a->free_list.size();
}

static int alloc_locked(w4a16_page_allocator* a, int n, int32_t* pages) {
  if ((int)a->free_list.size() < n)
    return w4::set_error(W4A16_ERR_NO_PAGES, "page_alloc: %d pages wanted, %d free", n, (int)a->free_list.size());
  for (int i = 0; i < n; ++i) {
    const int32_t p = a->free_list.back();
    a->free_list.pop_back();
    a->used[p] = 1;
    pages[i] = p;
  }
  return W4A16_OK;
}

static int free_locked(w4a16_page_allocator* a, const int32_t* pages, int n) {
  // validate everything first: a bad call frees nothing
  std::vector<int32_t> seen;
  seen.reserve(n);
  for (int i = 0; i < n; ++i) {
    const int32_t p = pages[i];
    if (p < 0 || p >= a->num_pages)
      return w4::set_error(W4A16_ERR_INVALID_ARG, "page_free: page %d outside [0, %d)", p, a->num_pages);
    if (!a->used[p]) return w4::set_error(W4A16_ERR_INVALID_ARG, "page_free: page %d is not handed out", p);
    seen.push_back(p);
  }
  std::sort(seen.begin(), seen.end());
  if (std::adjacent_find(seen.begin(), seen.end()) != seen.end())
    return w4::set_error(W4A16_ERR_INVALID_ARG, "page_free: a page appears twice in one call");
  for (int i = 0; i < n; ++i) {
    a->used[pages[i]] = 0;
    a->free_list.push_back(pages[i]);
  }
  return W4A16_OK;
}

extern "C" int w4a16_page_alloc(w4a16_page_allocator* a, int n, int32_t* pages) {
  W4_CHECK_ARG(a && (pages || n == 0), "page_alloc: null argument");
  W4_CHECK_ARG(n >= 0, "page_alloc: n=%d", n);
  std::lock_guard<std::mutex> lk(a->mu);
  return alloc_locked(a, n, pages);
}

extern "C" int w4a16_page_free(w4a16_page_allocator* a, const int32_t* pages, int n) {
  W4_CHECK_ARG(a && (pages || n == 0), "page_free: null argument");
  W4_CHECK_ARG(n >= 0, "page_free: n=%d", n);
  std::lock_guard<std::mutex> lk(a->mu);
  return free_locked(a, pages, n);
}

extern "C" int w4a16_seq_reserve(w4a16_page_allocator* a, int32_t* row, int max_blocks, int len) {
  W4_CHECK_ARG(a && row, "seq_reserve: null argument");
  W4_CHECK_ARG(max_blocks >= 1 && len >= 0, "seq_reserve: max_blocks=%d len=%d", max_blocks, len);
  const int need = (len + 15) / 16;
  W4_CHECK_SHAPE(need <= max_blocks, "seq_reserve: %d tokens need %d pages > max_blocks %d", len, need, max_blocks);
  std::lock_guard<std::mutex> lk(a->mu);
  int missing = 0;
  for (int i = 0; i < need; ++i) missing += row[i] < 0;
  std::vector<int32_t> got(missing);
  const int rc = alloc_locked(a, missing, got.data());
  if (rc) return rc;
  int k = 0;
  for (int i = 0; i < need; ++i)
    if (row[i] < 0) row[i] = got[k++];
  return W4A16_OK;
}

extern "C" int w4a16_seq_release(w4a16_page_allocator* a, int32_t* row, int max_blocks) {
  W4_CHECK_ARG(a && row, "seq_release: null argument");
  W4_CHECK_ARG(max_blocks >= 1, "seq_release: max_blocks=%d", max_blocks);
  std::lock_guard<std::mutex> lk(a->mu);
  std::vector<int32_t> pages;
  for (int i = 0; i < max_blocks; ++i)
    if (row[i] >= 0) pages.push_back(row[i]);
  const int rc = free_locked(a, pages.data(), (int)pages.size());
  if (rc) return rc;
  for (int i = 0; i < max_blocks; ++i) row[i] = -1;
  return W4A16_OK;
}

// ---------------------------------------------------------------------------
// Continuous batching
// ---------------------------------------------------------------------------
namespace {
struct BatchSeq {
  std::vector<int32_t> prompt;
  int max_new = 0;
  std::vector<int32_t> out;      // generated tokens
  std::vector<int32_t> row;      // block-table row (host), -1 = no page
  int len = 0;                   // tokens in the KV cache
  int fed = 0;                   // prompt tokens fed so far
  bool done = false;
  int restarts = 0;
};
}  // namespace

struct w4a16_batcher {
  w4a16_model* model = nullptr;
  w4a16_page_allocator* alloc = nullptr;
  int max_batch = 0, max_blocks = 0, max_context = 0;
  std::map<int, BatchSeq> seqs;
  std::deque<int> waiting;       // sequence ids, front first
  std::vector<int> active;       // admitted sequence ids, in admission order
  int next_id = 0;
  long steps = 0, preemptions = 0;
  int32_t *h_tok = nullptr, *h_out = nullptr, *h_bt = nullptr, *h_lens = nullptr;  // pinned
  int32_t *d_tok = nullptr, *d_out = nullptr, *d_bt = nullptr, *d_lens = nullptr;
  std::mutex mu;
};

extern "C" int w4a16_batcher_create(w4a16_model* model, int num_pages, int max_batch, int max_blocks,
                                    int max_context, w4a16_batcher** out) {
  W4_CHECK_ARG(model && out, "batcher_create: null argument");
  *out = nullptr;
  W4_CHECK_ARG(num_pages >= 1 && max_batch >= 1 && max_blocks >= 1 && max_context >= 1,
               "batcher_create: bad sizes");
  W4_CHECK_SHAPE(max_context <= max_blocks * 16, "batcher_create: max_context %d > max_blocks*16", max_context);
  auto* b = new w4a16_batcher();
  int rc = w4a16_page_allocator_create(num_pages, &b->alloc);
  if (rc) {
    delete b;
    return rc;
  }
  b->model = model;
  b->max_batch = max_batch;
  b->max_blocks = max_blocks;
  b->max_context = max_context;
  const size_t nt = (size_t)max_batch * 4, nbt = (size_t)max_batch * max_blocks * 4;
  cudaError_t e = cudaHostAlloc(&b->h_tok, nt, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(&b->h_out, nt, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(&b->h_lens, nt, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(&b->h_bt, nbt, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaMalloc(&b->d_tok, nt);
  if (e == cudaSuccess) e = cudaMalloc(&b->d_out, nt);
  if (e == cudaSuccess) e = cudaMalloc(&b->d_lens, nt);
  if (e == cudaSuccess) e = cudaMalloc(&b->d_bt, nbt);
  if (e != cudaSuccess) {
    w4a16_batcher_destroy(b);
    return w4::set_error(W4A16_ERR_CUDA, "batcher_create: %s", cudaGetErrorString(e));
  }
  *out = b;
  return W4A16_OK;
}

extern "C" void w4a16_batcher_destroy(w4a16_batcher* b) {
  if (!b) return;
  if (b->h_tok) cudaFreeHost(b->h_tok);
  if (b->h_out) cudaFreeHost(b->h_out);
  if (b->h_lens) cudaFreeHost(b->h_lens);
  if (b->h_bt) cudaFreeHost(b->h_bt);
  if (b->d_tok) cudaFree(b->d_tok);
  if (b->d_out) cudaFree(b->d_out);
  if (b->d_lens) cudaFree(b->d_lens);
  if (b->d_bt) cudaFree(b->d_bt);
  w4a16_page_allocator_destroy(b->alloc);
  delete b;
}

extern "C" int w4a16_batcher_submit(w4a16_batcher* b, const int32_t* prompt, int prompt_len, int max_new_tokens,
                                    int* seq_id) {
  W4_CHECK_ARG(b && prompt && seq_id, "batcher_submit: null argument");
  W4_CHECK_ARG(prompt_len >= 1 && max_new_tokens >= 1, "batcher_submit: prompt_len=%d max_new_tokens=%d",
               prompt_len, max_new_tokens);
  // the last generated token is never fed back, so the cache holds at most
  // prompt_len + max_new_tokens - 1 tokens
  W4_CHECK_SHAPE(prompt_len + max_new_tokens - 1 <= b->max_context,
                 "batcher_submit: %d + %d tokens exceed max_context %d", prompt_len, max_new_tokens, b->max_context);
  // alone in the pool a sequence always fits, so the oldest one always progresses
  const int need = (prompt_len + max_new_tokens - 1 + 15) / 16;
  if (need > b->alloc->num_pages)
    return w4::set_error(W4A16_ERR_NO_PAGES, "batcher_submit: the sequence needs %d pages, the pool has %d", need,
                         b->alloc->num_pages);
  std::lock_guard<std::mutex> lk(b->mu);
  BatchSeq s;
  s.prompt.assign(prompt, prompt + prompt_len);
  s.max_new = max_new_tokens;
  s.row.assign(b->max_blocks, -1);
  const int id = b->next_id++;
  b->seqs.emplace(id, std::move(s));
  b->waiting.push_back(id);
  *seq_id = id;
  return W4A16_OK;
}

// free a sequence's pages and send it back to the front of the queue
static void preempt(w4a16_batcher* b, int id) {
  BatchSeq& s = b->seqs.at(id);
  w4a16_seq_release(b->alloc, s.row.data(), b->max_blocks);
  s.len = 0;
  s.fed = 0;
  s.out.clear();
  ++s.restarts;
  ++b->preemptions;
  b->active.erase(std::find(b->active.begin(), b->active.end(), id));
  b->waiting.push_front(id);
}

extern "C" int w4a16_batcher_step(w4a16_batcher* b, w4a16_stream_t stream, int* n_active) {
  W4_CHECK_ARG(b, "batcher_step: null batcher");
  std::lock_guard<std::mutex> lk(b->mu);
  // admit waiting sequences while there are slots and a page for their first token
  while (!b->waiting.empty() && (int)b->active.size() < b->max_batch) {
    const int id = b->waiting.front();
    if (w4a16_seq_reserve(b->alloc, b->seqs.at(id).row.data(), b->max_blocks, 1) != W4A16_OK) break;
    b->waiting.pop_front();
    b->active.push_back(id);
  }
  // the page of each active sequence's next position; if the pool is empty,
  // preempt the most recently admitted sequence and try again
  for (size_t i = 0; i < b->active.size();) {
    BatchSeq& s = b->seqs.at(b->active[i]);
    if (w4a16_seq_reserve(b->alloc, s.row.data(), b->max_blocks, s.len + 1) == W4A16_OK) {
      ++i;
      continue;
    }
    preempt(b, b->active.back());  // retry sequence i with the victim's pages (or stop: it was the victim)
  }
  const int B = (int)b->active.size();
  if (n_active) *n_active = B;
  if (B == 0) return W4A16_OK;
  for (int r = 0; r < B; ++r) {
    const BatchSeq& s = b->seqs.at(b->active[r]);
    b->h_tok[r] = s.fed < (int)s.prompt.size() ? s.prompt[s.fed] : s.out.back();
    b->h_lens[r] = s.len;  // decode_step adds this step's token on the device
    std::copy(s.row.begin(), s.row.end(), b->h_bt + (size_t)r * b->max_blocks);
  }
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(b->d_tok, b->h_tok, (size_t)B * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(b->d_lens, b->h_lens, (size_t)B * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b->d_bt, b->h_bt, (size_t)B * b->max_blocks * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return w4::set_error(W4A16_ERR_CUDA, "batcher_step: upload: %s", cudaGetErrorString(e));
  // one graph per batch size: the device buffers stay the same, B picks the bucket
  int rc = decode_step(b->model, b->d_tok, b->d_out, b->d_bt, b->max_blocks, b->d_lens, B, nullptr, 1, stream);
  if (rc) return rc;
  e = cudaMemcpyAsync(b->h_out, b->d_out, (size_t)B * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return w4::set_error(W4A16_ERR_CUDA, "batcher_step: %s", cudaGetErrorString(e));
  ++b->steps;
  // advance every sequence; finished ones give their pages back
  std::vector<int> still;
  for (int r = 0; r < B; ++r) {
    const int id = b->active[r];
    BatchSeq& s = b->seqs.at(id);
    s.len += 1;
    const bool prompt_token = s.fed < (int)s.prompt.size();
    if (prompt_token) ++s.fed;
    if (!prompt_token || s.fed == (int)s.prompt.size()) s.out.push_back(b->h_out[r]);
    if ((int)s.out.size() >= s.max_new) {
      s.done = true;
      w4a16_seq_release(b->alloc, s.row.data(), b->max_blocks);
    } else {
      still.push_back(id);
    }
  }
  b->active.swap(still);
  return W4A16_OK;
}

extern "C" int w4a16_batcher_poll(w4a16_batcher* b, int seq_id, int32_t* tokens, int cap, int* n_tokens, int* done) {
  W4_CHECK_ARG(b && n_tokens && done, "batcher_poll: null argument");
  std::lock_guard<std::mutex> lk(b->mu);
  auto it = b->seqs.find(seq_id);
  W4_CHECK_ARG(it != b->seqs.end(), "batcher_poll: unknown sequence %d", seq_id);
  const BatchSeq& s = it->second;
  const int n = std::min(cap, (int)s.out.size());
  if (tokens) std::copy(s.out.begin(), s.out.begin() + std::max(0, n), tokens);
  *n_tokens = (int)s.out.size();
  *done = s.done ? 1 : 0;
  return W4A16_OK;
}

extern "C" int w4a16_batcher_stats(w4a16_batcher* b, long* steps, long* preemptions, int* waiting, int* active,
                                   int* free_pages) {
  W4_CHECK_ARG(b, "batcher_stats: null batcher");
  std::lock_guard<std::mutex> lk(b->mu);
  if (steps) *steps = b->steps;
  if (preemptions) *preemptions = b->preemptions;
  if (waiting) *waiting = (int)b->waiting.size();
  if (active) *active = (int)b->active.size();
  if (free_pages) *free_pages = w4a16_page_free_count(b->alloc);
  return W4A16_OK;
}
