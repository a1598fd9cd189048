// Stall-free batching (Algorithm 3 of "Taming Throughput-Latency Tradeoff in
// LLM Inference with Sarathi-Serve", section 2 Q2 item 2 and the section 3
// flowchart) with a paged KV allocator.  Pure host code.
//
// Every iteration: all running decodes first (decodes never stall), then the
// next chunk of the prompt currently in prefill, sized by the remaining token
// budget, then the flowchart's admission loop: waiting requests, first come
// first served, each with its first chunk, while the head of the queue can be
// allocated, the budget lasts and the batch is under `max_chunks` chunks
// (max_chunks = 1: a new request only when no prompt is in prefill).  A
// chunk that stops short of its prompt's end fills the budget, so at most one
// prompt is unfinished at any time.  The budget is rounded down to a whole
// number of GEMM row tiles (the same digest, section 2 Q2 item 3).  Pages are
// handed out lowest id first: a prompt's pages at admission, a decode's page
// when its slot starts a new page; they return when the request finishes.
#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

#include "internal.h"

namespace {

struct Req {
  int32_t id = 0;
  double arrival = 0.0;
  int32_t prompt_len = 0, output_len = 0;
  bool has_tokens = false;
  std::vector<int32_t> prompt;
  int32_t prefill_done = 0, generated = 0;
  std::vector<int32_t> pages;
  int32_t last_token = 0;
};

struct Chunk {
  Req* r;
  int32_t start, len;
};

}  // namespace

struct sar_sched {
  sar_sched_cfg cfg{};
  int32_t tau = 0;
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_pages;
  std::vector<Req*> waiting;   // insertion order
  std::vector<Req*> running;   // admission order
  int32_t n_finished = 0;
  // the last batch
  std::vector<Chunk> chunks;
  std::vector<Req*> decodes;
  bool pending = false;
  // storage behind the returned sar_batch
  std::vector<sar_prefill> out_pre;
  std::vector<sar_decode> out_dec;
  std::vector<int32_t> out_bt;
  std::vector<int32_t> out_tokens;

  ~sar_sched() {
    for (Req* r : waiting) delete r;
    for (Req* r : running) delete r;
  }
};

extern "C" {

int sar_sched_create(const sar_sched_cfg* cfg, sar_sched** out) {
  using sar::set_error;
  if (!cfg || !out) return set_error(SAR_ERR_INVALID_ARG, "sched: null argument");
  if (cfg->tile <= 0 || cfg->tau < cfg->tile)
    return set_error(SAR_ERR_INVALID_ARG, "sched: token budget smaller than one tile");
  if (cfg->page_size <= 0 || cfg->num_pages < 0 || cfg->max_batch <= 0 || cfg->max_chunks < 0)
    return set_error(SAR_ERR_INVALID_ARG, "sched: bad page size, page count, batch or chunk cap");
  sar_sched* s = new sar_sched();
  s->cfg = *cfg;
  s->tau = (cfg->tau / cfg->tile) * cfg->tile;
  for (int32_t p = 0; p < cfg->num_pages; ++p) s->free_pages.push(p);
  *out = s;
  return SAR_OK;
}

int sar_sched_destroy(sar_sched* s) {
  delete s;
  return SAR_OK;
}

int sar_sched_add(sar_sched* s, int32_t req, double arrival, int32_t prompt_len, int32_t output_len,
                  const int32_t* prompt_tokens) {
  using sar::set_error;
  if (!s) return set_error(SAR_ERR_INVALID_ARG, "sched: null scheduler");
  if (prompt_len <= 0 || output_len <= 0) return set_error(SAR_ERR_INVALID_ARG, "sched: empty prompt or output");
  Req* r = new Req();
  r->id = req;
  r->arrival = arrival;
  r->prompt_len = prompt_len;
  r->output_len = output_len;
  if (prompt_tokens) {
    r->has_tokens = true;
    r->prompt.assign(prompt_tokens, prompt_tokens + prompt_len);
  }
  s->waiting.push_back(r);
  return SAR_OK;
}

int sar_sched_next(sar_sched* s, double now, sar_batch* out, const int32_t** tokens_out) {
  using sar::set_error;
  if (!s || !out) return set_error(SAR_ERR_INVALID_ARG, "sched: null argument");
  const int32_t ps = s->cfg.page_size;
  int32_t n_t = 0;
  s->decodes.clear();
  s->chunks.clear();
  // 1. one decode token for every running request whose prompt is done
  for (Req* r : s->running) {
    if (r->prefill_done == r->prompt_len && r->generated < r->output_len) {
      const int32_t ctx = r->prompt_len + r->generated - 1;
      if (ctx % ps == 0) {
        if (s->free_pages.empty()) return set_error(SAR_ERR_NO_PAGES, "sched: KV page pool exhausted");
        r->pages.push_back(s->free_pages.top());
        s->free_pages.pop();
      }
      s->decodes.push_back(r);
      ++n_t;
    }
  }
  // 2. the next chunk of the prompt in prefill, if any
  Req* ongoing = nullptr;
  for (Req* r : s->running)
    if (r->prefill_done < r->prompt_len) {
      ongoing = r;
      break;
    }
  if (ongoing) {
    const int32_t c = std::min(ongoing->prompt_len - ongoing->prefill_done, s->tau - n_t);
    if (c > 0) {
      s->chunks.push_back({ongoing, ongoing->prefill_done, c});
      n_t += c;
    }
  }
  // 3. admit waiting requests first come first served while the head fits
  if (!ongoing || s->cfg.max_chunks != 1) {
    std::vector<Req*> ready;
    for (Req* r : s->waiting)
      if (r->arrival <= now) ready.push_back(r);
    std::stable_sort(ready.begin(), ready.end(), [](const Req* a, const Req* b) {
      return a->arrival < b->arrival || (a->arrival == b->arrival && a->id < b->id);
    });
    for (Req* r : ready) {
      if (s->cfg.max_chunks > 0 && (int32_t)s->chunks.size() >= s->cfg.max_chunks) break;
      const int32_t need = (r->prompt_len + ps - 1) / ps;
      if (!(n_t < s->tau && (int64_t)s->free_pages.size() >= (int64_t)need + 1 &&
            (int32_t)s->running.size() < s->cfg.max_batch))
        break;
      s->waiting.erase(std::find(s->waiting.begin(), s->waiting.end(), r));
      for (int32_t i = 0; i < need; ++i) {
        r->pages.push_back(s->free_pages.top());
        s->free_pages.pop();
      }
      s->running.push_back(r);
      const int32_t c = std::min(r->prompt_len, s->tau - n_t);
      s->chunks.push_back({r, 0, c});
      n_t += c;
    }
  }
  // descriptor in scheduler-owned storage (block tables copied)
  size_t bt_total = 0;
  for (const Chunk& c : s->chunks) bt_total += c.r->pages.size();
  for (Req* r : s->decodes) bt_total += r->pages.size();
  s->out_bt.resize(bt_total);
  s->out_pre.resize(s->chunks.size());
  s->out_dec.resize(s->decodes.size());
  size_t off = 0;
  *out = sar_batch{};
  out->in_kind = SAR_IN_TOKENS;
  for (size_t i = 0; i < s->chunks.size(); ++i) {
    const Chunk& c = s->chunks[i];
    std::copy(c.r->pages.begin(), c.r->pages.end(), s->out_bt.begin() + off);
    s->out_pre[i] = sar_prefill{c.r->id, c.start, c.len, s->out_bt.data() + off, (int32_t)c.r->pages.size()};
    off += c.r->pages.size();
  }
  if (!s->chunks.empty()) {
    out->has_prefill = 1;
    out->prefill = s->out_pre[0];
    out->n_more_prefill = (int32_t)s->chunks.size() - 1;
    out->more_prefill = s->chunks.size() > 1 ? s->out_pre.data() + 1 : nullptr;
  }
  for (size_t i = 0; i < s->decodes.size(); ++i) {
    Req* r = s->decodes[i];
    std::copy(r->pages.begin(), r->pages.end(), s->out_bt.begin() + off);
    s->out_dec[i].req = r->id;
    s->out_dec[i].ctx_len = r->prompt_len + r->generated - 1;
    s->out_dec[i].block_table = s->out_bt.data() + off;
    s->out_dec[i].n_blocks = (int32_t)r->pages.size();
    off += r->pages.size();
  }
  out->n_decode = (int32_t)s->decodes.size();
  out->decode = s->out_dec.data();
  // input ids when every running request brought its prompt tokens
  bool known = true;
  for (Req* r : s->running) known = known && r->has_tokens;
  s->out_tokens.clear();
  if (known) {
    for (const Chunk& c : s->chunks)
      s->out_tokens.insert(s->out_tokens.end(), c.r->prompt.begin() + c.start, c.r->prompt.begin() + c.start + c.len);
    for (Req* r : s->decodes) s->out_tokens.push_back(r->last_token);
  }
  if (tokens_out) *tokens_out = known ? s->out_tokens.data() : nullptr;
  s->pending = true;
  return SAR_OK;
}

int sar_sched_commit(sar_sched* s, const int32_t* sampled, int32_t n_sampled, int32_t* n_finished) {
  using sar::set_error;
  if (!s) return set_error(SAR_ERR_INVALID_ARG, "sched: null scheduler");
  if (!s->pending) return set_error(SAR_ERR_INVALID_ARG, "sched: commit without a batch");
  const int32_t rows = (int32_t)(s->chunks.size() + s->decodes.size());
  if (n_sampled != rows || (rows > 0 && !sampled))
    return set_error(SAR_ERR_INVALID_ARG, "sched: one sampled token per logits row expected");
  int32_t i = 0;
  for (const Chunk& c : s->chunks) {
    c.r->prefill_done += c.len;
    if (c.r->prefill_done == c.r->prompt_len) {
      c.r->generated = 1;
      c.r->last_token = sampled[i];
    }
    ++i;
  }
  for (Req* r : s->decodes) {
    r->generated += 1;
    r->last_token = sampled[i++];
  }
  int32_t done = 0;
  std::vector<Req*> keep;
  for (Req* r : s->running) {
    if (r->generated >= r->output_len) {
      for (int32_t p : r->pages) s->free_pages.push(p);
      delete r;
      ++done;
    } else {
      keep.push_back(r);
    }
  }
  s->running.swap(keep);
  s->n_finished += done;
  s->chunks.clear();
  s->decodes.clear();
  s->pending = false;
  if (n_finished) *n_finished = done;
  return SAR_OK;
}

int sar_sched_stats(const sar_sched* s, int32_t* waiting, int32_t* running, int32_t* finished,
                    int32_t* free_pages) {
  if (!s) return sar::set_error(SAR_ERR_INVALID_ARG, "sched: null scheduler");
  if (waiting) *waiting = (int32_t)s->waiting.size();
  if (running) *running = (int32_t)s->running.size();
  if (finished) *finished = s->n_finished;
  if (free_pages) *free_pages = (int32_t)s->free_pages.size();
  return SAR_OK;
}

}  // extern "C"
