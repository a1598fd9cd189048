// Stall-free batching (Algorithm 3 of "Taming Throughput-Latency Tradeoff in
// LLM Inference with Sarathi-Serve", section 2 Q2 item 2 and the section 3
// flowchart) with a paged KV allocator.  Pure host code.
//
// Every iteration: all running decodes first (decodes never stall), then at
// most one chunk of the prompt currently in prefill, sized by the remaining
// token budget; only when no prompt is in prefill is the next waiting request
// admitted (first come, first served).  The budget is rounded down to a whole
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

}  // namespace

struct sar_sched {
  sar_sched_cfg cfg{};
  int32_t tau = 0;
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_pages;
  std::vector<Req*> waiting;   // insertion order
  std::vector<Req*> running;   // admission order
  int32_t n_finished = 0;
  // the last batch
  Req* chunk_req = nullptr;
  int32_t chunk_start = 0, chunk_len = 0;
  std::vector<Req*> decodes;
  bool pending = false;
  // storage behind the returned sar_batch
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
  if (cfg->page_size <= 0 || cfg->num_pages < 0 || cfg->max_batch <= 0)
    return set_error(SAR_ERR_INVALID_ARG, "sched: bad page size, page count or batch cap");
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
  s->chunk_req = nullptr;
  s->chunk_len = 0;
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
  // 2. the ongoing prefill, if any, else 3. admit the next waiting request
  Req* ongoing = nullptr;
  for (Req* r : s->running)
    if (r->prefill_done < r->prompt_len) {
      ongoing = r;
      break;
    }
  if (ongoing) {
    const int32_t c = std::min(ongoing->prompt_len - ongoing->prefill_done, s->tau - n_t);
    if (c > 0) {
      s->chunk_req = ongoing;
      s->chunk_start = ongoing->prefill_done;
      s->chunk_len = c;
      n_t += c;
    }
  } else {
    Req* head = nullptr;
    for (Req* r : s->waiting)
      if (r->arrival <= now && (!head || r->arrival < head->arrival || (r->arrival == head->arrival && r->id < head->id)))
        head = r;
    if (head && n_t < s->tau) {
      const int32_t need = (head->prompt_len + ps - 1) / ps;
      if ((int64_t)s->free_pages.size() >= (int64_t)need + 1 && (int32_t)s->running.size() < s->cfg.max_batch) {
        s->waiting.erase(std::find(s->waiting.begin(), s->waiting.end(), head));
        for (int32_t i = 0; i < need; ++i) {
          head->pages.push_back(s->free_pages.top());
          s->free_pages.pop();
        }
        s->running.push_back(head);
        s->chunk_req = head;
        s->chunk_start = 0;
        s->chunk_len = std::min(head->prompt_len, s->tau - n_t);
        n_t += s->chunk_len;
      }
    }
  }
  // descriptor in scheduler-owned storage (block tables copied)
  size_t bt_total = s->chunk_req ? s->chunk_req->pages.size() : 0;
  for (Req* r : s->decodes) bt_total += r->pages.size();
  s->out_bt.resize(bt_total);
  s->out_dec.resize(s->decodes.size());
  size_t off = 0;
  *out = sar_batch{};
  out->in_kind = SAR_IN_TOKENS;
  if (s->chunk_req) {
    Req* r = s->chunk_req;
    std::copy(r->pages.begin(), r->pages.end(), s->out_bt.begin());
    out->has_prefill = 1;
    out->prefill.req = r->id;
    out->prefill.start_pos = s->chunk_start;
    out->prefill.len = s->chunk_len;
    out->prefill.block_table = s->out_bt.data();
    out->prefill.n_blocks = (int32_t)r->pages.size();
    off = r->pages.size();
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
    if (s->chunk_req)
      s->out_tokens.insert(s->out_tokens.end(), s->chunk_req->prompt.begin() + s->chunk_start,
                           s->chunk_req->prompt.begin() + s->chunk_start + s->chunk_len);
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
  const int32_t rows = (s->chunk_req ? 1 : 0) + (int32_t)s->decodes.size();
  if (n_sampled != rows || (rows > 0 && !sampled))
    return set_error(SAR_ERR_INVALID_ARG, "sched: one sampled token per logits row expected");
  int32_t i = 0;
  if (s->chunk_req) {
    Req* r = s->chunk_req;
    r->prefill_done += s->chunk_len;
    if (r->prefill_done == r->prompt_len) {
      r->generated = 1;
      r->last_token = sampled[0];
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
  s->chunk_req = nullptr;
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
