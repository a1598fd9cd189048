// Model, paged KV cache and the hybrid step: host orchestration of the kernels.
//
// One step ("SARATHI: Efficient LLM Inference by Piggybacking Decodes with
// Chunked Prefills", reading notes, part 2 section 3 -- merge, split, merge):
//   rows [0, Lp) are the prefill chunks, rows [Lp, Lp+Bd) the decodes, all in
//   one [M, H] residual buffer; per layer
//     RMSNorm -> QKV GEMM (all rows) -> rotary + KV-page append (all rows) ->
//     chunk attention on rows [0, Lp) | decode attention on rows [Lp, M),
//     both reading the pages and writing disjoint row ranges of one buffer ->
//     O GEMM + residual -> RMSNorm -> gate/up GEMM with SiLU*up epilogue ->
//     down GEMM + residual;
//   then the final norm on the rows whose next token is sampled and the LM head.
// The per-step metadata (positions, page slots, block tables, the decode
// work split) is planned on the host and shipped in one async copy.
#include <cuda.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

using sar::set_error;
using sar::cuda_error;

namespace {

constexpr int kMetaRing = 4;
constexpr int kSmallStepRows = 256;  // steps this small use the swap tiling (tokens on the MMA's N side)

using st16 = uint16_t;  // one element of the storage type (fp16 or bf16)
using WMaps = CUtensorMap[sar::kWeightBoxes];  // one weight matrix, every box height

struct LayerW {
  st16 *wqkv = nullptr, *wo = nullptr, *wgu = nullptr, *wd = nullptr;
  float *n1 = nullptr, *n2 = nullptr;
  WMaps m_qkv, m_o, m_gu, m_d;  // weight maps, box rows 32 / 64 / 128 / 256
  bool set = false;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct EventPair {
  cudaEvent_t a = nullptr, b = nullptr;
  int kind = 0;
};

}  // namespace

struct sar_model {
  sar_dims d{};
  int qkv_n = 0;        // (qh + 2 kvh) * head_dim
  int qd = 0, kvd = 0;  // q width, kv width
  uint8_t* arena = nullptr;
  std::vector<LayerW> L;
  st16 *embed = nullptr, *lm_head = nullptr;
  float* final_norm = nullptr;
  WMaps m_head;
  bool head_set = false;
  double* inv_freq = nullptr;
  // workspace
  uint8_t* ws = nullptr;
  st16 *xn = nullptr, *attn = nullptr, *act = nullptr, *hrows = nullptr;
  float2* rope_cs = nullptr;  // (cos, sin) of this step's positions, [head_dim / 4][max_tokens] float4 pairs
  float* hres = nullptr;   // residual stream, fp32
  float* qkv32 = nullptr;  // QKV projection in fp32, q and k rotated by the projection's epilogue
  float* gu32 = nullptr;   // small steps: gate/up projection accumulated split-K in fp32
  void* in_stage = nullptr;
  float* partials = nullptr;
  size_t partials_cap = 0;  // floats
  float* logits_stage = nullptr;
  size_t logits_stage_rows = 0;
  int* err = nullptr;
  // step metadata: pinned host ring + device buffer
  int32_t* meta_host[kMetaRing] = {};
  cudaEvent_t meta_ev[kMetaRing] = {};
  size_t meta_cap = 0;  // int32 elements per buffer
  int meta_slot = 0;
  int32_t* meta_dev = nullptr;
  size_t meta_dev_cap = 0;
  // two-stream attention split
  bool overlap = false;
  // key-range splits of chunk-attention tiles (changes the summation order)
  bool chunk_split = false;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaStream_t capture = nullptr;  // steps are captured into graphs here (never the legacy stream)
  // profiling (off while a step is being captured into a graph)
  bool prof = false;
  bool capturing = false;
  std::vector<EventPair> ev_used, ev_free;
  double prof_ms[SAR_K_COUNT] = {};
  int64_t prof_n[SAR_K_COUNT] = {};
};

struct sar_kv {
  const sar_model* m = nullptr;
  int page_size = 0, num_pages = 0;
  uint16_t *k = nullptr, *v = nullptr;
  size_t layer_elems = 0;
  std::vector<CUtensorMap> tmk, tmv;  // per layer: decode attention's view of the pages
};

namespace {

int check(cudaError_t e, const char* what) { return cuda_error(e, what); }

// The device error record [code, site, detail, 0] of the single-kernel entry
// points on the current device, allocated (and zeroed) at its first use there.
std::mutex g_op_flags_mu;
std::map<int, int*> g_op_flags;
int op_flags(int** out) {
  int dev = 0;
  SAR_TRY(check(cudaGetDevice(&dev), "op flags: current device"));
  std::lock_guard<std::mutex> lk(g_op_flags_mu);
  int*& f = g_op_flags[dev];
  if (!f) {
    int* p = nullptr;
    SAR_TRY(check(cudaMalloc(&p, 16), "op flags: allocate"));
    const int rc = check(cudaMemset(p, 0, 16), "op flags: clear");
    if (rc != SAR_OK) {
      cudaFree(p);
      return rc;
    }
    f = p;
  }
  *out = f;
  return SAR_OK;
}

// ---- profiling helpers -----------------------------------------------------
EventPair* prof_begin(sar_model* m, int kind, cudaStream_t s) {
  if (!m->prof || m->capturing) return nullptr;
  EventPair ep;
  if (!m->ev_free.empty()) {
    ep = m->ev_free.back();
    m->ev_free.pop_back();
  } else {
    cudaEventCreate(&ep.a);
    cudaEventCreate(&ep.b);
  }
  ep.kind = kind;
  cudaEventRecord(ep.a, s);
  m->ev_used.push_back(ep);
  return &m->ev_used.back();
}
void prof_end(sar_model* m, cudaStream_t s) {
  if (!m->prof || m->capturing || m->ev_used.empty()) return;
  cudaEventRecord(m->ev_used.back().b, s);
}

struct Prof {
  sar_model* m;
  cudaStream_t s;
  Prof(sar_model* m_, int kind, cudaStream_t s_) : m(m_), s(s_) { prof_begin(m, kind, s); }
  ~Prof() { prof_end(m, s); }
};

int weight_maps(WMaps& maps, const void* w, int rows, int cols, int storage) {
  for (int i = 0; i < sar::kWeightBoxes; ++i) SAR_TRY(sar::make_tmap_16(&maps[i], w, rows, cols, 32u << i, storage));
  return SAR_OK;
}

// GEMM over `rows` activation rows with the weight maps of one matrix.
int run_gemm(sar_model* m, const st16* a, int rows, const WMaps& wmaps, int N, int K, int epi,
             void* c, const void* r, cudaStream_t s, const sar::RopeEpi* rope = nullptr,
             int variant = SAR_GEMM_AUTO) {
  sar::GemmCfg cfg;
  SAR_TRY(sar::gemm_config(rows, N, K, epi, variant, &cfg, c == r));
  CUtensorMap amap;
  SAR_TRY(sar::make_tmap_16(&amap, a, rows, K, cfg.swap ? cfg.b_box_rows : cfg.a_box_rows, m->d.storage));
  const CUtensorMap& wm = wmaps[sar::weight_box_index(cfg)];
  return sar::gemm_launch(cfg, amap, wm, rows, N, K, epi, m->d.storage, c, r, m->err, s, rope);
}

// ---- step planning -----------------------------------------------------------
struct Plan {
  int M = 0, Lp = 0, Bd = 0, R = 0;
  // offsets into the metadata block (int32 elements)
  size_t o_pos = 0, o_slot = 0, o_pbt = 0, o_nkeys = 0, o_btoff = 0, o_btlen = 0, o_pbeg = 0, o_pcnt = 0,
         o_items = 0, o_bt = 0, o_rows = 0, o_tiles = 0, o_comb = 0, total = 0;
  int n_items = 0, n_parts = 0, n_tiles = 0, n_comb = 0, n_cparts = 0;
  int chunk_dual = 0;  // the chunk tile table lists tile pairs (the two-tile kernel)
};

// The batch's prefill chunks in row order: `prefill` (if has_prefill), then more_prefill[].
std::vector<sar_prefill> batch_chunks(const sar_batch* b) {
  std::vector<sar_prefill> c;
  if (b->has_prefill) c.push_back(b->prefill);
  for (int i = 0; i < b->n_more_prefill; ++i) c.push_back(b->more_prefill[i]);
  return c;
}

// What the planner needs to know about the model, the cache and the device.
struct PlanEnv {
  sar_dims d;
  int page_size = 0, num_pages = 0, sms = 0;
  bool has_embed = false;
  bool chunk_split = false;
};

PlanEnv plan_env(const sar_model* m, const sar_kv* kv) {
  PlanEnv e;
  e.d = m->d;
  e.page_size = kv->page_size;
  e.num_pages = kv->num_pages;
  e.sms = sar::num_sms();
  e.has_embed = m->embed != nullptr;
  e.chunk_split = m->chunk_split;
  return e;
}

// Query rows per CTA of the chunk-attention kernel the step will launch.
int chunk_tile_rows(const sar_dims& d, int page_size) {
  sar::ChunkAttnArgs probe{};
  probe.d = d.head_dim;
  probe.page_size = page_size;
  probe.qh = d.n_q_heads;
  probe.kvh = d.n_kv_heads;
  probe.window = d.sliding_window;
  return sar::chunk_attention_tc_supported(probe) ? sar::kChunkTileRowsTc : sar::kChunkTileRows;
}

int validate_and_plan(const PlanEnv& env, const sar_batch* b, Plan* p, std::vector<int32_t>* meta) {
  const sar_dims& d = env.d;
  if (b->n_decode < 0 || (b->n_decode > 0 && !b->decode)) return set_error(SAR_ERR_INVALID_ARG, "step: bad decode list");
  if (b->n_more_prefill < 0 || (b->n_more_prefill > 0 && !b->more_prefill))
    return set_error(SAR_ERR_INVALID_ARG, "step: bad chunk list");
  const std::vector<sar_prefill> chunks = batch_chunks(b);
  int64_t lp64 = 0;
  for (const sar_prefill& c : chunks) {
    if (c.len <= 0 || c.start_pos < 0 || !c.block_table) return set_error(SAR_ERR_INVALID_ARG, "step: bad prefill chunk");
    lp64 += c.len;
  }
  if (lp64 > d.max_tokens) return set_error(SAR_ERR_INVALID_ARG, "step: Lp + Bd exceeds max_tokens");
  const int Lp = (int)lp64;
  const int Bd = b->n_decode;
  const int M = Lp + Bd;
  if (M == 0) return set_error(SAR_ERR_INVALID_ARG, "step: empty batch");
  if (M > d.max_tokens) return set_error(SAR_ERR_INVALID_ARG, "step: Lp + Bd exceeds max_tokens");
  if (Bd > d.max_decodes) return set_error(SAR_ERR_INVALID_ARG, "step: Bd exceeds max_decodes");
  if (b->in_kind != SAR_IN_HIDDEN && b->in_kind != SAR_IN_TOKENS) return set_error(SAR_ERR_INVALID_ARG, "step: bad in_kind");
  if (b->in_kind == SAR_IN_TOKENS && (d.vocab == 0 || !env.has_embed))
    return set_error(SAR_ERR_INVALID_ARG, "step: token input without an embedding");
  const int ps = env.page_size;
  // a position's page and offset: shifts and masks for the usual power-of-two
  // page sizes (the planner runs on the host before every step, and an integer
  // division per row was most of its time)
  const int ps_shift = (ps & (ps - 1)) == 0 ? __builtin_ctz((unsigned)ps) : -1;
  auto page_of_pos = [&](int pos) { return ps_shift >= 0 ? pos >> ps_shift : pos / ps; };
  auto off_of_pos = [&](int pos) { return ps_shift >= 0 ? pos & (ps - 1) : pos % ps; };
  auto check_bt = [&](const int32_t* bt, int nb, int last_pos) -> int {
    if (nb < 0 || (int64_t)nb * ps <= last_pos) return set_error(SAR_ERR_INVALID_ARG, "step: block table does not cover the positions");
    const int need = page_of_pos(last_pos) + 1;
    for (int i = 0; i < need; ++i)
      if (bt[i] < 0 || bt[i] >= env.num_pages) return set_error(SAR_ERR_BOUNDS, "step: page id out of range");
    return SAR_OK;
  };
  for (const sar_prefill& c : chunks) SAR_TRY(check_bt(c.block_table, c.n_blocks, c.start_pos + c.len - 1));
  // a decode with nk keys reads from the 16-key block holding its oldest
  // visible key (the kernel masks the keys of that block before it)
  auto first_key = [&](int nk) { return d.sliding_window > 0 ? std::max(0, nk - d.sliding_window) / 16 * 16 : 0; };
  // the work split is sized from the keys a decode's pages can hold (at most
  // the window's span), not from its exact count, so that the plan's shape --
  // item and partial counts -- stays the same while a decode's context grows
  // within its pages (a captured step graph can then be re-pointed at the
  // next step); a decode's last range may be short or empty
  auto span_of = [&](int ctx) {
    const int cap = (page_of_pos(ctx) + 1) * ps;
    return d.sliding_window > 0 ? std::min(cap, d.sliding_window + 15) : cap;
  };
  int64_t total_keys = 0;
  for (int i = 0; i < Bd; ++i) {
    const sar_decode& dc = b->decode[i];
    if (dc.ctx_len < 0 || !dc.block_table) return set_error(SAR_ERR_INVALID_ARG, "step: bad decode entry");
    // (the page ids themselves are range-checked as they are copied below)
    if (dc.n_blocks < 0 || (int64_t)dc.n_blocks * ps <= dc.ctx_len)
      return set_error(SAR_ERR_INVALID_ARG, "step: block table does not cover the positions");
    total_keys += span_of(dc.ctx_len);
  }
  // decode work split: key ranges of `split` keys, a resident slot's share of
  // the whole launch (two CTAs resident per SM), up to 4096 keys -- with each
  // decode's ranges rounded up, about 2-4 CTAs per SM; fewer, longer ranges
  // measured faster than more, shorter ones (less set-up and merging per key):
  // on the tau = 512 step 93.6 us at a slot's share against 97.4 at half of
  // it, 104 at two thirds or a third, 111 at a quarter
  const int sms = env.sms;
  int64_t split = (total_keys * d.n_kv_heads) / (2LL * sms);
  split = std::max<int64_t>(128, std::min<int64_t>(4096, (split + 15) / 16 * 16));
  const int split32 = (int)split;
  // scratch arrays kept per thread, so a step's planning allocates nothing
  // once they have grown to the batch's size
  thread_local std::vector<int32_t> items, pbeg, pcnt, nkeys, btoff, btlen, bt, tail_items, rows, pbt, tiles, comb;
  thread_local std::vector<uint64_t> order;
  items.clear();
  bt.clear();
  tail_items.clear();
  rows.clear();
  pbt.clear();
  tiles.clear();
  comb.clear();
  pbeg.assign(Bd, -1);
  pcnt.assign(Bd, 0);
  nkeys.resize(Bd);
  btoff.resize(Bd);
  btlen.resize(Bd);
  int n_parts = 0;
  for (int i = 0; i < Bd; ++i) {
    const sar_decode& dc = b->decode[i];
    const int nk = dc.ctx_len + 1;
    nkeys[i] = nk;
    btoff[i] = (int32_t)bt.size();
    const int nb = page_of_pos(dc.ctx_len) + 1;
    btlen[i] = nb;
    {
      // copy the pages the positions use, checking each id on the way
      const size_t o0 = bt.size();
      bt.resize(o0 + nb);
      int32_t* dst = bt.data() + o0;
      const int32_t* src = dc.block_table;
      uint32_t bad = 0;
      for (int k = 0; k < nb; ++k) {
        const int32_t v = src[k];
        dst[k] = v;
        bad |= (uint32_t)v >= (uint32_t)env.num_pages ? 1u : 0u;
      }
      if (bad) return set_error(SAR_ERR_BOUNDS, "step: page id out of range");
    }
    const int kfirst = first_key(nk);
    const int span = span_of(dc.ctx_len);
    const int ns = (span + split32 - 1) / split32;
    // equal ranges (16-key multiples) rather than full ranges plus a remainder
    const int len = ((span + ns - 1) / ns + 15) / 16 * 16;
    pcnt[i] = ns;
    if (ns > 1) {
      pbeg[i] = n_parts;
    }
    for (int sidx = 0; sidx < ns; ++sidx) {
      const int k0 = kfirst + sidx * len;
      const int k1 = std::max(k0, std::min(nk, k0 + len));
      const int part = ns > 1 ? n_parts + sidx : -1;
      tail_items.insert(tail_items.end(), {i, k0, k1, part});
    }
    if (ns > 1) n_parts += ns;
  }
  // longest ranges first, so the grid's last CTAs are its shortest (equal
  // lengths in planning order: one sort of (length, index) keys)
  {
    const size_t n_items = tail_items.size() / 4;
    order.resize(n_items);
    for (size_t t = 0; t < n_items; ++t) {
      const uint32_t len = (uint32_t)(tail_items[4 * t + 2] - tail_items[4 * t + 1]);
      order[t] = ((uint64_t)(0xFFFFFFFFu - len) << 32) | (uint64_t)t;
    }
    std::sort(order.begin(), order.end());
    items.resize(4 * n_items);
    for (size_t t = 0; t < n_items; ++t)
      std::memcpy(items.data() + 4 * t, tail_items.data() + 4 * (order[t] & 0xFFFFFFFFu), 16);
  }
  // rows whose logits are returned: every chunk's last row, then every decode row
  {
    int r0 = 0;
    for (const sar_prefill& c : chunks) {
      r0 += c.len;
      rows.push_back(r0 - 1);
    }
  }
  for (int i = 0; i < Bd; ++i) rows.push_back(Lp + i);
  // chunk block tables (each cut to the pages its positions use) and the
  // chunk-attention tiles: {first batch row, first position, rows, block-table
  // offset, block-table length, first and end 128-key block, partial slot},
  // the most keys first (the longest CTAs start first)
  const int tile_rows = chunk_tile_rows(d, ps);
  int n_cparts = 0;
  {
    struct Tile {
      std::array<int32_t, 8> e;
      int keys;
    };
    std::vector<Tile> tl;
    std::vector<std::pair<int, int>> chunk_tiles;  // (first entry of tl, count) per chunk
    int r0 = 0;
    for (const sar_prefill& c : chunks) {
      const int t_first = (int)tl.size();
      const int off = (int)pbt.size();
      const int nb = page_of_pos(c.start_pos + c.len - 1) + 1;
      pbt.insert(pbt.end(), c.block_table, c.block_table + nb);
      for (int q0 = 0; q0 < c.len; q0 += tile_rows) {
        const int rws = std::min(tile_rows, c.len - q0);
        const int pos0 = c.start_pos + q0;
        const int first = d.sliding_window > 0 ? std::max(0, pos0 - d.sliding_window + 1) : 0;
        const int kb0 = first / sar::kChunkTileRowsTc, kb1 = (pos0 + rws + sar::kChunkTileRowsTc - 1) / sar::kChunkTileRowsTc;
        tl.push_back({{r0 + q0, pos0, rws, off, nb, kb0, kb1, -1}, pos0 + rws - first});
      }
      chunk_tiles.push_back({t_first, (int)tl.size() - t_first});
      r0 += c.len;
    }
    // Key-range splits (tcgen05 kernel, one CTA per SM): when the tiles x
    // heads fill at most half the SMs, each tile's key blocks are shared out
    // over s = min(4, SMs / CTAs) CTAs (at least two blocks each) so that the
    // shares still run in one wave; a merge kernel combines them.  Past one
    // wave the shares' extra partial traffic and the merge cost more than the
    // shorter tail saves (Yi-34B, 112 CTAs in four shares: chunk attention
    // 13% slower; Mistral-7B, 64 CTAs in two: 33% faster).
    int s = 1;
    if (env.chunk_split && tile_rows == sar::kChunkTileRowsTc && !tl.empty()) {
      const long ctas = (long)tl.size() * d.n_q_heads, slots = std::max(1, sms);
      s = (int)std::min<long>(4, slots / ctas);
      if (s < 2) s = 1;
    }
    // Tile pairs (one CTA per pair of consecutive tiles of a chunk and head,
    // sharing their key blocks; a chunk's odd last tile pairs with an empty
    // one) when the one-tile grid needs more waves than the pair grid by a
    // margin: a pair takes ~1.9 times a tile's time per key block (one set of
    // softmax warps serves both tiles, and the softmax chain sets the pace of
    // either kernel), so pairs win where they save waves --
    // 4 tiles x 56 heads (224 CTAs on 152 SMs, two waves) run as 112 pairs in
    // one -- and not where one-tile CTAs fill their waves about as well.
    // Full causal attention and whole key ranges only.
    bool dual = false;
    p->chunk_dual = 0;
    if (s == 1 && d.sliding_window == 0 && tile_rows == sar::kChunkTileRowsTc && !tl.empty()) {
      long pairs = 0;
      for (const auto& ct : chunk_tiles) pairs += (ct.second + 1) / 2;
      const long slots = std::max(1, sms);
      const long w1 = ((long)tl.size() * d.n_q_heads + slots - 1) / slots;
      const long w2 = (pairs * d.n_q_heads + slots - 1) / slots;
      dual = 19 * w2 < 10 * w1;
    }
    std::vector<Tile> ent;
    if (dual) {
      struct Pair {
        Tile a, b;
        int keys;
      };
      std::vector<Pair> pr;
      for (const auto& ct : chunk_tiles)
        for (int i = 0; i < ct.second; i += 2) {
          const Tile& ta = tl[ct.first + i];
          Tile tb = ta;
          if (i + 1 < ct.second)
            tb = tl[ct.first + i + 1];
          else
            tb.e[2] = 0;  // no second tile: 0 rows over the first one's key blocks
          pr.push_back({ta, tb, std::max(ta.keys, tb.keys)});
        }
      std::stable_sort(pr.begin(), pr.end(), [](const Pair& x, const Pair& y) { return x.keys > y.keys; });
      for (const Pair& q : pr) {
        tiles.insert(tiles.end(), q.a.e.begin(), q.a.e.end());
        tiles.insert(tiles.end(), q.b.e.begin(), q.b.e.end());
      }
      p->chunk_dual = 1;
      tl.clear();  // nothing left for the one-tile table below
    }
    for (const Tile& t : tl) {
      const int nbk = t.e[6] - t.e[5];
      const int ss = std::min(s, nbk / 2);
      if (ss <= 1) {
        ent.push_back(t);
        continue;
      }
      comb.insert(comb.end(), {t.e[0], t.e[2], n_cparts, ss});
      for (int i = 0; i < ss; ++i) {
        Tile x = t;
        x.e[5] = t.e[5] + (int)((long)nbk * i / ss);
        x.e[6] = t.e[5] + (int)((long)nbk * (i + 1) / ss);
        x.e[7] = n_cparts + i;
        x.keys = (x.e[6] - x.e[5]) * sar::kChunkTileRowsTc;
        ent.push_back(x);
      }
      n_cparts += ss;
    }
    std::stable_sort(ent.begin(), ent.end(), [](const Tile& x, const Tile& y) { return x.keys > y.keys; });
    for (const Tile& t : ent) tiles.insert(tiles.end(), t.e.begin(), t.e.end());
  }

  p->M = M;
  p->Lp = Lp;
  p->Bd = Bd;
  p->R = (int)rows.size();
  p->n_items = (int)items.size() / 4;
  p->n_parts = n_parts;
  p->n_tiles = (int)tiles.size() / 8;
  p->n_comb = (int)comb.size() / 4;
  p->n_cparts = n_cparts;
  size_t o = 0;
  auto take = [&](size_t n) { size_t r = o; o += (n + 3) & ~size_t(3); return r; };  // 16-byte aligned pieces
  p->o_pos = take(M);
  p->o_slot = take(M);
  p->o_pbt = take(pbt.size());
  p->o_nkeys = take(Bd);
  p->o_btoff = take(Bd);
  p->o_btlen = take(Bd);
  p->o_pbeg = take(Bd);
  p->o_pcnt = take(Bd);
  p->o_items = take(items.size());
  p->o_bt = take(bt.size());
  p->o_rows = take(rows.size());
  p->o_tiles = take(tiles.size());
  p->o_comb = take(comb.size());
  p->total = o;
  meta->resize(o);  // every array is written below; the 16-byte padding between them is never read
  int32_t* mt = meta->data();
  {
    int r = 0;
    for (const sar_prefill& c : chunks) {
      int pg = page_of_pos(c.start_pos), off = off_of_pos(c.start_pos);
      for (int i = 0; i < c.len; ++i, ++r) {
        mt[p->o_pos + r] = c.start_pos + i;
        mt[p->o_slot + r] = c.block_table[pg] * ps + off;
        if (++off == ps) {
          off = 0;
          ++pg;
        }
      }
    }
  }
  for (int i = 0; i < Bd; ++i) {
    const int pos = b->decode[i].ctx_len;
    mt[p->o_pos + Lp + i] = pos;
    mt[p->o_slot + Lp + i] = b->decode[i].block_table[page_of_pos(pos)] * ps + off_of_pos(pos);
  }
  if (!pbt.empty()) std::memcpy(mt + p->o_pbt, pbt.data(), pbt.size() * 4);
  std::memcpy(mt + p->o_nkeys, nkeys.data(), Bd * 4);
  std::memcpy(mt + p->o_btoff, btoff.data(), Bd * 4);
  std::memcpy(mt + p->o_btlen, btlen.data(), Bd * 4);
  std::memcpy(mt + p->o_pbeg, pbeg.data(), Bd * 4);
  std::memcpy(mt + p->o_pcnt, pcnt.data(), Bd * 4);
  std::memcpy(mt + p->o_items, items.data(), items.size() * 4);
  std::memcpy(mt + p->o_bt, bt.data(), bt.size() * 4);
  std::memcpy(mt + p->o_rows, rows.data(), rows.size() * 4);
  if (!tiles.empty()) std::memcpy(mt + p->o_tiles, tiles.data(), tiles.size() * 4);
  if (!comb.empty()) std::memcpy(mt + p->o_comb, comb.data(), comb.size() * 4);
  return SAR_OK;
}

int ensure_meta(sar_model* m, size_t n) {
  if (n > m->meta_cap) {
    for (int i = 0; i < kMetaRing; ++i) {
      if (m->meta_host[i]) {
        cudaEventSynchronize(m->meta_ev[i]);
        cudaFreeHost(m->meta_host[i]);
        m->meta_host[i] = nullptr;
      }
    }
    size_t cap = std::max<size_t>(n * 2, 1 << 16);
    for (int i = 0; i < kMetaRing; ++i)
      SAR_TRY(check(cudaMallocHost(&m->meta_host[i], cap * 4), "meta pinned buffer"));
    m->meta_cap = cap;
  }
  if (n > m->meta_dev_cap) {
    if (m->meta_dev) {
      SAR_TRY(check(cudaDeviceSynchronize(), "meta resize sync"));
      cudaFree(m->meta_dev);
      m->meta_dev = nullptr;
    }
    size_t cap = std::max<size_t>(n * 2, 1 << 16);
    SAR_TRY(check(cudaMalloc(&m->meta_dev, cap * 4), "meta device buffer"));
    m->meta_dev_cap = cap;
  }
  return SAR_OK;
}

// One partials buffer per step: the decode split partials [parts][qh][d + 2],
// then (256-byte aligned) the chunk key-range partials [slots][128][qh][d + 4].
size_t decode_partials_floats(const Plan& p, const sar_dims& d) {
  return ((size_t)p.n_parts * d.n_q_heads * (d.head_dim + 2) + 63) & ~(size_t)63;
}
size_t partials_floats(const Plan& p, const sar_dims& d) {
  return std::max<size_t>(64, decode_partials_floats(p, d) +
                                  (size_t)p.n_cparts * sar::kChunkTileRowsTc * d.n_q_heads * (d.head_dim + 4));
}

int ensure_partials(sar_model* m, size_t floats) {
  if (floats <= m->partials_cap) return SAR_OK;
  if (m->partials) {
    SAR_TRY(check(cudaDeviceSynchronize(), "partials resize sync"));
    cudaFree(m->partials);
    m->partials = nullptr;
  }
  size_t cap = std::max<size_t>(floats * 2, 1 << 20);
  SAR_TRY(check(cudaMalloc(&m->partials, cap * 4), "decode partials"));
  m->partials_cap = cap;
  return SAR_OK;
}

// Checks the model state and plans the step (host only).
int plan_step(sar_model* m, sar_kv* kv, const sar_batch* b, bool logits, Plan* p, std::vector<int32_t>* meta) {
  const sar_dims& d = m->d;
  for (int l = 0; l < d.n_layers; ++l)
    if (!m->L[l].set) return set_error(SAR_ERR_INVALID_ARG, "step: layer weights not set");
  if (logits && (d.vocab == 0 || !m->head_set)) return set_error(SAR_ERR_INVALID_ARG, "step: logits requested without a head");
  return validate_and_plan(plan_env(m, kv), b, p, meta);
}

// Launches the step's kernels on `s`, reading the plan's metadata at device
// address `md` and keeping decode split partials in `partials`.
int launch_step(sar_model* m, sar_kv* kv, const sar_batch* b, const Plan& p, const int32_t* md, float* partials,
                const void* in, float* h, float* logits, void* layer_out, cudaStream_t s) {
  const sar_dims& d = m->d;
  const int M = p.M, H = d.hidden;
  // Small steps (the swap tiling): a weight tile per CTA leaves most SMs idle
  // for the QKV and gate/up projections (48 and 224 tiles at Mistral's
  // shape), so when the tiling's cost model splits K they accumulate split-K
  // into fp32 scratch cleared by the preceding norm, and small kernels apply
  // the rotary embedding + KV append and silu(gate)*up afterwards.
  bool qkv_split = false, gu_split = false;
  if (M <= kSmallStepRows && m->gu32) {
    sar::GemmCfg gc;
    qkv_split = sar::gemm_config(M, m->qkv_n, H, SAR_EPI_RESIDUAL, SAR_GEMM_AUTO, &gc, true) == SAR_OK &&
                gc.swap && gc.splits > 1;
    gu_split = sar::gemm_config(M, 2 * d.ffn, H, SAR_EPI_RESIDUAL, SAR_GEMM_AUTO, &gc, true) == SAR_OK &&
               gc.swap && gc.splits > 1;
  }
  float* qkv_zero = qkv_split ? m->qkv32 : nullptr;
  const size_t qkv_zero_n = qkv_split ? (size_t)M * m->qkv_n : 0;

  for (int l = 0; l < d.n_layers; ++l) {
    LayerW& w = m->L[l];
    if (l == 0) {
      // a0 + a1: stacked rows (chunk first, then decodes) into the fp32
      // residual stream, normalised for layer 0 in the same pass; also clears
      // the logits rows, which the LM head GEMM adds its K ranges into
      Prof pr(m, SAR_K_EMBED, s);
      SAR_TRY(sar::launch_input_norm(b->in_kind, in, m->embed, d.vocab, h, w.n1, m->xn, M, H, d.rms_eps, d.storage,
                                     m->err, s, logits, logits ? (size_t)p.R * d.vocab : 0, md + p.o_pos,
                                     m->inv_freq, m->rope_cs, d.head_dim / 2, d.max_tokens, qkv_zero, qkv_zero_n));
    } else {
      Prof pr(m, SAR_K_RMSNORM, s);
      SAR_TRY(sar::launch_rmsnorm(h, w.n1, m->xn, M, H, d.rms_eps, nullptr, d.storage, s, qkv_zero, qkv_zero_n));
    }
    uint16_t* kc = kv->k + (size_t)l * kv->layer_elems;
    uint16_t* vc = kv->v + (size_t)l * kv->layer_elems;
    {
      // a2 + a3: the projection's epilogue rotates q and k at the rows'
      // positions and appends k and v into their page slots
      Prof pr(m, SAR_K_GEMM_QKV, s);
      sar::RopeEpi rp;
      rp.pos = md + p.o_pos;
      rp.slot = md + p.o_slot;
      rp.cs = m->rope_cs;
      rp.cs_ld = d.max_tokens;
      rp.k_cache = kc;
      rp.v_cache = vc;
      rp.qh = d.n_q_heads;
      rp.kvh = d.n_kv_heads;
      rp.hd = d.head_dim;
      rp.page_size = kv->page_size;
      rp.num_pages = kv->num_pages;
      rp.kmap = &kv->tmk[l];
      rp.vmap = &kv->tmv[l];
      if (qkv_split) {
        SAR_TRY(run_gemm(m, m->xn, M, w.m_qkv, m->qkv_n, H, SAR_EPI_RESIDUAL, m->qkv32, m->qkv32, s));
        SAR_TRY(sar::launch_rope_append(m->qkv32, m->qkv_n, M, rp, d.storage, m->err, s));
      } else {
        SAR_TRY(run_gemm(m, m->xn, M, w.m_qkv, m->qkv_n, H, sar::kEpiRope, m->qkv32, nullptr, s, &rp));
      }
    }
    // two-stream split: chunk attention forks onto the side stream after the
    // QKV projection and joins before the O projection
    const bool ov = m->overlap && (!m->prof || m->capturing) && p.Lp > 0 && p.Bd > 0;
    cudaStream_t sc = s;
    if (ov) {
      SAR_TRY(check(cudaEventRecord(m->ev_fork, s), "overlap: fork"));
      SAR_TRY(check(cudaStreamWaitEvent(m->side, m->ev_fork, 0), "overlap: side wait"));
      sc = m->side;
    }
    sar::ChunkAttnArgs ca{};
    if (p.Lp > 0) {
      ca.q32 = m->qkv32;
      ca.ld32 = m->qkv_n;
      ca.out = m->attn;
      ca.k_cache = kc;
      ca.v_cache = vc;
      ca.bt = md + p.o_pbt;
      ca.tiles = md + p.o_tiles;
      ca.n_tiles = p.n_tiles;
      ca.ld = m->qkv_n;
      ca.ld_out = m->qd;
      ca.qh = d.n_q_heads;
      ca.kvh = d.n_kv_heads;
      ca.d = d.head_dim;
      ca.page_size = kv->page_size;
      ca.num_pages = kv->num_pages;
      ca.storage = d.storage;
      ca.err = m->err;
      ca.window = d.sliding_window;
      ca.partials = partials + decode_partials_floats(p, d);
      ca.comb = md + p.o_comb;
      ca.n_comb = p.n_comb;
      ca.dual = p.chunk_dual;
    }
    sar::DecodeAttnArgs da{};
    if (p.Bd > 0) {
      da.qkv = nullptr;  // the fp32 query rows below are read instead
      da.out = m->attn + (size_t)p.Lp * m->qd;
      da.storage = d.storage;
      da.q32 = m->qkv32 + (size_t)p.Lp * m->qkv_n;
      da.ld32 = m->qkv_n;
      da.k_cache = kc;
      da.v_cache = vc;
      da.items = md + p.o_items;
      da.nkeys = md + p.o_nkeys;
      da.bt_off = md + p.o_btoff;
      da.bt_len = md + p.o_btlen;
      da.bt = md + p.o_bt;
      da.parts_begin = md + p.o_pbeg;
      da.parts_count = md + p.o_pcnt;
      da.partials = p.n_parts > 0 ? partials : nullptr;
      da.n_items = p.n_items;
      da.n_decode = p.Bd;
      da.ld = m->qkv_n;
      da.ld_out = m->qd;
      da.qh = d.n_q_heads;
      da.kvh = d.n_kv_heads;
      da.d = d.head_dim;
      da.page_size = kv->page_size;
      da.num_pages = kv->num_pages;
      da.err = m->err;
      da.window = d.sliding_window;
    }
    auto run_chunk = [&](cudaStream_t st) -> int {
      Prof pr(m, SAR_K_CHUNK_ATTN, s);
      if (sar::chunk_attention_tc_supported(ca)) return sar::launch_chunk_attention_tc(ca, kv->tmk[l], kv->tmv[l], st);
      return sar::launch_chunk_attention(ca, st);
    };
    // The chunk and decode attention kernels read the QKV projection's output
    // only.  When both run on this stream with the tcgen05 chunk kernel, the
    // decode kernel goes first and the chunk kernel right behind it, without
    // waiting for it: its CTAs take the SMs the decode kernel's draining tail
    // leaves idle (a memory-bound kernel's last, shortest ranges), and it
    // waits for the decode kernel only before exiting; the decodes' merge
    // follows.  (Not while profiling: the per-kernel events would serialise
    // the two anyway.)
    const bool behind = !ov && !m->prof && p.Lp > 0 && p.Bd > 0 && sar::chunk_attention_tc_supported(ca);
    if (behind) {
      da.defer_combine = true;
      ca.wait_at_end = 1;
      SAR_TRY(sar::launch_decode_attention(da, kv->tmk[l], kv->tmv[l], s));
      SAR_TRY(run_chunk(s));
      SAR_TRY(sar::launch_decode_combine(da, s));
    } else {
      if (p.Lp > 0) SAR_TRY(run_chunk(sc));
      if (p.Bd > 0) {
        // the merge of the key-range partials launched (and timed) on its own
        da.defer_combine = true;
        {
          Prof pr(m, SAR_K_DECODE_ATTN, s);
          SAR_TRY(sar::launch_decode_attention(da, kv->tmk[l], kv->tmv[l], s));
        }
        if (da.partials) {
          Prof pr(m, SAR_K_DECODE_COMBINE, s);
          SAR_TRY(sar::launch_decode_combine(da, s));
        }
      }
    }
    if (ov) {
      SAR_TRY(check(cudaEventRecord(m->ev_join, m->side), "overlap: join"));
      SAR_TRY(check(cudaStreamWaitEvent(s, m->ev_join, 0), "overlap: main wait"));
    }
    {
      Prof pr(m, SAR_K_GEMM_O, s);
      SAR_TRY(run_gemm(m, m->attn, M, w.m_o, H, m->qd, SAR_EPI_RESIDUAL, h, h, s));
    }
    {
      Prof pr(m, SAR_K_RMSNORM, s);
      SAR_TRY(sar::launch_rmsnorm(h, w.n2, m->xn, M, H, d.rms_eps, nullptr, d.storage, s,
                                  gu_split ? m->gu32 : nullptr, gu_split ? (size_t)M * 2 * d.ffn : 0));
    }
    {
      Prof pr(m, SAR_K_GEMM_GATEUP, s);
      if (gu_split) {
        SAR_TRY(run_gemm(m, m->xn, M, w.m_gu, 2 * d.ffn, H, SAR_EPI_RESIDUAL, m->gu32, m->gu32, s));
        SAR_TRY(sar::launch_swiglu_finish(m->gu32, m->act, M, d.ffn, d.storage, s));
      } else {
        SAR_TRY(run_gemm(m, m->xn, M, w.m_gu, 2 * d.ffn, H, SAR_EPI_SWIGLU, m->act, nullptr, s));
      }
    }
    {
      Prof pr(m, SAR_K_GEMM_DOWN, s);
      SAR_TRY(run_gemm(m, m->act, M, w.m_d, H, d.ffn, SAR_EPI_RESIDUAL, h, h, s));
    }
    if (layer_out)
      SAR_TRY(check(cudaMemcpyAsync(static_cast<float*>(layer_out) + (size_t)l * M * H, h, (size_t)M * H * 4,
                                    cudaMemcpyDeviceToDevice, s),
                    "layer output copy"));
  }
  if (logits) {
    {
      Prof pr(m, SAR_K_HEAD_NORM, s);
      SAR_TRY(sar::launch_rmsnorm(h, m->final_norm, m->hrows, p.R, H, d.rms_eps, md + p.o_rows, d.storage, s));
    }
    {
      Prof pr(m, SAR_K_GEMM_HEAD, s);
      // the LM head streams its whole weight (262 MB at Mistral's shape) for a
      // few sampled rows: the swap tiling shares its K slabs out over every SM
      // (65 rows, standalone, L2 flushed: 62.2 us against 65.2 us for AUTO's
      // 128x256 tiles on 125 SMs), and it stays ahead up to 128 rows
      SAR_TRY(run_gemm(m, m->hrows, p.R, m->m_head, d.vocab, H, SAR_EPI_RESIDUAL, logits, logits, s, nullptr,
                       p.R <= 128 ? SAR_GEMM_SWAP : SAR_GEMM_AUTO));
    }
  }
  return SAR_OK;
}

// The step proper, on device buffers: plan, stage the metadata through the
// pinned ring into the model's device buffer, launch.
int run_step(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, float* h, float* logits,
             void* layer_out, cudaStream_t s) {
  Plan p;
  thread_local std::vector<int32_t> meta;  // keeps its capacity from step to step
  SAR_TRY(plan_step(m, kv, b, logits != nullptr, &p, &meta));
  SAR_TRY(ensure_meta(m, p.total));
  SAR_TRY(ensure_partials(m, partials_floats(p, m->d)));
  const int slot = m->meta_slot;
  m->meta_slot = (slot + 1) % kMetaRing;
  SAR_TRY(check(cudaEventSynchronize(m->meta_ev[slot]), "meta ring wait"));
  std::memcpy(m->meta_host[slot], meta.data(), p.total * 4);
  SAR_TRY(check(cudaMemcpyAsync(m->meta_dev, m->meta_host[slot], p.total * 4, cudaMemcpyHostToDevice, s), "meta copy"));
  SAR_TRY(check(cudaEventRecord(m->meta_ev[slot], s), "meta event"));
  return launch_step(m, kv, b, p, m->meta_dev, m->partials, in, h, logits, layer_out, s);
}

}  // namespace

extern "C" {

int sar_model_create(const sar_dims* dims, sar_model** out) {
  if (!dims || !out) return set_error(SAR_ERR_INVALID_ARG, "model: null argument");
  const sar_dims& d = *dims;
  if (d.n_layers <= 0 || d.hidden <= 0 || d.n_q_heads <= 0 || d.n_kv_heads <= 0 || d.ffn <= 0 || d.vocab < 0 ||
      d.max_tokens <= 0 || d.max_decodes < 0 || d.max_decodes > d.max_tokens || d.sliding_window < 0)
    return set_error(SAR_ERR_INVALID_ARG, "model: bad dims");
  if (d.head_dim != 64 && d.head_dim != 128) return set_error(SAR_ERR_UNSUPPORTED, "model: head_dim must be 64 or 128");
  if (d.n_q_heads % d.n_kv_heads || d.n_q_heads / d.n_kv_heads > 8)
    return set_error(SAR_ERR_UNSUPPORTED, "model: n_q_heads must be 1..8 times n_kv_heads");
  if (d.hidden % 64 || d.ffn % 64 || (d.n_q_heads * d.head_dim) % 64 || (d.n_kv_heads * d.head_dim) % 64 ||
      d.vocab % 64)
    return set_error(SAR_ERR_UNSUPPORTED, "model: widths (and the vocabulary) must be multiples of 64");
  if (d.storage != SAR_STORAGE_F16 && d.storage != SAR_STORAGE_BF16)
    return set_error(SAR_ERR_INVALID_ARG, "model: storage must be SAR_STORAGE_F16 or SAR_STORAGE_BF16");
  sar_model* m = new sar_model();
  m->d = d;
  m->qd = d.n_q_heads * d.head_dim;
  m->kvd = d.n_kv_heads * d.head_dim;
  m->qkv_n = m->qd + 2 * m->kvd;
  const size_t H = d.hidden, F = d.ffn;
  const size_t per_layer = align256((size_t)m->qkv_n * H * 2) + align256(H * m->qd * 2) + align256(2 * F * H * 2) +
                           align256(H * F * 2) + 2 * align256(H * 4);
  const size_t head = d.vocab ? 2 * align256((size_t)d.vocab * H * 2) + align256(H * 4) : 0;
  cudaError_t e = cudaMalloc(&m->arena, per_layer * d.n_layers + head);
  if (e != cudaSuccess) {
    delete m;
    return cuda_error(e, "model: weight arena");
  }
  m->L.resize(d.n_layers);
  uint8_t* p = m->arena;
  auto take = [&](size_t bytes) { uint8_t* r = p; p += align256(bytes); return reinterpret_cast<st16*>(r); };
  auto takef = [&](size_t bytes) { uint8_t* r = p; p += align256(bytes); return reinterpret_cast<float*>(r); };
  for (int l = 0; l < d.n_layers; ++l) {
    LayerW& w = m->L[l];
    w.wqkv = take((size_t)m->qkv_n * H * 2);
    w.wo = take(H * m->qd * 2);
    w.wgu = take(2 * F * H * 2);
    w.wd = take(H * F * 2);
    w.n1 = takef(H * 4);
    w.n2 = takef(H * 4);
  }
  if (d.vocab) {
    m->embed = take((size_t)d.vocab * H * 2);
    m->lm_head = take((size_t)d.vocab * H * 2);
    m->final_norm = takef(H * 4);
  }
  // step workspace
  const size_t T = d.max_tokens;
  const size_t R = T;  // head rows: every chunk's last row and every decode row (at most all rows)
  const size_t Ts = std::min<size_t>(T, kSmallStepRows);  // rows of the small steps' split-K gate/up scratch
  const size_t ws = align256(T * H * 2) + align256(T * (d.head_dim / 2) * 8) + align256(T * m->qd * 2) + align256(T * F * 2) +
                    align256(T * H * 4) + align256(R * H * 2) + align256(T * H * 2) + align256(T * m->qkv_n * 4) +
                    align256(Ts * 2 * F * 4) + 256;
  e = cudaMalloc(&m->ws, ws);
  if (e == cudaSuccess) e = cudaMalloc(&m->err, 16);
  if (e == cudaSuccess) e = cudaMemset(m->err, 0, 16);
  if (e == cudaSuccess) e = cudaMalloc(&m->inv_freq, d.head_dim / 2 * sizeof(double));
  if (e != cudaSuccess) {
    sar_model_destroy(m);
    return cuda_error(e, "model: workspace");
  }
  p = m->ws;
  m->xn = take(T * H * 2);
  m->rope_cs = reinterpret_cast<float2*>(takef(T * (d.head_dim / 2) * 8));
  m->attn = take(T * m->qd * 2);
  m->act = take(T * F * 2);
  m->hres = takef(T * H * 4);
  m->hrows = take(R * H * 2);
  m->in_stage = take(T * H * 2);
  m->qkv32 = takef(T * m->qkv_n * 4);
  m->gu32 = takef(Ts * 2 * F * 4);
  // rotary frequencies base^(-2i/d), double precision
  std::vector<double> inv(d.head_dim / 2);
  for (int i = 0; i < d.head_dim / 2; ++i) inv[i] = std::pow((double)d.rope_base, -2.0 * i / d.head_dim);
  e = cudaMemcpy(m->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice);
  for (int i = 0; i < kMetaRing && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&m->meta_ev[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(m->meta_ev[i], 0);
  }
  if (e != cudaSuccess) {
    sar_model_destroy(m);
    return cuda_error(e, "model: init");
  }
  *out = m;
  return SAR_OK;
}

int sar_model_set_layer(sar_model* m, int32_t layer, const sar_layer_weights* w, void* stream) {
  if (!m || !w || layer < 0 || layer >= m->d.n_layers) return set_error(SAR_ERR_INVALID_ARG, "set_layer: bad argument");
  if (!w->wq || !w->wk || !w->wv || !w->wo || !w->wg || !w->wu || !w->wd || !w->norm1 || !w->norm2)
    return set_error(SAR_ERR_INVALID_ARG, "set_layer: null weight");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerW& L = m->L[layer];
  const int H = m->d.hidden, F = m->d.ffn, st = m->d.storage;
  // bf16 in, storage type out; Q/K/V stacked, gate/up interleaved in 64-row blocks
  SAR_TRY(sar::launch_convert_rows(w->wq, L.wqkv, m->qd, H, 0, 0, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wk, L.wqkv + (size_t)m->qd * H, m->kvd, H, 0, 0, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wv, L.wqkv + (size_t)(m->qd + m->kvd) * H, m->kvd, H, 0, 0, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wo, L.wo, H, m->qd, 0, 0, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wg, L.wgu, F, H, 1, 0, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wu, L.wgu, F, H, 1, 1, st, s));
  SAR_TRY(sar::launch_convert_rows(w->wd, L.wd, H, F, 0, 0, st, s));
  SAR_TRY(sar::launch_bf16_to_f32(w->norm1, L.n1, H, s));
  SAR_TRY(sar::launch_bf16_to_f32(w->norm2, L.n2, H, s));
  SAR_TRY(weight_maps(L.m_qkv, L.wqkv, m->qkv_n, H, st));
  SAR_TRY(weight_maps(L.m_o, L.wo, H, m->qd, st));
  SAR_TRY(weight_maps(L.m_gu, L.wgu, 2 * F, H, st));
  SAR_TRY(weight_maps(L.m_d, L.wd, H, F, st));
  L.set = true;
  return SAR_OK;
}

int sar_model_set_head(sar_model* m, const void* embed, const void* final_norm, const void* lm_head, void* stream) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "set_head: null model");
  if (m->d.vocab == 0) return set_error(SAR_ERR_INVALID_ARG, "set_head: model has no vocabulary");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = m->d.hidden, V = m->d.vocab, st = m->d.storage;
  if (embed) SAR_TRY(sar::launch_convert_rows(embed, m->embed, V, H, 0, 0, st, s));
  if (final_norm) SAR_TRY(sar::launch_bf16_to_f32(final_norm, m->final_norm, H, s));
  if (lm_head) {
    SAR_TRY(sar::launch_convert_rows(lm_head, m->lm_head, V, H, 0, 0, st, s));
    SAR_TRY(weight_maps(m->m_head, m->lm_head, V, H, st));
  }
  if (final_norm && lm_head) m->head_set = true;
  return SAR_OK;
}

int sar_model_destroy(sar_model* m) {
  if (!m) return SAR_OK;
  cudaDeviceSynchronize();
  for (int i = 0; i < kMetaRing; ++i) {
    if (m->meta_host[i]) cudaFreeHost(m->meta_host[i]);
    if (m->meta_ev[i]) cudaEventDestroy(m->meta_ev[i]);
  }
  if (m->ev_fork) cudaEventDestroy(m->ev_fork);
  if (m->ev_join) cudaEventDestroy(m->ev_join);
  if (m->side) cudaStreamDestroy(m->side);
  if (m->capture) cudaStreamDestroy(m->capture);
  for (auto& ep : m->ev_used) { cudaEventDestroy(ep.a); cudaEventDestroy(ep.b); }
  for (auto& ep : m->ev_free) { cudaEventDestroy(ep.a); cudaEventDestroy(ep.b); }
  cudaFree(m->meta_dev);
  cudaFree(m->partials);
  cudaFree(m->inv_freq);
  cudaFree(m->err);
  cudaFree(m->ws);
  cudaFree(m->arena);
  delete m;
  return SAR_OK;
}

int sar_sync_status(sar_model* m) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "sync_status: null model");
  int h[4] = {0, 0, 0, 0};
  SAR_TRY(check(cudaDeviceSynchronize(), "sync_status: device synchronise"));
  SAR_TRY(check(cudaMemcpy(h, m->err, 16, cudaMemcpyDeviceToHost), "sync_status: read flags"));
  SAR_TRY(check(cudaMemset(m->err, 0, 16), "sync_status: clear flags"));
  if (h[0] != 0)
    return set_error(h[0], "device flag: code " + std::to_string(h[0]) + " at site " + std::to_string(h[1]) +
                               " (detail " + std::to_string(h[2]) + ")");
  return SAR_OK;
}

int sar_kv_create(const sar_model* m, int32_t page_size, int32_t num_pages, sar_kv** out) {
  if (!m || !out) return set_error(SAR_ERR_INVALID_ARG, "kv: null argument");
  if (page_size != 16 && page_size != 32 && page_size != 64) return set_error(SAR_ERR_INVALID_ARG, "kv: page size must be 16, 32 or 64");
  if (num_pages <= 0) return set_error(SAR_ERR_INVALID_ARG, "kv: no pages");
  sar_kv* kv = new sar_kv();
  kv->m = m;
  kv->page_size = page_size;
  kv->num_pages = num_pages;
  kv->layer_elems = (size_t)num_pages * m->d.n_kv_heads * page_size * m->d.head_dim;
  const size_t bytes = kv->layer_elems * m->d.n_layers * 2;
  cudaError_t e = cudaMalloc(&kv->k, bytes);
  if (e == cudaSuccess) e = cudaMalloc(&kv->v, bytes);
  if (e == cudaSuccess) e = cudaMemset(kv->k, 0, bytes);
  if (e == cudaSuccess) e = cudaMemset(kv->v, 0, bytes);
  if (e != cudaSuccess) {
    cudaFree(kv->k);
    cudaFree(kv->v);
    delete kv;
    return cuda_error(e, "kv: arena");
  }
  kv->tmk.resize(m->d.n_layers);
  kv->tmv.resize(m->d.n_layers);
  for (int l = 0; l < m->d.n_layers; ++l) {
    int rc = sar::make_kv_tmap(&kv->tmk[l], kv->k + (size_t)l * kv->layer_elems, num_pages, m->d.n_kv_heads,
                               page_size, m->d.head_dim, m->d.storage);
    if (rc == SAR_OK)
      rc = sar::make_kv_tmap(&kv->tmv[l], kv->v + (size_t)l * kv->layer_elems, num_pages, m->d.n_kv_heads,
                             page_size, m->d.head_dim, m->d.storage);
    if (rc != SAR_OK) {
      sar_kv_destroy(kv);
      return rc;
    }
  }
  *out = kv;
  return SAR_OK;
}

int sar_kv_layer_ptr(sar_kv* kv, int32_t layer, int32_t kind, void** out) {
  if (!kv || !out || layer < 0 || layer >= kv->m->d.n_layers || (kind != 0 && kind != 1))
    return set_error(SAR_ERR_INVALID_ARG, "kv_layer_ptr: bad argument");
  *out = (kind == 0 ? kv->k : kv->v) + (size_t)layer * kv->layer_elems;
  return SAR_OK;
}

int sar_kv_destroy(sar_kv* kv) {
  if (!kv) return SAR_OK;
  cudaDeviceSynchronize();
  cudaFree(kv->k);
  cudaFree(kv->v);
  delete kv;
  return SAR_OK;
}

int sar_step(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out, float* logits_out,
             void* layer_out, void* stream) {
  if (!m || !kv || !b || !in) return set_error(SAR_ERR_INVALID_ARG, "step: null argument");
  if (kv->m != m) return set_error(SAR_ERR_INVALID_ARG, "step: KV cache belongs to another model");
  // the kernels move these with 16-byte (outputs) and 8-byte (bf16 input rows) accesses
  if ((reinterpret_cast<uintptr_t>(hidden_out) & 15) || (reinterpret_cast<uintptr_t>(logits_out) & 15) ||
      (b->in_kind == SAR_IN_HIDDEN && (reinterpret_cast<uintptr_t>(in) & 7)))
    return set_error(SAR_ERR_INVALID_ARG, "step: hidden_out / logits_out must be 16-byte and in 8-byte aligned");
  float* h = hidden_out ? static_cast<float*>(hidden_out) : m->hres;
  return run_step(m, kv, b, in, h, logits_out, layer_out, static_cast<cudaStream_t>(stream));
}

int sar_step_host(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out, float* logits_out,
                  void* layer_out, void* stream) {
  if (!m || !kv || !b || !in) return set_error(SAR_ERR_INVALID_ARG, "step_host: null argument");
  if (layer_out) return set_error(SAR_ERR_INVALID_ARG, "step_host: layer outputs are only returned on device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (b->n_more_prefill < 0 || (b->n_more_prefill > 0 && !b->more_prefill))
    return set_error(SAR_ERR_INVALID_ARG, "step_host: bad chunk list");
  int64_t M = b->n_decode;
  for (const sar_prefill& c : batch_chunks(b)) M += c.len;
  if (M <= 0 || M > m->d.max_tokens) return set_error(SAR_ERR_INVALID_ARG, "step_host: bad row count");
  const int R = (b->has_prefill ? 1 : 0) + b->n_more_prefill + b->n_decode;
  const size_t in_bytes = b->in_kind == SAR_IN_TOKENS ? (size_t)M * 4 : (size_t)M * m->d.hidden * 2;
  SAR_TRY(check(cudaMemcpyAsync(m->in_stage, in, in_bytes, cudaMemcpyHostToDevice, s), "step_host: input copy"));
  if (logits_out && (size_t)R > m->logits_stage_rows) {
    if (m->logits_stage) {
      SAR_TRY(check(cudaStreamSynchronize(s), "step_host: logits stage resize"));
      cudaFree(m->logits_stage);
      m->logits_stage = nullptr;
      m->logits_stage_rows = 0;
    }
    const size_t rows = std::max<size_t>((size_t)R, (size_t)m->d.max_decodes + 1);
    SAR_TRY(check(cudaMalloc(&m->logits_stage, rows * m->d.vocab * 4), "step_host: logits stage"));
    m->logits_stage_rows = rows;
  }
  SAR_TRY(run_step(m, kv, b, m->in_stage, m->hres, logits_out ? m->logits_stage : nullptr, nullptr, s));
  if (hidden_out)
    SAR_TRY(check(cudaMemcpyAsync(hidden_out, m->hres, (size_t)M * m->d.hidden * 4, cudaMemcpyDeviceToHost, s), "step_host: hidden copy"));
  if (logits_out)
    SAR_TRY(check(cudaMemcpyAsync(logits_out, m->logits_stage, (size_t)R * m->d.vocab * 4, cudaMemcpyDeviceToHost, s),
                  "step_host: logits copy"));
  return check(cudaStreamSynchronize(s), "step_host: synchronise");
}

int sar_sample_greedy(sar_model* m, const float* logits, int32_t rows, int32_t* tokens_out, void* stream) {
  if (!m || !logits || !tokens_out || rows < 0) return set_error(SAR_ERR_INVALID_ARG, "sample: bad argument");
  if (m->d.vocab == 0) return set_error(SAR_ERR_INVALID_ARG, "sample: model has no vocabulary");
  return sar::launch_argmax(logits, rows, m->d.vocab, tokens_out, static_cast<cudaStream_t>(stream));
}

int sar_model_set_chunk_split(sar_model* m, int32_t on) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "chunk_split: null model");
  m->chunk_split = on != 0;
  return SAR_OK;
}

int sar_model_set_overlap(sar_model* m, int32_t on) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "overlap: null model");
  if (on && !m->side) {
    int lo = 0, hi = 0;
    SAR_TRY(check(cudaDeviceGetStreamPriorityRange(&lo, &hi), "overlap: stream priorities"));
    SAR_TRY(check(cudaStreamCreateWithPriority(&m->side, cudaStreamNonBlocking, hi), "overlap: side stream"));
    SAR_TRY(check(cudaEventCreateWithFlags(&m->ev_fork, cudaEventDisableTiming), "overlap: fork event"));
    SAR_TRY(check(cudaEventCreateWithFlags(&m->ev_join, cudaEventDisableTiming), "overlap: join event"));
  }
  m->overlap = on != 0;
  return SAR_OK;
}

int sar_profile_enable(sar_model* m, int32_t on) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "profile: null model");
  m->prof = on != 0;
  return SAR_OK;
}

int sar_profile_read(sar_model* m, double* ms, int64_t* launches, int32_t n_kinds) {
  if (!m) return set_error(SAR_ERR_INVALID_ARG, "profile: null model");
  SAR_TRY(check(cudaDeviceSynchronize(), "profile: synchronise"));
  for (auto& ep : m->ev_used) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, ep.a, ep.b) == cudaSuccess) {
      m->prof_ms[ep.kind] += t;
      m->prof_n[ep.kind] += 1;
    }
    m->ev_free.push_back(ep);
  }
  m->ev_used.clear();
  for (int k = 0; k < n_kinds && k < SAR_K_COUNT; ++k) {
    if (ms) ms[k] = m->prof_ms[k];
    if (launches) launches[k] = m->prof_n[k];
  }
  for (int k = 0; k < SAR_K_COUNT; ++k) {
    m->prof_ms[k] = 0.0;
    m->prof_n[k] = 0;
  }
  return SAR_OK;
}

int sar_model_debug_buffer(sar_model* m, int32_t which, void** out) {
  if (!m || !out) return set_error(SAR_ERR_INVALID_ARG, "debug_buffer: null argument");
  switch (which) {
    case 0: *out = m->xn; break;
    case 1: *out = m->rope_cs; break;
    case 2: *out = m->attn; break;
    case 3: *out = m->act; break;
    case 4: *out = m->hres; break;
    case 5: *out = m->qkv32; break;
    default: return set_error(SAR_ERR_INVALID_ARG, "debug_buffer: unknown buffer");
  }
  return SAR_OK;
}

// ---- single-kernel entry points ------------------------------------------------

int sar_op_gemm(const void* a, const void* w, void* c, const void* residual, int32_t M, int32_t N, int32_t K,
                int32_t epilogue, int32_t variant, int32_t storage, void* stream) {
  if (!a || !w || !c) return set_error(SAR_ERR_INVALID_ARG, "op_gemm: null pointer");
  if (epilogue < SAR_EPI_STORE || epilogue > SAR_EPI_F32) return set_error(SAR_ERR_INVALID_ARG, "op_gemm: bad epilogue");
  if (storage != SAR_STORAGE_F16 && storage != SAR_STORAGE_BF16) return set_error(SAR_ERR_INVALID_ARG, "op_gemm: bad storage");
  int* err = nullptr;
  SAR_TRY(op_flags(&err));
  sar::GemmCfg cfg;
  SAR_TRY(sar::gemm_config(M, N, K, epilogue, variant, &cfg, epilogue == SAR_EPI_RESIDUAL && c == residual));
  CUtensorMap amap, wmap;
  SAR_TRY(sar::make_tmap_16(&amap, a, M, K, cfg.swap ? cfg.b_box_rows : cfg.a_box_rows, storage));
  SAR_TRY(sar::make_tmap_16(&wmap, w, N, K, cfg.swap ? cfg.a_box_rows : cfg.b_box_rows, storage));
  return sar::gemm_launch(cfg, amap, wmap, M, N, K, epilogue, storage, c, residual, err, static_cast<cudaStream_t>(stream));
}

int sar_op_wait_check(int64_t limit_ns, int32_t arrivals, void* stream) {
  if (limit_ns <= 0 || arrivals < 0 || arrivals > 2) return set_error(SAR_ERR_INVALID_ARG, "op_wait_check: bad argument");
  int* err = nullptr;
  SAR_TRY(op_flags(&err));
  return sar::launch_wait_check((uint64_t)limit_ns, arrivals, err, static_cast<cudaStream_t>(stream));
}

int sar_op_sync_status(void) {
  int* err = nullptr;
  SAR_TRY(op_flags(&err));
  int h[4] = {0, 0, 0, 0};
  SAR_TRY(check(cudaDeviceSynchronize(), "op_sync_status: device synchronise"));
  SAR_TRY(check(cudaMemcpy(h, err, 16, cudaMemcpyDeviceToHost), "op_sync_status: read flags"));
  SAR_TRY(check(cudaMemset(err, 0, 16), "op_sync_status: clear flags"));
  if (h[0] != 0)
    return set_error(h[0], "device flag: code " + std::to_string(h[0]) + " at site " + std::to_string(h[1]) +
                               " (detail " + std::to_string(h[2]) + ")");
  return SAR_OK;
}

int sar_plan_inspect(const sar_dims* dims, int32_t page_size, int32_t num_pages, int32_t sms, int32_t chunk_split,
                     const sar_batch* b, int32_t* layout, int32_t* meta, int64_t meta_cap, int64_t* meta_n) {
  if (!dims || !b || !layout || sms <= 0 || page_size <= 0 || num_pages <= 0)
    return set_error(SAR_ERR_INVALID_ARG, "plan_inspect: bad argument");
  PlanEnv env;
  env.d = *dims;
  env.page_size = page_size;
  env.num_pages = num_pages;
  env.sms = sms;
  env.has_embed = dims->vocab > 0;
  env.chunk_split = chunk_split != 0;
  Plan p;
  std::vector<int32_t> v;
  SAR_TRY(validate_and_plan(env, b, &p, &v));
  const int32_t l[25] = {p.M, p.Lp, p.Bd, p.R, p.n_items, p.n_parts, p.n_tiles, chunk_tile_rows(env.d, page_size),
                         (int32_t)p.o_pos, (int32_t)p.o_slot, (int32_t)p.o_pbt, (int32_t)p.o_nkeys,
                         (int32_t)p.o_btoff, (int32_t)p.o_btlen, (int32_t)p.o_pbeg, (int32_t)p.o_pcnt,
                         (int32_t)p.o_items, (int32_t)p.o_bt, (int32_t)p.o_rows, (int32_t)p.o_tiles,
                         (int32_t)p.total, p.n_comb, p.n_cparts, (int32_t)p.o_comb, p.chunk_dual};
  std::memcpy(layout, l, sizeof(l));
  if (meta_n) *meta_n = (int64_t)v.size();
  if (meta) {
    if ((int64_t)v.size() > meta_cap) return set_error(SAR_ERR_INVALID_ARG, "plan_inspect: metadata buffer too small");
    std::memcpy(meta, v.data(), v.size() * 4);
  }
  return SAR_OK;
}

int sar_op_rmsnorm(const void* x, const void* gain, void* y, int32_t rows, int32_t hidden, float eps, int32_t storage,
                   void* stream) {
  if (!x || !gain || !y || rows < 0 || hidden <= 0) return set_error(SAR_ERR_INVALID_ARG, "op_rmsnorm: bad argument");
  if (storage != SAR_STORAGE_F16 && storage != SAR_STORAGE_BF16) return set_error(SAR_ERR_INVALID_ARG, "op_rmsnorm: bad storage");
  return sar::launch_rmsnorm(static_cast<const float*>(x), static_cast<const float*>(gain), y, rows, hidden, eps,
                             nullptr, storage, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---- CUDA graphs of a step -------------------------------------------------

struct sar_graph {
  sar_model* m = nullptr;
  sar_kv* kv = nullptr;
  Plan p;
  int in_kind = 0;
  // the captured step's buffers (for sar_graph_launch_host)
  void* in = nullptr;
  float* hidden = nullptr;
  float* logits = nullptr;
  int32_t* md = nullptr;       // the graph's own device copy of the step metadata
  int32_t* md_host = nullptr;  // pinned staging for sar_graph_update
  float* partials = nullptr;   // the graph's own decode split partials
  int32_t* tokens = nullptr;   // greedy picks of the captured logits rows
  cudaEvent_t staged = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  // sar_graph_enqueue_host_tokens: the input copy's own stream (so that it can
  // run while an earlier step computes), the copy's completion, and the
  // enqueued step's (token ids in host memory)
  cudaStream_t copy = nullptr;
  cudaEvent_t in_ready = nullptr;
  cudaEvent_t done = nullptr;
};

namespace {

// Two plans launch the same kernels with the same grids and argument
// addresses when every size and metadata offset agrees.
bool same_shape(const Plan& a, const Plan& b) {
  return a.M == b.M && a.Lp == b.Lp && a.Bd == b.Bd && a.R == b.R && a.n_items == b.n_items &&
         a.n_parts == b.n_parts && a.n_tiles == b.n_tiles && a.total == b.total && a.o_pos == b.o_pos &&
         a.o_slot == b.o_slot && a.o_pbt == b.o_pbt && a.o_nkeys == b.o_nkeys && a.o_btoff == b.o_btoff &&
         a.o_btlen == b.o_btlen && a.o_pbeg == b.o_pbeg && a.o_pcnt == b.o_pcnt && a.o_items == b.o_items &&
         a.o_bt == b.o_bt && a.o_rows == b.o_rows && a.o_tiles == b.o_tiles && a.n_comb == b.n_comb &&
         a.n_cparts == b.n_cparts && a.o_comb == b.o_comb && a.chunk_dual == b.chunk_dual;
}

}  // namespace

extern "C" {

int sar_graph_destroy(sar_graph* g) {
  if (!g) return SAR_OK;
  if (g->staged) cudaEventSynchronize(g->staged);
  if (g->done) cudaEventSynchronize(g->done);
  if (g->copy) cudaStreamSynchronize(g->copy);
  if (g->in_ready) cudaEventDestroy(g->in_ready);
  if (g->done) cudaEventDestroy(g->done);
  if (g->copy) cudaStreamDestroy(g->copy);
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  if (g->staged) cudaEventDestroy(g->staged);
  if (g->md_host) cudaFreeHost(g->md_host);
  cudaFree(g->md);
  cudaFree(g->partials);
  cudaFree(g->tokens);
  delete g;
  return SAR_OK;
}

int sar_graph_create(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out,
                     float* logits_out, void* layer_out, void* stream, sar_graph** out) {
  if (!m || !kv || !b || !in || !out) return set_error(SAR_ERR_INVALID_ARG, "graph: null argument");
  if (kv->m != m) return set_error(SAR_ERR_INVALID_ARG, "graph: cache of another model");
  if ((reinterpret_cast<uintptr_t>(hidden_out) & 15) || (reinterpret_cast<uintptr_t>(logits_out) & 15))
    return set_error(SAR_ERR_INVALID_ARG, "graph: outputs must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sar_graph* g = new sar_graph();
  g->m = m;
  g->kv = kv;
  g->in_kind = b->in_kind;
  g->in = const_cast<void*>(in);
  g->hidden = static_cast<float*>(hidden_out);
  g->logits = logits_out;
  std::vector<int32_t> meta;
  int rc = plan_step(m, kv, b, logits_out != nullptr, &g->p, &meta);
  // everything the captured launches point at is allocated and filled before the capture
  const size_t parts = partials_floats(g->p, m->d);
  if (rc == SAR_OK) rc = check(cudaMalloc(&g->md, g->p.total * 4), "graph: metadata");
  if (rc == SAR_OK) rc = check(cudaMallocHost(&g->md_host, g->p.total * 4), "graph: metadata staging");
  if (rc == SAR_OK) rc = check(cudaMalloc(&g->partials, parts * 4), "graph: partials");
  if (rc == SAR_OK && logits_out)
    rc = check(cudaMalloc(&g->tokens, std::max<size_t>(16, (size_t)g->p.R * 4)), "graph: token ids");
  if (rc == SAR_OK) rc = check(cudaEventCreateWithFlags(&g->staged, cudaEventDisableTiming), "graph: event");
  if (rc == SAR_OK) {
    std::memcpy(g->md_host, meta.data(), g->p.total * 4);
    rc = check(cudaMemcpyAsync(g->md, g->md_host, g->p.total * 4, cudaMemcpyHostToDevice, s), "graph: metadata copy");
  }
  if (rc == SAR_OK) rc = check(cudaEventRecord(g->staged, s), "graph: staged");
  if (rc == SAR_OK) rc = check(cudaStreamSynchronize(s), "graph: synchronise");
  if (rc == SAR_OK && m->overlap && !m->side) rc = sar_model_set_overlap(m, 1);
  // capture on the model's own stream (the caller's may be the legacy stream,
  // which cannot be captured); the graph then launches on any stream
  if (rc == SAR_OK && !m->capture)
    rc = check(cudaStreamCreateWithFlags(&m->capture, cudaStreamNonBlocking), "graph: capture stream");
  if (rc == SAR_OK) {
    cudaStream_t cs = m->capture;
    rc = check(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "graph: begin capture");
    if (rc == SAR_OK) {
      m->capturing = true;
      const int lrc = launch_step(m, kv, b, g->p, g->md, g->partials, in, static_cast<float*>(hidden_out ? hidden_out : m->hres),
                                  logits_out, layer_out, cs);
      m->capturing = false;
      const int erc = check(cudaStreamEndCapture(cs, &g->graph), "graph: end capture");
      rc = lrc != SAR_OK ? lrc : erc;
    }
  }
  if (rc == SAR_OK) rc = check(cudaGraphInstantiate(&g->exec, g->graph, 0), "graph: instantiate");
  if (rc != SAR_OK) {
    sar_graph_destroy(g);
    return rc;
  }
  *out = g;
  return SAR_OK;
}

int sar_graph_update(sar_graph* g, const sar_batch* b, void* stream) {
  if (!g || !b) return set_error(SAR_ERR_INVALID_ARG, "graph: null argument");
  if (b->in_kind != g->in_kind) return set_error(SAR_ERR_INVALID_ARG, "graph: input kind differs from the captured step");
  Plan p;
  thread_local std::vector<int32_t> meta;  // keeps its capacity from update to update
  SAR_TRY(plan_step(g->m, g->kv, b, false, &p, &meta));
  if (!same_shape(p, g->p))
    return set_error(SAR_ERR_INVALID_ARG, "graph: the batch's plan differs in shape from the captured step");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SAR_TRY(check(cudaEventSynchronize(g->staged), "graph: staging wait"));
  std::memcpy(g->md_host, meta.data(), p.total * 4);
  SAR_TRY(check(cudaMemcpyAsync(g->md, g->md_host, p.total * 4, cudaMemcpyHostToDevice, s), "graph: metadata copy"));
  return check(cudaEventRecord(g->staged, s), "graph: staged");
}

int sar_graph_launch(sar_graph* g, void* stream) {
  if (!g) return set_error(SAR_ERR_INVALID_ARG, "graph: null graph");
  SAR_TRY(check(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)), "graph: launch"));
  return SAR_OK;
}

namespace {

// Host <-> device copy of a step's rows (UVA picks the direction).  A grid-wide
// copy kernel over pinned memory measured no faster than the copy engine here:
// the host link, not the engine, sets the rate.
int host_copy(void* dst, const void* src, size_t n, cudaStream_t s) {
  return check(cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, s), "host copy");
}

}  // namespace

int sar_graph_launch_host(sar_graph* g, const void* in, float* logits_out, float* hidden_out, void* stream) {
  if (!g || !in) return set_error(SAR_ERR_INVALID_ARG, "graph: null argument");
  if ((logits_out && !g->logits) || (hidden_out && !g->hidden))
    return set_error(SAR_ERR_INVALID_ARG, "graph: output not captured");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t M = (size_t)g->p.M, H = (size_t)g->m->d.hidden;
  const size_t in_bytes = g->in_kind == SAR_IN_TOKENS ? M * 4 : M * H * 2;
  SAR_TRY(host_copy(g->in, in, in_bytes, s));
  SAR_TRY(check(cudaGraphLaunch(g->exec, s), "graph: launch"));
  if (logits_out) SAR_TRY(host_copy(logits_out, g->logits, (size_t)g->p.R * g->m->d.vocab * 4, s));
  if (hidden_out) SAR_TRY(host_copy(hidden_out, g->hidden, M * H * 4, s));
  return check(cudaStreamSynchronize(s), "graph: synchronise");
}

int sar_graph_launch_host_tokens(sar_graph* g, const void* in, int32_t* tokens_out, void* stream) {
  if (!g || !in || !tokens_out) return set_error(SAR_ERR_INVALID_ARG, "graph: null argument");
  if (!g->logits) return set_error(SAR_ERR_INVALID_ARG, "graph: logits not captured");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t M = (size_t)g->p.M, H = (size_t)g->m->d.hidden;
  const size_t in_bytes = g->in_kind == SAR_IN_TOKENS ? M * 4 : M * H * 2;
  SAR_TRY(host_copy(g->in, in, in_bytes, s));
  SAR_TRY(check(cudaGraphLaunch(g->exec, s), "graph: launch"));
  SAR_TRY(sar::launch_argmax(g->logits, g->p.R, g->m->d.vocab, g->tokens, s));
  SAR_TRY(host_copy(tokens_out, g->tokens, (size_t)g->p.R * 4, s));
  return check(cudaStreamSynchronize(s), "graph: synchronise");
}

int sar_graph_enqueue_host_tokens(sar_graph* g, const void* in, int32_t* tokens_out, void* stream) {
  if (!g || !in || !tokens_out) return set_error(SAR_ERR_INVALID_ARG, "graph: null argument");
  if (!g->logits) return set_error(SAR_ERR_INVALID_ARG, "graph: logits not captured");
  if (!g->copy) {
    SAR_TRY(check(cudaStreamCreateWithFlags(&g->copy, cudaStreamNonBlocking), "graph: copy stream"));
    SAR_TRY(check(cudaEventCreateWithFlags(&g->in_ready, cudaEventDisableTiming), "graph: event"));
    SAR_TRY(check(cudaEventCreateWithFlags(&g->done, cudaEventDisableTiming), "graph: event"));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t M = (size_t)g->p.M, H = (size_t)g->m->d.hidden;
  const size_t in_bytes = g->in_kind == SAR_IN_TOKENS ? M * 4 : M * H * 2;
  // the input buffer is rewritten once this graph's previous step has ended
  // (a no-op wait before the first enqueue)
  SAR_TRY(check(cudaStreamWaitEvent(g->copy, g->done, 0), "graph: copy wait"));
  SAR_TRY(host_copy(g->in, in, in_bytes, g->copy));
  SAR_TRY(check(cudaEventRecord(g->in_ready, g->copy), "graph: input copied"));
  SAR_TRY(check(cudaStreamWaitEvent(s, g->in_ready, 0), "graph: input wait"));
  SAR_TRY(check(cudaGraphLaunch(g->exec, s), "graph: launch"));
  SAR_TRY(sar::launch_argmax(g->logits, g->p.R, g->m->d.vocab, g->tokens, s));
  SAR_TRY(host_copy(tokens_out, g->tokens, (size_t)g->p.R * 4, s));
  return check(cudaEventRecord(g->done, s), "graph: step enqueued");
}

int sar_graph_wait(sar_graph* g) {
  if (!g) return set_error(SAR_ERR_INVALID_ARG, "graph: null graph");
  if (!g->done) return SAR_OK;
  return check(cudaEventSynchronize(g->done), "graph: wait");
}

}  // extern "C"
