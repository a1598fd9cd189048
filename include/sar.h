/*
 * sar.h -- C ABI of the hybrid-batch decoder step (chunked prefill + piggybacked
 * decodes) for one GB300 GPU.
 *
 * The step follows the scheme of "SARATHI: Efficient LLM Inference by
 * Piggybacking Decodes with Chunked Prefills" (reading notes, part 2 section 3,
 * "merge / split / merge"): one prefill chunk of Lp tokens and Bd decode tokens
 * are stacked into a single [Lp+Bd, H] activation; every projection runs as one
 * GEMM over all rows; attention is split by row range (the chunk attends
 * causally to its own keys and to the earlier chunks' keys in the paged KV
 * cache; each decode attends to its own paged history); the two attention
 * outputs are written back into one contiguous buffer.  The scheduler entry
 * points restate Algorithm 3 (stall-free batching) of "Taming
 * Throughput-Latency Tradeoff in LLM Inference with Sarathi-Serve" (section 2,
 * Q2 item 2; section 3 flowchart).
 *
 * Conventions
 *  - Every call returns an int status (SAR_OK = 0).  On failure
 *    sar_last_error() returns a thread-local message.  Validation errors are
 *    returned before anything is launched.
 *  - "device" pointers are CUDA device addresses on the current device;
 *    "host" pointers are ordinary host memory.  A stream argument is a
 *    cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Matrices are row-major.  Weights use the linear-layer layout
 *    [out_features, in_features] and are passed in bf16.  Inside, the model
 *    stores weights, activations and the KV cache in one 16-bit storage type
 *    (fp16 by default, bf16 on request), accumulates every product in fp32
 *    and carries the residual stream between layers in fp32.
 *  - Work on a stream is asynchronous; device-side error flags (a wait that
 *    gave up, an index out of bounds) are read back by sar_sync_status().
 */
#ifndef SAR_H
#define SAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum {
  SAR_OK = 0,
  SAR_ERR_INVALID_ARG = 1, /* bad argument or batch descriptor               */
  SAR_ERR_NO_PAGES = 2,    /* KV page pool exhausted (scheduler)             */
  SAR_ERR_OOM = 3,         /* device allocation failed                        */
  SAR_ERR_CUDA = 4,        /* a CUDA runtime call failed                      */
  SAR_ERR_BOUNDS = 5,      /* a device-side bounds check fired               */
  SAR_ERR_TIMEOUT = 6,     /* a device-side wait gave up (kernel returned)   */
  SAR_ERR_UNSUPPORTED = 7  /* shape outside what the kernels implement       */
};

typedef struct sar_model sar_model;
typedef struct sar_kv sar_kv;
typedef struct sar_sched sar_sched;
typedef struct sar_graph sar_graph;

/* Thread-local text of the last error (never NULL). */
const char* sar_last_error(void);

/* Number of kernels this library has launched in this process. */
int64_t sar_launch_count(void);

/* ---- model ------------------------------------------------------------- */

/* Storage type of weights, activations and KV pages.  fp16 keeps 3 more
 * mantissa bits than bf16 at the same width and tensor-core rate; bf16 weights
 * convert to it exactly (apart from magnitudes below 2^-14). */
enum { SAR_STORAGE_F16 = 0, SAR_STORAGE_BF16 = 1 };

/* Decoder shape (Llama/Mistral-style: RMSNorm, GQA attention with rotary
 * embedding, SwiGLU FFN).  head_dim must be 64 or 128; hidden, ffn and
 * n_q_heads*head_dim multiples of 64; n_q_heads a multiple of n_kv_heads with
 * at most 8 query heads per KV head.  vocab = 0 means no embedding / head.
 * max_tokens bounds Lp+Bd of any step (sizes the step workspace);
 * max_decodes bounds Bd; storage is SAR_STORAGE_F16 or SAR_STORAGE_BF16. */
typedef struct sar_dims {
  int32_t n_layers;
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t ffn;
  int32_t vocab;
  float rms_eps;
  float rope_base;
  int32_t max_tokens;
  int32_t max_decodes;
  int32_t storage;
  /* Sliding-window attention: a query at position p sees the keys at
   * positions (p - sliding_window, p], itself included; 0 = every earlier
   * position (full causal).  Mistral-7B's attention is listed as GQA with a
   * sliding window (Sarathi-Serve digest, appendix table of evaluated
   * models); the pages give no window length. */
  int32_t sliding_window;
} sar_dims;

/* One layer's weights: device bf16, [out, in] row-major; norm gains bf16 [hidden]. */
typedef struct sar_layer_weights {
  const void* wq; /* [n_q_heads*head_dim, hidden]  */
  const void* wk; /* [n_kv_heads*head_dim, hidden] */
  const void* wv; /* [n_kv_heads*head_dim, hidden] */
  const void* wo; /* [hidden, n_q_heads*head_dim]  */
  const void* wg; /* [ffn, hidden] */
  const void* wu; /* [ffn, hidden] */
  const void* wd; /* [hidden, ffn] */
  const void* norm1;
  const void* norm2;
} sar_layer_weights;

/* Creates a model on the current device and allocates its weight arena and
 * step workspace (sized by max_tokens).  The model owns that memory until
 * sar_model_destroy. */
int sar_model_create(const sar_dims* dims, sar_model** out);

/* Copies layer `layer`'s bf16 weights into the model's arena, converting
 * them to the storage type and repacking them (Q/K/V fused into one
 * [q+2kv, hidden] matrix; gate and up interleaved in blocks of 64 rows so one
 * GEMM epilogue forms silu(gate)*up; norm gains kept in fp32).  Runs on
 * `stream`; the caller may free its tensors once the stream has passed the
 * copies (e.g. after a stream synchronise). */
int sar_model_set_layer(sar_model* m, int32_t layer, const sar_layer_weights* w, void* stream);

/* Copies the embedding [vocab, hidden], final norm gain [hidden] and LM head
 * [vocab, hidden] (device bf16).  Any of them may be NULL if unused. */
int sar_model_set_head(sar_model* m, const void* embed, const void* final_norm,
                       const void* lm_head, void* stream);

int sar_model_destroy(sar_model* m);

/* Reads back and clears the model's device error flags (synchronises the
 * device).  Returns SAR_OK, SAR_ERR_TIMEOUT or SAR_ERR_BOUNDS. */
int sar_sync_status(sar_model* m);

/* ---- paged KV cache ---------------------------------------------------- */

/* One device arena for K and one for V, each laid out
 * [n_layers][num_pages][n_kv_heads][page_size][head_dim] in the model's
 * storage type, zeroed.
 * page_size must be 16, 32 or 64 tokens. */
int sar_kv_create(const sar_model* m, int32_t page_size, int32_t num_pages, sar_kv** out);

/* Device address of layer `layer`'s K (kind 0) or V (kind 1) pages, so that a
 * caller can inject cache state (e.g. a recorded or synthetic history). */
int sar_kv_layer_ptr(sar_kv* kv, int32_t layer, int32_t kind, void** out);

int sar_kv_destroy(sar_kv* kv);

/* ---- one hybrid step --------------------------------------------------- */

/* A prefill chunk: prompt positions [start_pos, start_pos+len) of request
 * `req`.  block_table (host int32[n_blocks]) lists the request's pages in
 * position order and must cover positions [0, start_pos+len). */
typedef struct sar_prefill {
  int32_t req;
  int32_t start_pos;
  int32_t len;
  const int32_t* block_table;
  int32_t n_blocks;
} sar_prefill;

/* A decode: ctx_len tokens are already cached; the new token sits at position
 * ctx_len, is appended at slot ctx_len and attends to ctx_len+1 keys.
 * block_table must cover positions [0, ctx_len]. */
typedef struct sar_decode {
  int32_t req;
  int32_t ctx_len;
  const int32_t* block_table;
  int32_t n_blocks;
} sar_decode;

enum { SAR_IN_HIDDEN = 0, SAR_IN_TOKENS = 1 };

/* Prefill chunks followed by n_decode decodes -- the batch Algorithm 3
 * builds (Sarathi-Serve digest, section 3 flowchart: the ongoing prompt's
 * chunk, then the first chunks of newly admitted requests, then decodes).
 * The chunks are `prefill` (when has_prefill) and then more_prefill[0 ..
 * n_more_prefill), each of a different request; their rows are stacked in
 * that order ([0, Lp) with Lp the sum of their lengths), then the decode
 * rows [Lp, Lp+n_decode). */
typedef struct sar_batch {
  int32_t has_prefill;
  sar_prefill prefill;
  int32_t n_decode;
  const sar_decode* decode; /* host array [n_decode] */
  int32_t in_kind;          /* SAR_IN_HIDDEN or SAR_IN_TOKENS */
  int32_t n_more_prefill;   /* further chunks (0 = at most the one above) */
  const sar_prefill* more_prefill; /* host array [n_more_prefill] */
} sar_batch;

/* Runs every layer over the stacked rows M = Lp + n_decode and then the head.
 * A request may appear in at most one chunk or decode of a batch.
 * hidden_out and logits_out must be 16-byte aligned, bf16 `in` 8-byte aligned
 * (else SAR_ERR_INVALID_ARG before any launch).
 *   in         device: bf16 [M, hidden] (SAR_IN_HIDDEN) or int32 [M] token ids
 *   hidden_out device fp32 [M, hidden]: last layer's residual stream (before
 *              the final norm); may be NULL
 *   logits_out device fp32 [R, vocab], R = chunks + n_decode: logits of
 *              every chunk's last row (in chunk order) then of every decode
 *              row; may be NULL (head skipped); must be NULL when vocab = 0
 *   layer_out  device fp32 [n_layers, M, hidden]: every layer's output; may be NULL
 * New K/V of all rows are written into `kv`.  Asynchronous on `stream`; the
 * host block tables are consumed before the call returns. */
int sar_step(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out,
             float* logits_out, void* layer_out, void* stream);

/* Same step with HOST buffers (in, hidden_out, logits_out, layer_out as
 * above, each in host memory, NULL where unused).  Copies inputs to the
 * device and results back on `stream` and returns once they are in host
 * memory.  Pinned host memory makes the copies asynchronous to the host. */
int sar_step_host(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out,
                  float* logits_out, void* layer_out, void* stream);

/* ---- one step as a CUDA graph ------------------------------------------ */

/* Captures the step of batch `b` into a CUDA graph (the pages batch steps
 * with CUDA graphs to cut launch overhead, SARATHI technique write-up,
 * section 3.3).  The graph keeps its own device copy of the step's metadata
 * (positions, slots, block tables, the decode and chunk work plans) and its
 * own decode split partials; it reads `in` and writes hidden_out /
 * logits_out / layer_out at the addresses given here (device buffers, as for
 * sar_step; hidden_out may be NULL).  Nothing runs on the GPU but the
 * metadata copy: launch the graph to run the step.  Returns any error
 * sar_step would return for `b`, before capturing. */
int sar_graph_create(sar_model* m, sar_kv* kv, const sar_batch* b, const void* in, void* hidden_out,
                     float* logits_out, void* layer_out, void* stream, sar_graph** out);

/* Points the graph at another batch whose plan has the same shape (the same
 * row, chunk-tile, decode-item, split and block-table counts, so the same
 * grids and metadata layout), copying its metadata on `stream` ahead of the
 * next launch there; SAR_ERR_INVALID_ARG otherwise (the graph is unchanged).
 * The caller puts the batch's inputs into the captured `in` buffer. */
int sar_graph_update(sar_graph* g, const sar_batch* b, void* stream);

/* Runs the captured step on `stream`. */
int sar_graph_launch(sar_graph* g, void* stream);

/* The captured step with HOST buffers: copies `in` (host, the captured input's
 * size and kind) into the captured input buffer, runs the graph, copies the
 * captured logits (R x vocab fp32) and/or hidden rows (M x hidden fp32) to the
 * host buffers that are not NULL, and returns once they are in host memory.
 * Each output requested must have been captured (non-NULL at create time).
 * Pinned host memory makes the copies asynchronous to the host. */
int sar_graph_launch_host(sar_graph* g, const void* in, float* logits_out, float* hidden_out, void* stream);

/* The captured step with HOST buffers, sampled greedily on the device: copies
 * `in` as sar_graph_launch_host does, runs the graph, picks each captured
 * logits row's argmax (as sar_sample_greedy: lowest index on ties) into the
 * graph's own device array and copies the R token ids to `tokens_out` (host
 * int32 [R], the rows of sar_batch's logits order); returns once they are in
 * host memory.  The logits must have been captured.  This is a serving step's
 * round trip: the host needs the next tokens, not the logits. */
int sar_graph_launch_host_tokens(sar_graph* g, const void* in, int32_t* tokens_out, void* stream);

/* sar_graph_launch_host_tokens without the wait, for a serving loop that
 * plans and stages the next step while this one runs: the copy of `in` goes
 * on the graph's own copy stream (created on first use) once the graph's
 * previous enqueued step has ended, and can therefore run while other work
 * computes on `stream`; the captured step waits for it on `stream`, then the
 * greedy picks and their copy into `tokens_out` follow there.  Returns once
 * everything is enqueued.  `in` must stay unchanged and `tokens_out` unread
 * until sar_graph_wait(g) returns.  Steps enqueued on one stream run in
 * order; a sar_graph_update of another graph may be called in between (its
 * metadata copy is ordered on the stream it is given). */
int sar_graph_enqueue_host_tokens(sar_graph* g, const void* in, int32_t* tokens_out, void* stream);

/* Waits for the graph's last sar_graph_enqueue_host_tokens step: its token
 * ids are then in host memory.  Returns at once if none was enqueued. */
int sar_graph_wait(sar_graph* g);

int sar_graph_destroy(sar_graph* g);

/* Greedy sampling: tokens_out[r] = argmax_v logits[r, v] (lowest index on
 * ties), device fp32 [rows, vocab] -> device int32 [rows]. */
int sar_sample_greedy(sar_model* m, const float* logits, int32_t rows, int32_t* tokens_out,
                      void* stream);

/* ---- decode attention without allocation ------------------------------- */

/* Paged decode attention that allocates nothing.  The paper has no
 * counterpart to this entry point.  It is for callers that cannot call
 * cudaMalloc: code that runs while another component captures a CUDA graph on
 * the same stream, runtimes that hand out a fixed memory budget up front and
 * own every allocation, hosts that forbid allocation on the serving path.
 * It computes what the decode rows of sar_step compute for a model without a
 * sliding window -- every decode's query heads against its own paged history
 * of all ctx_lens[b] + 1 keys (it takes no window argument) -- but
 * plans the key splits on the device and keeps the split partials in one
 * file-scope device array of 8 MiB, so it needs no workspace and no pinned
 * staging buffer.  Every GPU that loads the library holds that array until
 * the process exits.
 *   q            device rows of the storage type, row b at q + b*q_stride
 *                (n_q_heads * head_dim values, already rotated)
 *   k_pages/v_pages  device pages of one layer, [num_pages][n_kv_heads][page_size][head_dim]
 *   ctx_lens     device int32 [n_decode]; max_ctx (host) bounds them
 *   block_tables device int32 [n_decode][bt_stride], row b = decode b's pages in order
 *   out          device rows of the storage type, row b at out + b*out_stride
 *   storage      SAR_STORAGE_F16 or SAR_STORAGE_BF16 (pages and out; q too,
 *                unless SAR_Q_F32 is OR-ed in: then q rows are fp32 and
 *                q_stride counts floats, as the step's own fp32 queries are)
 *   err_flag     device int32[4] or NULL: first device-side failure (code, site, detail).
 *                A decode whose ctx_lens[b] + 1 exceeds what max_ctx planned
 *                for is skipped and its out rows are left as they were; only
 *                err_flag (SAR_ERR_BOUNDS) tells, so pass one.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  Calls
 * share the array and keep its last contents (every partial is written before
 * it is read, so nothing needs clearing); two calls whose work overlaps on the
 * GPU race on it.  Contexts are split into ranges of `split` keys, the
 * smallest power of two in [256, 4096] for which the partials,
 * n_decode * ceil((max_ctx+1)/split) * n_q_heads * (head_dim+2) * 4 bytes, fit
 * in 8 MiB; when none does the call returns SAR_ERR_INVALID_ARG before any
 * launch. */
enum { SAR_Q_F32 = 0x100 };
int sar_decode_attention_noalloc(const void* q, int32_t q_stride, const void* k_pages,
                                 const void* v_pages, int32_t num_pages, int32_t page_size,
                                 int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t n_decode, const int32_t* ctx_lens, int32_t max_ctx,
                                 const int32_t* block_tables, int32_t bt_stride, void* out,
                                 int32_t out_stride, int32_t storage, int32_t* err_flag,
                                 void* stream);

/* ---- per-kernel timing (CUDA events on the step's stream) -------------- */

enum {
  SAR_K_EMBED = 0,
  SAR_K_RMSNORM,
  SAR_K_GEMM_QKV,
  SAR_K_ROPE_APPEND,
  SAR_K_CHUNK_ATTN,
  SAR_K_DECODE_ATTN,
  SAR_K_GEMM_O,
  SAR_K_GEMM_GATEUP,
  SAR_K_GEMM_DOWN,
  SAR_K_HEAD_NORM,
  SAR_K_GEMM_HEAD,
  SAR_K_DECODE_COMBINE, /* the merge of the decodes' key-range partials */
  SAR_K_COUNT
};

/* When on, sar_step records an event pair around every kernel group. */
int sar_profile_enable(sar_model* m, int32_t on);

/* When on, a step that has both prefill chunks and decodes runs the chunk
 * attention on a second (high-priority) stream concurrently with the decode
 * attention, forked after the QKV projection and joined before the O
 * projection by events -- the pages' two-stream split of the hybrid batch
 * (SARATHI technique write-up, section 3.3).  Results are identical either
 * way (the two kernels write disjoint rows).  Off by default; ignored while
 * profiling.  Creates the stream and events on first use. */
int sar_model_set_overlap(sar_model* m, int32_t on);

/* When on, a step whose chunk-attention query tiles x heads would leave SMs
 * idle (a short chunk deep into a long prompt) shares each tile's keys out over
 * up to four CTAs and merges their partial results (the split form decode
 * attention uses for long contexts).  Off by default: the merged sums are
 * rounded in another order than an unsplit tile's, so a chunked prefill and a
 * one-shot prefill of the same prompt no longer agree as closely (over the
 * 60-layer Yi-34B shape: relative L2 6e-3 instead of below 1e-3). */
int sar_model_set_chunk_split(sar_model* m, int32_t on);

/* Synchronises, then returns per kind the accumulated milliseconds and the
 * number of timed launches since the last reset, and resets them. */
int sar_profile_read(sar_model* m, double* ms, int64_t* launches, int32_t n_kinds);

/* ---- stall-free scheduler (host only) ---------------------------------- */

/* tau: token budget, rounded down to a multiple of `tile` (must be >= tile).
 * page_size/num_pages: the KV pool the scheduler hands pages from.
 * max_batch: most requests holding pages at once.
 * max_chunks: most prefill chunks in one batch; 0 = no cap (Algorithm 3's
 * admission loop: after the ongoing prompt's chunk, waiting requests are
 * admitted first come first served while they can be allocated and the
 * budget lasts); 1 = one chunk per batch, a new request only when no prompt
 * is unfinished. */
typedef struct sar_sched_cfg {
  int32_t tau;
  int32_t tile;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_batch;
  int32_t max_chunks;
} sar_sched_cfg;

int sar_sched_create(const sar_sched_cfg* cfg, sar_sched** out);

/* Queues a request.  prompt_tokens (host int32[prompt_len]) may be NULL; when
 * every queued request has them, sar_sched_next also returns input ids. */
int sar_sched_add(sar_sched* s, int32_t req, double arrival, int32_t prompt_len,
                  int32_t output_len, const int32_t* prompt_tokens);

/* Builds the next batch at time `now` (requests with arrival <= now are
 * eligible): all running decodes, then the unfinished prompt's next chunk
 * (at most one prompt is unfinished at any time), then new requests' first
 * chunks while the budget lasts (see max_chunks).  The first chunk is
 * out->prefill, the others out->more_prefill.  `out`
 * points into scheduler-owned memory valid until the next call.  tokens_out
 * (nullable) receives a pointer to M input ids, or NULL if unknown.
 * Returns SAR_ERR_NO_PAGES if a decode needs a page and none is free. */
int sar_sched_next(sar_sched* s, double now, sar_batch* out, const int32_t** tokens_out);

/* Advances state with the sampled token of every logits row of the last
 * batch (each chunk's last row in chunk order, then decodes).  n_finished (nullable)
 * receives how many requests completed; their pages are returned. */
int sar_sched_commit(sar_sched* s, const int32_t* sampled, int32_t n_sampled,
                     int32_t* n_finished);

/* Queue sizes: waiting, running, finished, free pages. */
int sar_sched_stats(const sar_sched* s, int32_t* waiting, int32_t* running, int32_t* finished,
                    int32_t* free_pages);

int sar_sched_destroy(sar_sched* s);

#ifdef __cplusplus
}
#endif

#endif /* SAR_H */
