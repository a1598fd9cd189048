// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "../../include/sar.h"
#include "../../include/sar_ops.h"

// Returns the status of `x` from the enclosing function unless it is SAR_OK.
#define SAR_TRY(x)                  \
  do {                              \
    int _rc = (x);                  \
    if (_rc != SAR_OK) return _rc;  \
  } while (0)

namespace sar {

// ---- errors / bookkeeping (api.cpp) ----------------------------------------
int set_error(int code, const std::string& msg);
int cuda_error(cudaError_t e, const char* what);
void count_launches(int64_t n);
int num_sms();
// Raises kernel `fn`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device): the attribute belongs to the device's
// context, so a process that drives several devices (or threads that race
// a first call) sets it on each.  Thread-safe.
int ensure_smem_attr(const void* fn, int bytes, const char* what);
// Resident clusters of `fn` for the launch shape `qc` (cluster attribute
// included) on the current device, computed once per (kernel, cluster size,
// device).  Thread-safe.
int max_active_clusters(const void* fn, const cudaLaunchConfig_t& qc, int cl, int* out, const char* what);

// Kernels of a step are launched with programmatic stream serialisation: the
// next kernel's CTAs may become resident while the previous kernel drains and
// run their set-up (barriers, tensor memory, descriptor prefetch), then wait
// in pdl_wait() until the previous kernel has completed.  SAR_PDL=0 in the
// environment launches them normally.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- GEMM (gemm_tc.cu) -----------------------------------------------------

// Encodes a 2D 16-bit (storage type) tensor map over row-major [rows, cols]
// with a 64-column x box_rows box and 128-byte swizzle.
int make_tmap_16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 int storage);

struct GemmCfg {
  int swap = 0;     // weights on the MMA M side
  int msub = 1;     // 128-row A sub-tiles per tile (non-swap only)
  int bn = 256;     // MMA N extent: weight rows (non-swap) or token rows (swap)
  int m_tiles = 0;  // tiles along the token dimension
  int n_tiles = 0;  // tiles along the weight-row dimension
  int stages = 0;
  int smem = 0;
  int grid = 0;
  // box rows the two tensor maps must be encoded with
  int a_box_rows = 128;
  int b_box_rows = 256;
  int splits = 1;        // K ranges per tile (in-place fp32 residual epilogue only)
  int kb_per_split = 0;  // 64-wide K slabs per range
  int pair = 0;          // 2-CTA tiles: M = 256 MMAs over a CTA pair (cl = 2)
  int stage_bytes = 0;   // shared memory of one pipeline stage (per CTA)
  int per_sm = 1;        // CTAs resident per SM (2: swap tiling, half the stages each)
  int cl = 1;            // CTAs per cluster: 2 for a CTA pair, else 1
  int m_groups = 0;      // token-tile groups of cl tiles
  int sk = 0;            // stream-K: equal K-slab shares over all resident clusters (residual epilogue)
  int tma_out = 0;       // the in-place residual epilogue adds its tile through TMA reductions (non-swap)
};

// Box rows of the weight maps a model keeps per matrix (index i: 32 << i); the
// GEMM reads the weight tile through the map whose box is bn / cl rows (a pair CTA: its half)
// (swap tiling: 128).
constexpr int kWeightBoxes = 4;
inline int weight_box_index(const GemmCfg& c) {
  const int rows = c.swap ? c.a_box_rows : c.b_box_rows;
  return rows == 32 ? 0 : rows == 64 ? 1 : rows == 128 ? 2 : 3;
}

// Epilogue of the fused QKV projection (internal, after the public SAR_EPI_*):
// C (fp32 [M, (qh + 2 kvh) * hd]) receives q and k rotated at their rows'
// positions and v as projected; k and v are also rounded once to the storage
// type and written into their rows' page slots.
constexpr int kEpiRope = 4;
struct RopeEpi {
  const int32_t* pos = nullptr;   // [M] absolute position of each row (unused: the table holds it)
  const int32_t* slot = nullptr;  // [M] page * page_size + offset
  // (cos, sin) of pos * theta_i, frequency-major so that consecutive rows are
  // adjacent: the float4 (cos, sin of frequency 2i; cos, sin of 2i + 1) of
  // row r is at cs4(i * cs_ld + r), cs_ld >= the step's rows
  const float2* cs = nullptr;
  int cs_ld = 0;
  void* k_cache = nullptr;        // layer base [num_pages][kvh][page_size][hd], storage type
  void* v_cache = nullptr;
  // the layer's pages as tensor maps (16-row x 64-column boxes, make_kv_tmap):
  // head_dim 128 k/v rows of page-aligned 16-row runs are stored through them
  const CUtensorMap* kmap = nullptr;
  const CUtensorMap* vmap = nullptr;
  int qh = 0, kvh = 0, hd = 0, page_size = 0, num_pages = 0;
};

// Picks a tiling for C[M, .] = A[M, K] . W[N, K]^T (variant = SAR_GEMM_*).
// Returns SAR_OK or SAR_ERR_UNSUPPORTED.
// in_place: the residual epilogue writes into its own residual (C == R), which
// allows split-K with atomic fp32 adds.
int gemm_config(int M, int N, int K, int epi, int variant, GemmCfg* cfg, bool in_place = false);

// Launches with maps already encoded: `act_map` over the activations (rows M),
// `w_map` over the weights; which one is the MMA's A operand depends on cfg.swap.
// `rope` is required for (and only read by) kEpiRope.
int gemm_launch(const GemmCfg& cfg, const CUtensorMap& act_map, const CUtensorMap& w_map, int M,
                int N, int K, int epi, int storage, void* c, const void* residual, int* err,
                cudaStream_t s, const RopeEpi* rope = nullptr);

// ---- elementwise kernels (elementwise.cu) ----------------------------------
// x: fp32 residual rows; y: storage-type rows; row_index (optional) gathers rows.
// zero (optional): zero_n floats to clear, split over the blocks.
// One-thread kernel whose barrier completes only with two arrivals; it
// arrives `arrivals` times and waits with a limit of limit_ns.
int launch_wait_check(uint64_t limit_ns, int arrivals, int* err, cudaStream_t s);
int launch_rmsnorm(const float* x, const float* gain, void* y, int rows, int hidden, float eps,
                   const int32_t* row_index, int storage, cudaStream_t s, float* zero = nullptr,
                   size_t zero_n = 0);
// The step's first kernel: stacked input rows (bf16 hidden rows, or token ids
// looked up in `table`) into the fp32 residual stream h and, normalised with
// `gain`, into y (storage type).  zero (optional): zero_n floats to clear.
// cs (optional): the step's rotary table (the RopeEpi layout, row stride cs_ld) of (cos, sin) of
// pos[r] * inv_freq[i], shared by every layer's QKV epilogue.
int launch_input_norm(int in_kind, const void* in, const void* table, int vocab, float* h, const float* gain,
                      void* y, int rows, int hidden, float eps, int storage, int* err, cudaStream_t s,
                      float* zero = nullptr, size_t zero_n = 0, const int32_t* pos = nullptr,
                      const double* inv_freq = nullptr, float2* cs = nullptr, int half_d = 0, int cs_ld = 0,
                      float* zero2 = nullptr, size_t zero2_n = 0);
// Small-row steps, whose QKV and gate/up projections accumulate split-K into
// fp32: the rotary embedding + KV-page append over qkv rows [rows][ld] in
// place, and silu(gate)*up from the packed fp32 gate/up rows [rows][2F].
int launch_rope_append(float* qkv, int ld, int rows, const RopeEpi& rp, int storage, int* err, cudaStream_t s);
int launch_swiglu_finish(const float* gu, void* act, int rows, int F, int storage, cudaStream_t s);
int launch_embed(const int32_t* tokens, const void* table, float* out, int rows, int hidden, int vocab,
                 int storage, int* err, cudaStream_t s);
int launch_bf16_to_f32(const void* src, float* dst, size_t n, cudaStream_t s);
// bf16 rows -> storage type; interleave=1 places row r of gate (up=0) or up
// (up=1) into the 64-row-block gate/up packing.
int launch_convert_rows(const void* src, void* dst, int rows, int cols, int interleave, int up, int storage,
                        cudaStream_t s);
int launch_argmax(const float* logits, int rows, int vocab, int32_t* out, cudaStream_t s);

// ---- attention (attn_decode.cu, attn_chunk.cu) -----------------------------
struct DecodeAttnArgs {
  const void* qkv;           // decode rows start here; row stride ld (storage type)
  const float* q32 = nullptr;  // when set: fp32 query rows (row stride ld32) used instead of qkv
  int ld32 = 0;
  void* out;                 // decode rows of the attention output; row stride ld_out
  const void* k_cache;
  const void* v_cache;
  const int32_t* items;      // [n_items][4]: decode b, key_begin, key_end, part (-1 = final)
  const int32_t* nkeys;      // [n_decode] keys each decode attends to (ctx + 1)
  const int32_t* bt_off;     // [n_decode] offset into bt
  const int32_t* bt_len;     // [n_decode]
  const int32_t* bt;         // flattened block tables
  const int32_t* parts_begin;  // [n_decode] first partial index (or -1)
  const int32_t* parts_count;  // [n_decode]
  float* partials;           // [n_parts][qh][d + 2]
  int n_items, n_decode, ld, ld_out, qh, kvh, d, page_size, num_pages, storage;
  int* err;
  // sliding window (planned items only): decode b sees keys [nkeys[b] - window, nkeys[b]); 0 = all
  int window = 0;
  // device-computed work split (used by the entry point that allocates nothing)
  const int32_t* ctx_lens = nullptr;  // [n_decode]
  int split_keys = 0, max_splits = 0, bt_stride = 0;
  // the partials' merge is launched separately (launch_decode_combine), so
  // that another kernel can run between the two
  bool defer_combine = false;
};
// Tensor map over one layer's K or V pages viewed as rows of head_dim values
// (one row per page x head x slot), 16-row x 64-column boxes, 128-byte swizzle.
int make_kv_tmap(CUtensorMap* map, const void* pages, int num_pages, int kvh, int page_size, int head_dim,
                 int storage);
int launch_decode_attention(const DecodeAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                            cudaStream_t s);
// The merge of a deferred launch (nothing to do when there are no partials).
int launch_decode_combine(const DecodeAttnArgs& a, cudaStream_t s);

struct ChunkAttnArgs {
  const float* q32;          // chunk query rows in fp32 (batch rows); row stride ld32
  int ld32;
  void* out;                 // attention rows (batch rows); row stride ld_out
  const void* k_cache;
  const void* v_cache;
  const int32_t* bt;         // the chunks' block tables, concatenated
  // [n_tiles][8] query tiles, one CTA each, in launch order: first batch row,
  // first position, rows (<= the kernel's tile rows), block-table offset into
  // bt, block-table length, first and end 128-key block, partial slot (-1: the
  // tile's whole key range, written to out); a tile's rows are consecutive
  // positions of one prompt, whose keys [0, last position] sit in its block
  // table.  The warp-MMA kernel reads the first five only.
  const int32_t* tiles;
  int n_tiles;
  // key-range splits (tcgen05 kernel): unnormalised partials
  // [slot][128 rows][qh][head_dim + 4] (O, then the row's maximum and sum),
  // and [n_comb][4] merges {first batch row, rows, first slot, slots}
  float* partials = nullptr;
  const int32_t* comb = nullptr;
  int n_comb = 0;
  int ld, ld_out, qh, kvh, d, page_size, num_pages, storage;
  int* err;
  int window = 0;            // the row at position p sees keys (p - window, p]; 0 = all of [0, p]
  // tcgen05 kernel launched right behind the decode attention kernel, whose
  // output it does not read: it starts without waiting for that kernel (its
  // inputs were complete before that kernel released its dependents) and its
  // last CTA waits for it before exiting, so the kernels after it see both
  int wait_at_end = 0;
  // tcgen05 kernel: the tile table lists tile pairs (entries 2i, 2i + 1: two
  // query tiles of one prompt's chunk over the same key blocks, the second
  // possibly with 0 rows), one CTA per pair and head; full causal attention
  // and whole key ranges only
  int dual = 0;
};
// Query rows per tile: the warp-MMA kernel (attn_chunk.cu) and the tcgen05 one.
constexpr int kChunkTileRows = 64;
constexpr int kChunkTileRowsTc = 128;
int launch_chunk_attention(const ChunkAttnArgs& a, cudaStream_t s);
// The same on the tcgen05 tensor cores (attn_chunk_tc.cu) for head_dim 128 and
// pages of a multiple of 16 keys, reading the pages through the per-layer
// tensor maps of the KV cache (16-key x 64-dim boxes).
bool chunk_attention_tc_supported(const ChunkAttnArgs& a);
int launch_chunk_attention_tc(const ChunkAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              cudaStream_t s);

}  // namespace sar
