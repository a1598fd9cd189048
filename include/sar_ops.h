/*
 * sar_ops.h -- single-kernel entry points of the hybrid step, for per-kernel
 * parity tests and for the tile-quantisation sweep.
 *
 * The GEMM is the "one GEMM per weight over all [Lp+Bd, H] rows" of
 * "SARATHI: Efficient LLM Inference by Piggybacking Decodes with Chunked
 * Prefills" (reading notes, part 2 section 3).  Its row-tile choice is what the
 * same notes' part 3 section 3 (tile quantisation: 257 rows need a third
 * 128-row block) and the Sarathi-Serve digest (section 2, Q2 item 3: 257 vs
 * 256 tokens costs +32% prefill time) are about; the variants below let a
 * caller pick the tiling and measure it.
 */
#ifndef SAR_OPS_H
#define SAR_OPS_H

#include <stdint.h>

#include "sar.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogues applied to the fp32 accumulator D = A . W^T. */
enum {
  SAR_EPI_STORE = 0,    /* C [M, N] in the storage type = D                          */
  SAR_EPI_RESIDUAL = 1, /* C fp32 [M, N] = D + R (R fp32 [M, N]; R may equal C)      */
  SAR_EPI_SWIGLU = 2,   /* W is gate/up interleaved in 64-row blocks, [2F, K]; C [M, F]
                           in the storage type = silu(D_gate) * D_up                 */
  SAR_EPI_F32 = 3       /* C fp32 [M, N] = D                                         */
};

/* Tilings.  All run tcgen05 MMAs (16-bit x 16-bit -> fp32 in tensor memory) fed by
 * TMA from 128-byte-swizzled shared memory, in a persistent kernel. */
enum {
  SAR_GEMM_AUTO = 0,  /* the library's choice for (M, N, K)                        */
  SAR_GEMM_M128_N128 = 1, /* 128 token rows x 128 weight rows per tile              */
  SAR_GEMM_M128_N256 = 2, /* 128 token rows x 256 weight rows per tile              */
  SAR_GEMM_SWAP = 3,      /* weights on the MMA's M side (128 rows), tokens on its N
                             side padded to 16 (M <= 256): no 128-row quantisation */
  SAR_GEMM_M256_N128 = 4, /* 256 token rows (two 128-row MMAs sharing one weight
                             tile) x 128 weight rows per tile                        */
  SAR_GEMM_PAIR_N256 = 5, /* 256 token rows x 256 weight rows per tile over a pair of
                             CTAs (2-CTA cluster): one M = 256 MMA reads each CTA's
                             128 token rows and half of the weight rows, so each SM
                             loads half the weight tile                             */
  SAR_GEMM_PAIR_N128 = 6, /* the same with 128 weight rows per tile                 */
  SAR_GEMM_PAIR_N192 = 7, /* the same with 192 weight rows per tile (not for the
                             SwiGLU epilogue, whose gate/up blocks are 128 wide)    */
  /* Optional flag for the swap tiling with at most 128 token rows: two CTAs
   * per SM, each with half the pipeline, so twice as many weight slabs are in
   * flight per SM (the memory-bound regime). */
  SAR_GEMM_TWO_CTAS = 0x1000,
  /* Optional flag for the in-place fp32 residual epilogue (non-swap tilings):
   * stream-K.  Every resident CTA (pair) takes an equal, contiguous share of
   * all tiles' 64-wide K slabs, so a few tiles spread over all SMs instead of
   * leaving a partial wave; a share that covers part of a tile's K range adds
   * its partial sum into C atomically (as split-K does).  Each token group's
   * weight slabs are shared out separately, so the groups read a weight slab
   * at the same time (once from HBM).  AUTO does not take it. */
  SAR_GEMM_STREAM_K = 0x2000
};

/* C = epilogue(A . W^T).  A [M, K], W [N, K] in the storage type `storage`
 * (SAR_STORAGE_F16 or SAR_STORAGE_BF16; device, row-major, 16-byte aligned,
 * K a multiple of 64, N a multiple of 64, M >= 1).  For SAR_EPI_SWIGLU, N is
 * 2F (the packed rows) and C has F columns.  Returns SAR_ERR_UNSUPPORTED for
 * shapes a variant cannot take. */
int sar_op_gemm(const void* a, const void* w, void* c, const void* residual, int32_t M, int32_t N,
                int32_t K, int32_t epilogue, int32_t variant, int32_t storage, void* stream);

/* Device-side status of the single-kernel entry points (sar_op_gemm,
 * sar_op_wait_check) on the current device.  Their kernels record the first
 * failure -- a bounded wait that gave up (SAR_ERR_TIMEOUT) or an index out of
 * bounds (SAR_ERR_BOUNDS) -- in one record per device instead of trapping.
 * This call synchronises the device, reads the record, clears it and returns
 * its code (SAR_OK if none); sar_last_error() then names the kernel site and
 * a detail.  The record is shared by every stream and thread on the device. */
int sar_op_sync_status(void);

/* Exercises the bounded wait that every pipelined kernel uses (no counterpart
 * in the pages; the bound keeps a stuck pipeline from holding the GPU).  One
 * thread initialises a shared-memory barrier that needs two arrivals, arrives
 * `arrivals` times (0..2) and waits for it with a limit of limit_ns
 * nanoseconds (> 0).  With two arrivals the wait completes; with fewer it
 * runs out after about limit_ns, the kernel records SAR_ERR_TIMEOUT for
 * sar_op_sync_status() and returns, and the context stays usable.  Async on
 * `stream`. */
int sar_op_wait_check(int64_t limit_ns, int32_t arrivals, void* stream);

/* y = x * rsqrt(mean(x^2) + eps) * gain per row: x fp32 [rows, hidden] (the
 * residual stream), gain fp32 [hidden], y [rows, hidden] in `storage`. */
int sar_op_rmsnorm(const void* x, const void* gain, void* y, int32_t rows, int32_t hidden,
                   float eps, int32_t storage, void* stream);

/* Device address of a step workspace buffer, valid until sar_model_destroy;
 * after a step on a one-layer model it holds that layer's intermediates.
 *   0: normed rows     [max_tokens, hidden] (storage type)
 *   1: rotary table    fp32, (cos, sin) of each row's position times theta_i:
 *                      for row r and frequency i, at float index
 *                      4 * ((i / 2) * max_tokens + r) + 2 * (i % 2) (frequency
 *                      pairs major, so a warp's 32 rows read 512 contiguous bytes)
 *   2: attention rows  [max_tokens, n_q_heads * head_dim] (storage type)
 *   3: SwiGLU rows     [max_tokens, ffn] (storage type)
 *   4: residual stream fp32 [max_tokens, hidden] (when the step had no hidden_out)
 *   5: q|k|v rows      fp32 [max_tokens, (n_q_heads + 2 n_kv_heads) * head_dim]
 *                      (the projection with q and k rotated; k and v are
 *                      also in the pages, rounded to the storage type; for
 *                      head_dim 128 and more than 32 rows -- a QKV projection
 *                      on 128-row token tiles -- only q is kept in fp32; the
 *                      attention kernels read k and v from the pages) */
int sar_model_debug_buffer(sar_model* m, int32_t which, void** out);

/* The step planner on the host alone (no GPU, no model): plans batch `b` as
 * sar_step would for a model of `dims` (with chunk_split as set by
 * sar_model_set_chunk_split), a cache of num_pages pages of page_size tokens
 * and a device of `sms` SMs (sar_step plans for the current device's), with
 * the same validation and errors.  layout (int32[25])
 * receives M, Lp, Bd, R, decode work items, decode partials, chunk tiles,
 * rows per chunk tile, then the offsets (int32 elements) of the metadata
 * block's arrays -- row positions, row page slots, chunk block tables,
 * decode key counts, decode block-table offsets, decode block-table lengths,
 * first partial, partial count, work items [4 each: decode, first key, end
 * key, partial or -1], decode block tables, logits rows, chunk tiles [8 each:
 * first batch row, first position, rows, block-table offset, block-table
 * length, first and end 128-key block, key-range partial slot or -1] -- its
 * total length, then the chunk key-range merges, their partial slots and the
 * merges' offset [4 each: first batch row, rows, first slot, slots], then 1
 * when the chunk tiles are listed in pairs (entries 2i and 2i + 1: two query
 * tiles of one chunk, the second possibly of 0 rows, one CTA per pair and
 * head), else 0.  The
 * block itself (what the step ships to the device) is copied to meta
 * (int32[meta_cap], may be NULL) and its length to *meta_n. */
int sar_plan_inspect(const sar_dims* dims, int32_t page_size, int32_t num_pages, int32_t sms,
                     int32_t chunk_split, const sar_batch* b, int32_t* layout, int32_t* meta, int64_t meta_cap,
                     int64_t* meta_n);

#ifdef __cplusplus
}
#endif

#endif /* SAR_OPS_H */
