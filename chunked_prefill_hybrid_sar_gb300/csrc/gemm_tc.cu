// Projection / FFN / LM-head GEMM on the 5th-generation tensor cores.
//
// C = epilogue(A . W^T) with A = activations [M, K] and W = weights [N, K],
// both of the 16-bit storage type (fp16 by default, or bf16) and K-major.  This is the "one GEMM per weight over the stacked
// [Lp+Bd, H] rows" of the hybrid step ("SARATHI: Efficient LLM Inference by
// Piggybacking Decodes with Chunked Prefills", reading notes, part 2 section 3).
//
// Structure (persistent, one CTA per SM, 192 threads):
//   warp 0       TMA producer: 64-wide K slabs of the A and B tiles into a ring
//                of shared-memory stages (128-byte swizzle), mbarrier tx counts.
//   warp 1       allocates tensor memory; lane 0 issues tcgen05.mma
//                (kind::f16, 16-bit x 16-bit of one type -> fp32, M = 128 or 256, N = bn, K = 16) and
//                tcgen05.commit's each stage back to the producer.
//   warps 2..5   epilogue: tcgen05.ld of the fp32 accumulator (each warp owns
//                the 32 TMEM lanes of its warp-id % 4), fused epilogue, global
//                stores.  Two accumulators alternate so the epilogue of one
//                tile overlaps the MMAs of the next.
//
// CTA pairs (cta_group::2): the two CTAs of a 2-CTA cluster take two
// consecutive token tiles of one 256-row weight tile; each loads its own 128
// token rows and half of the weight rows, and the leader issues one M = 256
// MMA over both CTAs' shared memory.  No other tiling uses a cluster, and no
// load is multicast: every CTA's TMA loads fill its own shared memory only.
//
// Epilogues: 16-bit store, fp32 store, fp32 residual add (in place, optionally
// split-K; in the non-swap tilings each warp stages 32-row boxes in swizzled
// shared memory and adds them with TMA reductions, in the swap tiling with
// atomic adds), SwiGLU over 64-row gate/up block pairs (non-swap: staged boxes
// written by TMA stores), and the
// fused rotary + KV append of the QKV projection: q and k rotated at their
// rows' positions (rotate-half pairing, dims i and i + hd/2; "maintain an
// independent position_id for each chunk", SARATHI technique write-up section
// 6.1), written in fp32, k and v rounded once and stored into their rows'
// page slots.  Tiles are head-aligned; in the swap tiling the two halves of a
// head sit in different warps and meet through shared memory.
//
// Tilings: non-swap puts 128 token rows on the MMA M side (msub = 2 stacks two
// such MMAs on one weight tile for 256-row tiles); swap puts 128 weight rows
// on the M side and the tokens (padded to 16) on the N side, so a step with
// few rows pays no 128-row quantisation.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "tc05.cuh"

namespace sar {

namespace {

constexpr int kThreads = 192;
constexpr int kBK = 64;                   // K elements per stage (128 bytes)
constexpr int kTileA = 128 * kBK * 2;     // one 128-row slab: 16 KB
constexpr int kSmemLimit = 232448;        // 227 KB of dynamic shared memory
constexpr int kSmemPerSm = 233472;        // 228 KB of shared memory per SM
constexpr int kBarBytes = 1024;           // barriers + TMEM slot (+ alignment)
constexpr int kSwapXchg = 64 * 17 * 4;    // swap-mode SwiGLU exchange buffer
constexpr int kSwapXchgRope = 128 * 17 * 4;  // swap-mode rotary exchange buffer
// K-slabs of the weight tile prefetched into L2 ahead of the shared-memory
// ring (which holds 5-8 more).  A short distance: deep prefetches queue ahead
// of the ring's own loads (the tau = 512 step took 329.4 us at 16 slabs, 326.2
// at 8, 323.7 at 1-4, 325.0 with none)
constexpr int kPrefetch = 3;
constexpr int kEpiBox = 32;               // TMA epilogue boxes: 32 rows x 128 bytes (32 fp32 or 64 16-bit columns)
constexpr int kEpiBoxBytes = kEpiBox * kEpiBox * 4;
constexpr int kEpiStage = 4 * 2 * kEpiBoxBytes;  // two boxes per epilogue warp


struct Params {
  int M, N, K;
  int bn, m_tiles, n_tiles, k_blocks, stages, stage_bytes, tmem_cols;
  int splits, kb_per_split;  // split-K: `splits` K ranges per tile (residual epilogue only)
  int sk;                    // stream-K: equal shares of every token group's (weight tile, K slab) runs (residual only)
  int cl, m_groups;          // CTAs per cluster (2: CTA pair, else 1); token-tile groups
  int tma_out;               // residual epilogue through TMA reductions (the third tensor map)
  RopeEpi rope;              // kEpiRope only
  void* c;
  const void* r;
  int* err;
};

// Work unit u of a cluster -> (token tile, weight tile, K-slab range).  The
// `cl` CTAs of a cluster (a CTA pair, or one CTA) take consecutive token tiles
// of one weight tile; token-tile groups vary fastest so clusters running at
// the same time share the weight slab in L2.
struct Unit {
  int mt, nt, kb0, kb1;
};
__device__ __forceinline__ Unit unit_of(const Params& p, int u, int rank) {
  Unit w;
  const int mg = u % p.m_groups;
  w.mt = mg * p.cl + rank;
  const int r = u / p.m_groups;
  const int sp = r % p.splits;
  w.nt = r / p.splits;
  w.kb0 = sp * p.kb_per_split;
  w.kb1 = min(p.k_blocks, w.kb0 + p.kb_per_split);
  return w;
}

// A cluster's work: units cid, cid + C, ... (split-K units), or with
// stream-K one token group's equal share of its (weight tile, K slab) runs:
// cluster c takes group g = c % G and share j = c / G of the S = n_tiles x
// k_blocks slabs, [j*S/Cg, (j+1)*S/Cg) with Cg = C / G clusters per group,
// cut at weight-tile boundaries.  Clusters j of every group walk the same
// weight slabs at the same time, so each slab leaves HBM once and the other
// groups read it from L2 (as the groups of one split-K unit do).
struct Work {
  int t, end, step, g;
};
__device__ __forceinline__ Work work_begin(const Params& p, int cid, int n_clusters) {
  Work w;
  if (p.sk) {
    const int cg = n_clusters / p.m_groups;  // clusters per token group (the rest idle)
    const int j = cid / p.m_groups;
    const long long S = (long long)p.n_tiles * p.k_blocks;
    w.g = cid % p.m_groups;
    w.t = j < cg ? (int)(S * j / cg) : 0;
    w.end = j < cg ? (int)(S * (j + 1) / cg) : 0;
    w.step = 0;
  } else {
    w.t = cid;
    w.end = p.m_groups * p.n_tiles * p.splits;
    w.step = n_clusters;
    w.g = 0;
  }
  return w;
}
__device__ __forceinline__ bool work_next(const Params& p, Work& w, int rank, Unit& un) {
  if (w.t >= w.end) return false;
  if (p.sk) {
    un.nt = w.t / p.k_blocks;
    un.mt = w.g * p.cl + rank;
    un.kb0 = w.t - un.nt * p.k_blocks;
    un.kb1 = min(p.k_blocks, un.kb0 + (w.end - w.t));
    w.t += un.kb1 - un.kb0;
    return true;
  }
  un = unit_of(p, w.t, rank);
  w.t += w.step;
  return true;
}

__device__ __forceinline__ void next_stage(int& stage, uint32_t& phase, int stages) {
  if (++stage == stages) {
    stage = 0;
    phase ^= 1u;
  }
}

// Warp-uniform wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err, int site) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, site) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

template <typename T, int EPI, bool SWAP, int MSUB, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_kp,
                   const __grid_constant__ CUtensorMap tm_vp, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int stages = p.stages;
  uint8_t* bar_area = smem + stages * p.stage_bytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* empty_bar = full_bar + stages;
  uint64_t* accf_bar = empty_bar + stages;  // [2]
  uint64_t* acce_bar = accf_bar + 2;        // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
  float* xchg = reinterpret_cast<float*>(bar_area + kBarBytes);  // swap SwiGLU only
  // TMA epilogues (non-swap): each epilogue warp's two 4 KB boxes, 1024-byte aligned
  const uint32_t epi_stage = smem_u32(bar_area + kBarBytes);
  (void)epi_stage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      // released by this CTA's MMAs (pair: by the leader's, which read both CTAs' stages)
      mbar_init(smem_u32(&empty_bar[s]), 1u);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&accf_bar[s]), 1);
      // pair: one arrival per epilogue warp of both CTAs (only the leader's is waited on)
      mbar_init(smem_u32(&acce_bar[s]), PAIR ? 8u : 128u);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish<PAIR>();
  }
  tc_fence_before();
  __syncthreads();
  if (p.cl > 1) cluster_sync();  // the pair's barriers are initialised before either CTA's loads
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int rank = p.cl > 1 ? (int)cluster_ctarank() : 0;
  const int cid = blockIdx.x / p.cl, n_clusters = gridDim.x / p.cl;
  const int acc_cols = MSUB * p.bn;
  Unit un0;
  Work w0 = work_begin(p, cid, n_clusters);

  if (warp == 0 && lane == 0 && work_next(p, w0, rank, un0)) {
    // the weights do not depend on the previous kernel: start pulling this
    // CTA's first weight slabs into L2 while that kernel drains
    const Unit& un = un0;
    const void* w_map = SWAP ? (const void*)&tm_a : (const void*)&tm_b;
    const int w_row = SWAP ? un.nt * 128 : un.nt * p.bn + (PAIR ? rank * (p.bn / 2) : 0);
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    for (int kb = un.kb0; kb < un.kb0 + kPrefetch && kb < un.kb1; ++kb) tma_prefetch_l2(w_map, kb * kBK, w_row);
  }
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Work wk = work_begin(p, cid, n_clusters);
      Unit un;
      for (bool first = true; ok && work_next(p, wk, rank, un); first = false) {
        const int mt = un.mt, nt = un.nt;
        // A rows: tokens (non-swap) or weights (swap); B rows: the other one.
        const int a_row = SWAP ? nt * 128 : mt * 128 * MSUB;
        const int b_row = SWAP ? mt * p.bn : nt * p.bn;
        // the weight tile streams from HBM: pull it into L2 kPrefetch K-slabs ahead
        // of the shared-memory ring so the ring's loads hit L2
        const void* w_map = SWAP ? (const void*)&tm_a : (const void*)&tm_b;
        // weight rows this CTA fetches: the whole tile, or its half of the pair's tile
        const int slice = PAIR ? p.bn / 2 : 0;
        const int w_row = SWAP ? a_row : b_row + rank * slice;
        // (swap tiling: one CTA per weight tile, no reuse to gain from L2;
        // the first unit's first slabs were requested before the wait above)
        if (!SWAP && !first)
          for (int kb = un.kb0; kb < un.kb0 + kPrefetch && kb < un.kb1; ++kb) tma_prefetch_l2(w_map, kb * kBK, w_row);
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!SWAP && kb + kPrefetch < un.kb1) tma_prefetch_l2(w_map, (kb + kPrefetch) * kBK, w_row);
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.err, SITE_GEMM_PRODUCER)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * p.stage_bytes;
          const uint32_t fb = smem_u32(&full_bar[stage]);
          if constexpr (PAIR) {
            // both CTAs' loads count on the leader's barrier, which the leader's MMA waits on
            const uint32_t fb_lead = cluster_addr(fb, 0);
            if (rank == 0) mbar_expect_tx(fb, 2u * (uint32_t)p.stage_bytes);
            tma_load_2d_pair(smem_u32(st), &tm_a, kb * kBK, a_row, fb_lead);
            tma_load_2d_pair(smem_u32(st + kTileA), &tm_b, kb * kBK, b_row + rank * slice, fb_lead);
            next_stage(stage, phase, stages);
            continue;
          }
          mbar_expect_tx(fb, (uint32_t)p.stage_bytes);
#pragma unroll
          for (int s = 0; s < MSUB; ++s)
            tma_load_2d(smem_u32(st + s * kTileA), &tm_a, kb * kBK, a_row + s * 128, fb);
          tma_load_2d(smem_u32(st + MSUB * kTileA), &tm_b, kb * kBK, b_row, fb);
          next_stage(stage, phase, stages);
        }
      }
      if (p.cl > 1) {
        // pair: the leader's MMAs have released the last fills, so its commits
        // arrive on no barrier of this CTA after it leaves
        for (int i = 0; i < stages && ok; ++i) {
          ok = mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.err, SITE_GEMM_PRODUCER);
          next_stage(stage, phase, stages);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // pair: the leader issues the MMAs of both CTAs
    if (lane == 0 && (!PAIR || rank == 0)) {
      const uint32_t idesc = idesc_f16kind(PAIR ? 256 : 128, p.bn, Elem<T>::kMmaFormat);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int i = 0;
      Work wk = work_begin(p, cid, n_clusters);
      Unit un;
      for (; ok && work_next(p, wk, rank, un); ++i) {
        const int acc = i & 1;
        const uint32_t accph = (uint32_t)((i >> 1) & 1);
        if (!mbar_wait(smem_u32(&acce_bar[acc]), accph ^ 1u, p.err, SITE_GEMM_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * acc_cols);
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          // the stage's descriptors are built before its wait: between two
          // MMAs this thread issues only a constant step of each descriptor
          // (the issue of an MMA is accepted at the pipe's pace, and any
          // arithmetic between two issues adds to every MMA's time)
          const uint32_t a_base = smem_u32(smem + stage * p.stage_bytes);
          uint64_t adesc[MSUB];
#pragma unroll
          for (int s = 0; s < MSUB; ++s) adesc[s] = sw128_desc(a_base + s * kTileA);
          const uint64_t bdesc = sw128_desc(a_base + MSUB * kTileA);
          const uint32_t acc0 = kb != un.kb0 ? 1u : 0u;
          if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.err, SITE_GEMM_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
            for (int s = 0; s < MSUB; ++s)
              // K step kk: 32 bytes into the 128-byte swizzled rows (address field in 16-byte units)
              mma_f16<PAIR>(d_tmem + (uint32_t)(s * p.bn), adesc[s] + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2),
                            idesc, kk != 0 ? 1u : acc0);
          }
          if (PAIR)
            mma_commit_pair(smem_u32(&empty_bar[stage]));
          else
            mma_commit(smem_u32(&empty_bar[stage]));
          next_stage(stage, phase, stages);
        }
        if (ok) {
          if (PAIR)
            mma_commit_pair(smem_u32(&accf_bar[acc]));
          else
            mma_commit(smem_u32(&accf_bar[acc]));
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int lrow = q * 32 + lane;     // accumulator lane = row of the MMA's M side
    int i = 0;
    bool alive = true;  // false once a wait gave up: loads/stores stop, barriers stay matched
    int epi_n = 0;      // TMA epilogue boxes (reductions or stores) issued by this warp
    Work wk = work_begin(p, cid, n_clusters);
    Unit un;
    for (; work_next(p, wk, rank, un); ++i) {
      const int mt = un.mt, nt = un.nt;
      // a share of a tile's K range adds into C; a whole tile writes C = D + R
      const bool partial = p.splits > 1 || un.kb0 != 0 || un.kb1 != p.k_blocks;
      (void)partial;
      const int acc = i & 1;
      const uint32_t accph = (uint32_t)((i >> 1) & 1);
      // rotary epilogue (TMA path): the tile's first (cos, sin) chunk is
      // loaded while the MMAs still run, so its L2 latency is off the epilogue.
      // On this CTA's last tile the operand stages are idle once its MMAs have
      // completed: each warp then copies its 32 rows' whole (cos, sin) table
      // (32 float4 per row, 16 KB) into them in one batch, instead of paying
      // the L2 latency once per 16-frequency chunk
      const bool last_unit = wk.t >= wk.end;
      float4 cs_next[8];
      bool cs_ready = false;
      bool cs_smem = false;
      const uint32_t cs_base = smem_u32(smem) + (uint32_t)(q * 32 * 32 * 16);
      if constexpr (EPI == kEpiRope && !SWAP) {
        const int row = mt * MSUB * 128 + lrow;
        // (a tile of v heads only rotates nothing)
        const bool rotated = (nt * p.bn) / p.rope.hd < p.rope.qh + p.rope.kvh;
        cs_smem = last_unit && rotated && p.tma_out && p.rope.hd == 128 && MSUB == 1 &&
                  4 * 32 * 32 * 16 <= p.stages * p.stage_bytes;
        if (p.tma_out && p.rope.hd == 128 && row < p.M && !cs_smem) {
          const float4* csr0 = reinterpret_cast<const float4*>(p.rope.cs) + row;
#pragma unroll
          for (int e = 0; e < 8; ++e) cs_next[e] = __ldg(csr0 + e * (size_t)p.rope.cs_ld);
          cs_ready = true;
        }
      }
      (void)cs_ready;
      if (alive) alive = warp_wait(smem_u32(&accf_bar[acc]), accph, p.err, SITE_GEMM_EPILOGUE);
      if (!alive && !(SWAP && (EPI == SAR_EPI_SWIGLU || EPI == kEpiRope))) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * acc_cols);
      if constexpr (EPI == kEpiRope && !SWAP) {
        // every MMA of this CTA has completed (and with it every stage load):
        // the stages are free for this warp's [32 float4][32 rows] table
        const int row = mt * MSUB * 128 + lrow;
        if (cs_smem && row < p.M) {
          const float4* csr0 = reinterpret_cast<const float4*>(p.rope.cs) + row;
#pragma unroll 8
          for (int e = 0; e < 32; ++e) cp_async16(cs_base + (uint32_t)((e * 32 + lane) * 16), csr0 + e * (size_t)p.rope.cs_ld, 16);
          cp_async_commit();
          cp_async_wait<0>();  // this lane reads back only its own row's entries
        }
      }

      if constexpr (!SWAP) {
#pragma unroll 1
        for (int s = 0; s < MSUB; ++s) {
          const int row = (mt * MSUB + s) * 128 + lrow;
          const bool row_ok = row < p.M;
          const uint32_t sbase = tbase + (uint32_t)(s * p.bn);
          if constexpr (EPI == kEpiRope) {
            // head-aligned tile: q and k heads rotated (dim i with i + hd/2),
            // all written in fp32 to C; k and v also rounded into their page slot
            const RopeEpi& rp = p.rope;
            const int half = rp.hd >> 1;
            float* C = reinterpret_cast<float*>(p.c);
            int page = -1, off = 0;
            bool slot_ok = false;
            const int sl = row_ok ? rp.slot[row] : -1;
            if (row_ok) {
              page = sl >= 0 ? sl / rp.page_size : -1;
              off = sl - page * rp.page_size;
              slot_ok = sl >= 0 && page < rp.num_pages;
            }
            // k/v rows by TMA store (TMA path): each half-warp's 16 rows whose
            // slots are one whole page-aligned run of 16 (a chunk's rows)
            // leave as one 16-row box per dim half; other rows (decodes, a
            // chunk's ragged edges) are stored by their threads
            const int sl_b = __shfl_sync(0xffffffffu, sl, lane & 16);
            const unsigned runs = __ballot_sync(0xffffffffu, row_ok && slot_ok && sl_b >= 0 && (sl_b & 15) == 0 &&
                                                                 sl == sl_b + (lane & 15));
            const bool run0 = (runs & 0xffffu) == 0xffffu, run1 = (runs >> 16) == 0xffffu;
            const bool in_run = (lane < 16) ? run0 : run1;
            const int pg_b0 = __shfl_sync(0xffffffffu, page, 0), of_b0 = __shfl_sync(0xffffffffu, off, 0);
            const int pg_b1 = __shfl_sync(0xffffffffu, page, 16), of_b1 = __shfl_sync(0xffffffffu, off, 16);
            bool after_kv = false;  // the last staging use was a k/v head's
            // this row's (cos, sin) pairs: pair i at csr[i * cs_ld] (rows adjacent, so a
            // warp's 32 rows load one 512-byte run)
            const float4* csr = reinterpret_cast<const float4*>(rp.cs) + (row_ok ? row : 0);
            const size_t cld = (size_t)rp.cs_ld;
            // (TMA path: cs_next holds the next (cos, sin) chunk, loaded one chunk ahead)
            if (!cs_ready) {
#pragma unroll
              for (int e = 0; e < 8; ++e) cs_next[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll 1
            for (int hh = 0; hh < p.bn / rp.hd; ++hh) {
              const int col0 = nt * p.bn + hh * rp.hd;  // first column of this head
              const int head = col0 / rp.hd;
              if (col0 >= p.N) break;
              const bool is_v = head >= rp.qh + rp.kvh, is_k = !is_v && head >= rp.qh;
              T* dst = nullptr;
              if ((is_k || is_v) && slot_ok) {
                const int kh = head - rp.qh - (is_v ? rp.kvh : 0);
                dst = reinterpret_cast<T*>(is_v ? rp.v_cache : rp.k_cache) +
                      (((size_t)page * rp.kvh + kh) * rp.page_size + off) * rp.hd;
              }
              if ((is_k || is_v) && row_ok && !slot_ok && hh == 0)
                report(p.err, SAR_ERR_BOUNDS, SITE_ROPE_BOUNDS, row);
              float* crow = C + (size_t)row * p.N + col0;
              if (p.tma_out && rp.hd == 128 && (is_k || is_v)) {
                // k / v head: rotated (k) and rounded once; no fp32 copy (the
                // attention kernels read k and v from the pages).  The warp's
                // 32 rows are staged as 16-bit [2 dim halves][32 rows][128 B]
                // (128-byte swizzle) in its 8 KB for this head and the page-run
                // boxes go out by TMA into the cache's tensor map
                const uint32_t stg = epi_stage + (uint32_t)(q * 4 * kEpiBoxBytes + hh * 8192);
                if (lane == 0) bulk_wait_read_all();  // earlier stores have read the staging
                __syncwarp();
                // chunk 0 of this head (the tile's first, for s == 0 and head 0, already loaded)
                if (is_k && row_ok && !cs_smem && !(cs_ready && s == 0 && hh == 0)) {
#pragma unroll
                  for (int e = 0; e < 8; ++e) cs_next[e] = __ldg(csr + e * cld);
                }
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                  uint32_t x1[16], x2[16];
                  tmem_ld16(sbase + hh * 128 + j * 16, x1);
                  tmem_ld16(sbase + hh * 128 + 64 + j * 16, x2);
                  float r1[16], r2[16];
                  if (is_v) {
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                      r1[e] = __uint_as_float(x1[e]);
                      r2[e] = __uint_as_float(x2[e]);
                    }
                  } else {
                    float4 cc[8];
                    if (cs_smem) {
#pragma unroll
                      for (int e = 0; e < 8; ++e) cc[e] = lds_f4(cs_base + (uint32_t)(((j * 8 + e) * 32 + lane) * 16));
                    } else {
#pragma unroll
                      for (int e = 0; e < 8; ++e) cc[e] = cs_next[e];
                      if (row_ok && j < 3) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) cs_next[e] = __ldg(csr + ((j + 1) * 8 + e) * cld);
                      }
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                      const float4 t4 = cc[e >> 1];
                      const float tc = (e & 1) ? t4.z : t4.x, ts = (e & 1) ? t4.w : t4.y;
                      const float a1 = __uint_as_float(x1[e]), a2 = __uint_as_float(x2[e]);
                      r1[e] = a1 * tc - a2 * ts;
                      r2[e] = a2 * tc + a1 * ts;
                    }
                  }
                  uint32_t o1[8], o2[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    o1[e] = Elem<T>::pack(r1[2 * e], r1[2 * e + 1]);
                    o2[e] = Elem<T>::pack(r2[2 * e], r2[2 * e + 1]);
                  }
                  if (in_run) {
                    // dims [16j, 16j + 16) of each half: 16-byte chunks 2j and 2j + 1 of the row
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                      const uint32_t cofs = (uint32_t)(lane * 128 + (((2 * j + c) ^ (lane & 7)) << 4));
                      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + cofs), "r"(o1[4 * c]),
                                   "r"(o1[4 * c + 1]), "r"(o1[4 * c + 2]), "r"(o1[4 * c + 3])
                                   : "memory");
                      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + 4096 + cofs), "r"(o2[4 * c]),
                                   "r"(o2[4 * c + 1]), "r"(o2[4 * c + 2]), "r"(o2[4 * c + 3])
                                   : "memory");
                    }
                  } else if (dst) {
                    uint4* d1 = reinterpret_cast<uint4*>(dst + j * 16);
                    uint4* d2 = reinterpret_cast<uint4*>(dst + 64 + j * 16);
                    d1[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                    d1[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
                    d2[0] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                    d2[1] = make_uint4(o2[4], o2[5], o2[6], o2[7]);
                  }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
                __syncwarp();
                if (lane == 0 && (run0 || run1)) {
                  const CUtensorMap* kvmap = is_v ? &tm_vp : &tm_kp;
                  const int kh = head - rp.qh - (is_v ? rp.kvh : 0);
                  if (run0) {
                    const int kr = (pg_b0 * rp.kvh + kh) * rp.page_size + of_b0;
                    tma_store_2d(kvmap, 0, kr, stg);
                    tma_store_2d(kvmap, 64, kr, stg + 4096);
                  }
                  if (run1) {
                    const int kr = (pg_b1 * rp.kvh + kh) * rp.page_size + of_b1;
                    tma_store_2d(kvmap, 0, kr, stg + 2048);
                    tma_store_2d(kvmap, 64, kr, stg + 4096 + 2048);
                  }
                  bulk_commit();
                }
                ++epi_n;
                after_kv = true;
                continue;
              }
              if (p.tma_out && rp.hd == 128) {
                // q head: fp32 rows through shared memory: per round two
                // 32x32 boxes, columns [32bp, 32bp+32) and [64+32bp, 96+32bp) --
                // the rotate-half partners -- each written by one TMA store
                // (rows past M clipped).  Rounds alternate between two box
                // pairs, so a round waits only for the stores of the round
                // before last.  The (cos, sin) chunk of the next 16
                // frequencies is loaded one chunk ahead (into the next head's
                // first chunk), so its L2 latency overlaps this chunk's work.
                const int row0 = (mt * MSUB + s) * 128 + q * 32;
                const int heads = p.bn / rp.hd;
                auto rotates = [&](int h) {
                  const int c0 = nt * p.bn + h * rp.hd;
                  return h < heads && c0 < p.N && c0 / rp.hd < rp.qh + rp.kvh;
                };
                if (hh == 0 && row_ok && rotates(0) && !cs_smem && !(cs_ready && s == 0)) {
#pragma unroll
                  for (int e = 0; e < 8; ++e) cs_next[e] = __ldg(csr + e * cld);
                }
#pragma unroll 1
                for (int bp = 0; bp < 2; ++bp) {
                  const uint32_t b0 = epi_stage + (uint32_t)((q * 4 + (epi_n >> 1 & 1) * 2) * kEpiBoxBytes);
                  const uint32_t b1 = b0 + kEpiBoxBytes;
                  if (lane == 0) {
                    // the pair used two rounds ago has been read (all stores, after a k/v head's staging)
                    if (after_kv)
                      bulk_wait_read_all();
                    else
                      bulk_wait_read_all_but_one();
                  }
                  after_kv = false;
                  __syncwarp();
#pragma unroll 1
                  for (int jj = 0; jj < 2; ++jj) {
                    const int j = bp * 2 + jj;  // 16-column chunk of each half
                    uint32_t x1[16], x2[16];
                    tmem_ld16(sbase + hh * 128 + j * 16, x1);
                    tmem_ld16(sbase + hh * 128 + 64 + j * 16, x2);
                    float r1[16], r2[16];
                    if (is_v) {
                      tmem_wait_ld();
#pragma unroll
                      for (int e = 0; e < 16; ++e) {
                        r1[e] = __uint_as_float(x1[e]);
                        r2[e] = __uint_as_float(x2[e]);
                      }
                    } else {
                      float4 cc[8];
                      if (cs_smem) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) cc[e] = lds_f4(cs_base + (uint32_t)(((j * 8 + e) * 32 + lane) * 16));
                      } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) cc[e] = cs_next[e];
                        // the chunk after this one: j + 1 of this head, else chunk 0 of the next
                        const bool more = j < 3 || rotates(hh + 1);
                        if (row_ok && more) {
                          const int jn = (j + 1) & 3;
#pragma unroll
                          for (int e = 0; e < 8; ++e) cs_next[e] = __ldg(csr + (jn * 8 + e) * cld);
                        }
                      }
                      tmem_wait_ld();
#pragma unroll
                      for (int e = 0; e < 16; ++e) {
                        const float4 t4 = cc[e >> 1];
                        const float tc = (e & 1) ? t4.z : t4.x, ts = (e & 1) ? t4.w : t4.y;
                        const float a1 = __uint_as_float(x1[e]), a2 = __uint_as_float(x2[e]);
                        r1[e] = a1 * tc - a2 * ts;
                        r2[e] = a2 * tc + a1 * ts;
                      }
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                      const uint32_t off = (uint32_t)(lane * 128 + (((4 * jj + c) ^ (lane & 7)) << 4));
                      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(b0 + off), "f"(r1[4 * c]),
                                   "f"(r1[4 * c + 1]), "f"(r1[4 * c + 2]), "f"(r1[4 * c + 3])
                                   : "memory");
                      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(b1 + off), "f"(r2[4 * c]),
                                   "f"(r2[4 * c + 1]), "f"(r2[4 * c + 2]), "f"(r2[4 * c + 3])
                                   : "memory");
                    }
                  }
                  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
                  __syncwarp();
                  if (lane == 0) {
                    tma_store_2d(&tm_c, col0 + 32 * bp, row0, b0);
                    tma_store_2d(&tm_c, col0 + 64 + 32 * bp, row0, b1);
                    bulk_commit();
                  }
                  epi_n += 2;
                }
                continue;
              }
              if (is_v) {
#pragma unroll 1
                for (int j = 0; j < rp.hd / 16; ++j) {
                  uint32_t v[16];
                  tmem_ld16(sbase + hh * rp.hd + j * 16, v);
                  tmem_wait_ld();
                  if (!row_ok) continue;
                  float4* c4 = reinterpret_cast<float4*>(crow + j * 16);
                  uint32_t o[8];
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    c4[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                        __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
#pragma unroll
                  for (int e = 0; e < 8; ++e) o[e] = Elem<T>::pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                  if (dst) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + j * 16);
                    d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
                  }
                }
              } else {
                // the (cos, sin) pairs of the next 16 frequencies are loaded one
                // chunk ahead, so their L2 latency overlaps this chunk's work
                float4 cn[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) cn[e] = row_ok ? __ldg(csr + e * cld) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                for (int j = 0; j < half / 16; ++j) {
                  float4 cc[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) cc[e] = cn[e];
                  if (row_ok && j + 1 < half / 16) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) cn[e] = __ldg(csr + ((j + 1) * 8 + e) * cld);
                  }
                  uint32_t x1[16], x2[16];
                  tmem_ld16(sbase + hh * rp.hd + j * 16, x1);
                  tmem_ld16(sbase + hh * rp.hd + half + j * 16, x2);
                  tmem_wait_ld();
                  if (!row_ok) continue;
                  float r1[16], r2[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e) {
                    const float4 t4 = cc[e >> 1];
                    const float tc = (e & 1) ? t4.z : t4.x, ts = (e & 1) ? t4.w : t4.y;
                    const float a1 = __uint_as_float(x1[e]), a2 = __uint_as_float(x2[e]);
                    r1[e] = a1 * tc - a2 * ts;
                    r2[e] = a2 * tc + a1 * ts;
                  }
                  float4* c1 = reinterpret_cast<float4*>(crow + j * 16);
                  float4* c2 = reinterpret_cast<float4*>(crow + half + j * 16);
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    c1[e] = make_float4(r1[4 * e], r1[4 * e + 1], r1[4 * e + 2], r1[4 * e + 3]);
                    c2[e] = make_float4(r2[4 * e], r2[4 * e + 1], r2[4 * e + 2], r2[4 * e + 3]);
                  }
                  if (dst) {
                    uint32_t o1[8], o2[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                      o1[e] = Elem<T>::pack(r1[2 * e], r1[2 * e + 1]);
                      o2[e] = Elem<T>::pack(r2[2 * e], r2[2 * e + 1]);
                    }
                    uint4* d1 = reinterpret_cast<uint4*>(dst + j * 16);
                    uint4* d2 = reinterpret_cast<uint4*>(dst + half + j * 16);
                    d1[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                    d1[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
                    d2[0] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                    d2[1] = make_uint4(o2[4], o2[5], o2[6], o2[7]);
                  }
                }
              }
            }
          } else if (EPI == SAR_EPI_SWIGLU && p.tma_out) {
            // packed columns [h*128, h*128+64) gate, [h*128+64, h*128+128) up:
            // this warp's 32 rows x 64 outputs per block pair go through shared
            // memory (128-byte swizzle) to one TMA store; rows past M are clipped
            const int F = p.N >> 1;
            const int row0 = (mt * MSUB + s) * 128 + q * 32;
#pragma unroll 1
            for (int h = 0; h < p.bn / 128; ++h) {
              const int ocol = nt * (p.bn / 2) + h * 64;
              if (ocol >= F) break;
              const uint32_t box = epi_stage + (uint32_t)((q * 2 + (epi_n & 1)) * kEpiBoxBytes);
              if (lane == 0) bulk_wait_read_all_but_one();  // the box used two stores ago is read
              __syncwarp();
#pragma unroll 1
              for (int j = 0; j < 4; ++j) {
                uint32_t g[16], u[16];
                tmem_ld16(sbase + h * 128 + j * 16, g);
                tmem_ld16(sbase + h * 128 + 64 + j * 16, u);
                tmem_wait_ld();
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float a0 = silu(__uint_as_float(g[2 * e])) * __uint_as_float(u[2 * e]);
                  const float a1 = silu(__uint_as_float(g[2 * e + 1])) * __uint_as_float(u[2 * e + 1]);
                  o[e] = Elem<T>::pack(a0, a1);
                }
                // outputs j*16 .. j*16+15 of this row: 16-byte chunks 2j and 2j+1
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 box + (uint32_t)(lane * 128 + (((2 * j) ^ (lane & 7)) << 4))),
                             "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                             : "memory");
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 box + (uint32_t)(lane * 128 + (((2 * j + 1) ^ (lane & 7)) << 4))),
                             "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                             : "memory");
              }
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tm_c, ocol, row0, box);
                bulk_commit();
              }
              ++epi_n;
            }
          } else if constexpr (EPI == SAR_EPI_SWIGLU) {
            // packed columns [h*128, h*128+64) gate, [h*128+64, h*128+128) up
            const int F = p.N >> 1;
            T* C = reinterpret_cast<T*>(p.c);
#pragma unroll 1
            for (int h = 0; h < p.bn / 128; ++h) {
#pragma unroll 1
              for (int j = 0; j < 4; ++j) {
                uint32_t g[16], u[16];
                tmem_ld16(sbase + h * 128 + j * 16, g);
                tmem_ld16(sbase + h * 128 + 64 + j * 16, u);
                tmem_wait_ld();
                const int ocol = nt * (p.bn / 2) + h * 64 + j * 16;
                if (row_ok && ocol < F) {
                  uint32_t o[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    const float a0 = silu(__uint_as_float(g[2 * e])) * __uint_as_float(u[2 * e]);
                    const float a1 = silu(__uint_as_float(g[2 * e + 1])) * __uint_as_float(u[2 * e + 1]);
                    o[e] = Elem<T>::pack(a0, a1);
                  }
                  uint4* dst = reinterpret_cast<uint4*>(C + (size_t)row * F + ocol);
                  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
              }
            }
          } else if (EPI == SAR_EPI_RESIDUAL && p.tma_out) {
            // in place, C += D: this warp's 32 rows x 32 columns at a time go
            // through shared memory (128-byte swizzle, conflict-free) and are
            // added into C by one TMA reduction (element-wise atomic, so K
            // ranges of a split tile may land in any order); rows past M are
            // clipped by the tensor map
            const int row0 = (mt * MSUB + s) * 128 + q * 32;
#pragma unroll 1
            for (int j = 0; j < p.bn / kEpiBox; ++j) {
              const int col = nt * p.bn + j * kEpiBox;
              if (col >= p.N) break;
              uint32_t v0[16], v1[16];
              tmem_ld16(sbase + j * kEpiBox, v0);
              tmem_ld16(sbase + j * kEpiBox + 16, v1);
              tmem_wait_ld();
              const uint32_t box = epi_stage + (uint32_t)((q * 2 + (epi_n & 1)) * kEpiBoxBytes);
              if (lane == 0) bulk_wait_read_all_but_one();  // the box used two reductions ago is read
              __syncwarp();
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint32_t* v = c < 4 ? v0 : v1;
                const int e = (c & 3) * 4;
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 box + (uint32_t)(lane * 128 + ((c ^ (lane & 7)) << 4))),
                             "r"(v[e]), "r"(v[e + 1]), "r"(v[e + 2]), "r"(v[e + 3])
                             : "memory");
              }
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
              __syncwarp();
              if (lane == 0) {
                tma_reduce_add_2d(&tm_c, col, row0, box);
                bulk_commit();
              }
              ++epi_n;
            }
          } else {
#pragma unroll 1
            for (int j = 0; j < p.bn / 16; ++j) {
              uint32_t v[16];
              tmem_ld16(sbase + j * 16, v);
              tmem_wait_ld();
              const int col = nt * p.bn + j * 16;
              if (!row_ok || col >= p.N) continue;
              if constexpr (EPI == SAR_EPI_F32) {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.c) + (size_t)row * p.N + col);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
              } else if constexpr (EPI == SAR_EPI_RESIDUAL) {
                // fp32 residual stream: C = D + R, both fp32 (R may equal C)
                const float4* rs = reinterpret_cast<const float4*>(
                    reinterpret_cast<const float*>(p.r) + (size_t)row * p.N + col);
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.c) + (size_t)row * p.N + col);
                if (partial) {
                  // split-K / stream-K: every K range adds its share into C (== R) in place
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    atomicAdd(&dst[e], make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3])));
                  continue;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float4 r4 = rs[e];
                  dst[e] = make_float4(__uint_as_float(v[4 * e]) + r4.x, __uint_as_float(v[4 * e + 1]) + r4.y,
                                       __uint_as_float(v[4 * e + 2]) + r4.z, __uint_as_float(v[4 * e + 3]) + r4.w);
                }
              } else {
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = Elem<T>::pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.c) + (size_t)row * p.N + col);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
          }
        }
      } else {
        // swap: accumulator lane = weight row, TMEM column = token
        const int tok0 = mt * p.bn;
        if constexpr (EPI == kEpiRope) {
          // lane = output column n of one or two heads; the rotation partner
          // (dim i with i + hd/2) is lane ^ hd/2, exchanged through shared memory
          const RopeEpi& rp = p.rope;
          const int half = rp.hd >> 1;
          const int n = nt * 128 + lrow;
          const int head = n / rp.hd, local = n - head * rp.hd;
          const bool first = local < half;
          const int fi = first ? local : local - half;
          const bool is_v = head >= rp.qh + rp.kvh, is_k = !is_v && head >= rp.qh;
          const int kh = head - rp.qh - (is_v ? rp.kvh : 0);
          T* cache = reinterpret_cast<T*>(is_v ? rp.v_cache : rp.k_cache);
          float* C = reinterpret_cast<float*>(p.c);
#pragma unroll 1
          for (int j = 0; j < p.bn / 16; ++j) {
            uint32_t v[16];
            if (alive) {
              tmem_ld16(tbase + j * 16, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) xchg[lrow * 17 + e] = __uint_as_float(v[e]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (alive && n < p.N) {
              const int pl = lrow ^ half;
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int m = tok0 + j * 16 + e;
                if (m >= p.M) continue;
                const float x = __uint_as_float(v[e]);
                float r = x;
                if (!is_v) {
                  const float y = xchg[pl * 17 + e];
                  const float2 t = rp.cs[((size_t)(fi >> 1) * rp.cs_ld + m) * 2 + (fi & 1)];
                  r = first ? x * t.x - y * t.y : x * t.x + y * t.y;
                }
                C[(size_t)m * p.N + n] = r;
                if (is_k || is_v) {
                  const int sl = rp.slot[m];
                  const int page = sl >= 0 ? sl / rp.page_size : -1;
                  if (sl >= 0 && page < rp.num_pages)
                    cache[(((size_t)page * rp.kvh + kh) * rp.page_size + (sl - page * rp.page_size)) * rp.hd + local] =
                        Elem<T>::from(r);
                  else if (local == 0)
                    report(p.err, SAR_ERR_BOUNDS, SITE_ROPE_BOUNDS, m);
                }
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        } else if constexpr (EPI == SAR_EPI_SWIGLU) {
          // A tile = one packed block pair: lanes 0..63 gate, 64..127 up
          const int F = p.N >> 1;
          const int ocol = nt * 64 + (lrow & 63);
          T* C = reinterpret_cast<T*>(p.c);
#pragma unroll 1
          for (int j = 0; j < p.bn / 16; ++j) {
            uint32_t v[16];
            if (alive) {
              tmem_ld16(tbase + j * 16, v);
              tmem_wait_ld();
            }
            if (alive && lrow >= 64) {
#pragma unroll
              for (int e = 0; e < 16; ++e) xchg[(lrow - 64) * 17 + e] = __uint_as_float(v[e]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (alive && lrow < 64 && ocol < F) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int m = tok0 + j * 16 + e;
                if (m < p.M) {
                  const float a = silu(__uint_as_float(v[e])) * xchg[lrow * 17 + e];
                  C[(size_t)m * F + ocol] = Elem<T>::from(a);
                }
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        } else {
          const int n = nt * 128 + lrow;
#pragma unroll 1
          for (int j = 0; j < p.bn / 16; ++j) {
            uint32_t v[16];
            tmem_ld16(tbase + j * 16, v);
            tmem_wait_ld();
            if (n >= p.N) continue;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int m = tok0 + j * 16 + e;
              if (m >= p.M) break;
              const size_t idx = (size_t)m * p.N + n;
              float f = __uint_as_float(v[e]);
              if constexpr (EPI == SAR_EPI_F32) {
                reinterpret_cast<float*>(p.c)[idx] = f;
              } else if constexpr (EPI == SAR_EPI_RESIDUAL) {
                if (partial)
                  atomicAdd(reinterpret_cast<float*>(p.c) + idx, f);
                else
                  reinterpret_cast<float*>(p.c)[idx] = f + reinterpret_cast<const float*>(p.r)[idx];
              } else {
                reinterpret_cast<T*>(p.c)[idx] = Elem<T>::from(f);
              }
            }
          }
        }
      }
      tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();
        if (alive && lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&acce_bar[acc]), 0));
      } else {
        if (alive) mbar_arrive(smem_u32(&acce_bar[acc]));
      }
    }
    // the TMA reductions have written C before the CTA (and its shared memory) goes
    if (epi_n > 0 && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (p.cl > 1) cluster_sync();  // neither CTA of a pair leaves while the other may still address it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, (uint32_t)p.tmem_cols);
  }
}

template <typename T, int EPI, bool SWAP, int MSUB, bool PAIR>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&gemm_tc_kernel<T, EPI, SWAP, MSUB, PAIR>);
}

template <typename T>
const void* pick_kernel_t(int epi, bool swap, int msub, bool pair) {
#define SAR_PICK(E)                                                                               \
  if (epi == E) {                                                                                 \
    if (swap) return kernel_ptr<T, E, true, 1, false>();                                          \
    if (pair) return kernel_ptr<T, E, false, 1, true>();                                          \
    return msub == 2 ? kernel_ptr<T, E, false, 2, false>() : kernel_ptr<T, E, false, 1, false>(); \
  }
  SAR_PICK(SAR_EPI_STORE)
  SAR_PICK(SAR_EPI_RESIDUAL)
  SAR_PICK(SAR_EPI_SWIGLU)
  SAR_PICK(SAR_EPI_F32)
  SAR_PICK(kEpiRope)
#undef SAR_PICK
  return nullptr;
}

const void* pick_kernel(int storage, int epi, bool swap, int msub, bool pair) {
  return storage == SAR_STORAGE_BF16 ? pick_kernel_t<__nv_bfloat16>(epi, swap, msub, pair)
                                     : pick_kernel_t<__half>(epi, swap, msub, pair);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

int make_tmap_16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 int storage) {
  auto fn = encode_fn();
  if (!fn) return set_error(SAR_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * 2) % 16 || rows == 0 || box_rows == 0 ||
      box_rows > 256)
    return set_error(SAR_ERR_INVALID_ARG, "tensor map: pointer/stride not 16-byte aligned or bad box");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      storage == SAR_STORAGE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(SAR_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
  return SAR_OK;
}

// fp32 [rows, cols] row-major, boxes of box_rows x box_cols (box_cols * 4 =
// 128 bytes: 128-byte swizzle), for the epilogue's TMA reductions.
int make_tmap_f32_box(CUtensorMap* map, void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return set_error(SAR_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * 4) % 16 || rows == 0 || box_cols * 4 != 128)
    return set_error(SAR_ERR_INVALID_ARG, "tensor map (fp32 output): pointer/stride not 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(SAR_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
  return SAR_OK;
}

int gemm_config(int M, int N, int K, int epi, int variant, GemmCfg* cfg, bool in_place) {
  const bool two_ctas = (variant & SAR_GEMM_TWO_CTAS) != 0;
  const bool want_sk = (variant & SAR_GEMM_STREAM_K) != 0;
  variant &= ~(SAR_GEMM_TWO_CTAS | SAR_GEMM_STREAM_K);
  const bool auto_variant = variant == SAR_GEMM_AUTO;
  if (M < 1 || N < 64 || K < 64 || N % 64 || K % 64)
    return set_error(SAR_ERR_UNSUPPORTED, "gemm: need M >= 1, N and K multiples of 64");
  if (epi == SAR_EPI_SWIGLU && N % 128)
    return set_error(SAR_ERR_UNSUPPORTED, "gemm: SwiGLU needs whole 64-row gate/up block pairs");
  const int sms = num_sms();
  const int k_blocks = K / kBK;
  // split-K (K ranges added into an fp32 output in place) only for the
  // in-place residual epilogue; pick the split count with the best makespan
  const bool can_split = epi == SAR_EPI_RESIDUAL && in_place;
  // SM clocks per 64-wide K slab of one tile: the larger of the MMA time
  // (128 x bn x 64 takes 2*bn clocks per 128-row sub-tile) and the time to
  // stream its operands into shared memory (about 86 bytes per clock per SM,
  // as the 128x256 and CTA-pair tilings measure on the projection shapes)
  // (a pair tile: each SM computes its 128 rows x bn and loads half the weight rows)
  auto kslab_clocks = [](int msub, int bn, bool pair = false) -> long {
    return std::max<long>(2L * msub * bn, (msub * 16384L + (pair ? bn / 2 : bn) * 128L) / 86);
  };
  // slots: units running at once (SMs, SM pairs, or two CTAs per SM)
  auto best_split = [&](long tiles, long per_kb_work, int* splits, long slots) {
    long best = -1;
    for (int sp = 1; sp <= (can_split ? 4 : 1); ++sp) {
      const long kb = (k_blocks + sp - 1) / sp;
      if (sp > 1 && kb < 8) break;
      const long units = tiles * sp;
      // waves x unit work, plus a small charge per extra split for the atomic adds
      const long c = ((units + slots - 1) / slots) * kb * per_kb_work * (sp > 1 ? 21 : 20) / 20;
      if (best < 0 || c < best) {
        best = c;
        *splits = sp;
      }
    }
    return best;
  };
  GemmCfg c;
  if (variant == SAR_GEMM_AUTO) {
    // swap (tokens on the MMA's N side) only up to 32 rows: above that the
    // 128-row token tiles do as well or better (Mistral-shaped layer, the
    // four projections with L2 flushed: 48 and 64 rows 133.7 vs 137.9 us,
    // 96 rows 137.8 vs 143.9 us, 128 rows 139.9 vs 150.1 us; 256 rows: QKV
    // 29.3 vs 39.6 us, gate/up 74.4 vs 88.7 us), as the swap tiling's split-K
    // sums go through fp32 scratch and a finishing kernel where the 128-row
    // tiles fuse their epilogues; at 8 rows and fewer swap is far ahead
    // (131.7 vs 150.1 us)
    if (M <= 32) {
      variant = SAR_GEMM_SWAP;
    } else {
      // makespan estimate: waves x per-unit MMA work
      auto cost = [&](int msub, int bn, bool pair) {
        long m_tiles = (M + 128 * msub - 1) / (128 * msub);
        if (pair) m_tiles = (m_tiles + 1) / 2;  // a pair unit covers two token tiles on two SMs
        const long tiles = m_tiles * ((N + bn - 1) / bn);
        int sp = 1;
        return best_split(tiles, kslab_clocks(msub, bn, pair), &sp, pair ? sms / 2 : sms) * 1000 + tiles;
      };
      variant = SAR_GEMM_M128_N256;
      long best = (N % 256 == 0) ? cost(1, 256, false) : -1;
      if (best < 0 || cost(1, 128, false) < best) { variant = SAR_GEMM_M128_N128; best = cost(1, 128, false); }
      if (cost(2, 128, false) < best) { variant = SAR_GEMM_M256_N128; best = cost(2, 128, false); }
      if (N % 256 == 0 && cost(1, 256, true) < best) variant = SAR_GEMM_PAIR_N256;
    }
  }
  switch (variant) {
    case SAR_GEMM_M128_N128: c.swap = 0; c.msub = 1; c.bn = 128; break;
    case SAR_GEMM_M128_N256: c.swap = 0; c.msub = 1; c.bn = 256; break;
    case SAR_GEMM_M256_N128: c.swap = 0; c.msub = 2; c.bn = 128; break;
    case SAR_GEMM_PAIR_N256: c.swap = 0; c.msub = 1; c.bn = 256; c.pair = 1; break;
    case SAR_GEMM_PAIR_N128: c.swap = 0; c.msub = 1; c.bn = 128; c.pair = 1; break;
    case SAR_GEMM_PAIR_N192: c.swap = 0; c.msub = 1; c.bn = 192; c.pair = 1; break;
    case SAR_GEMM_SWAP:
      if (M > 256) return set_error(SAR_ERR_UNSUPPORTED, "gemm: swap tiling needs M <= 256");
      c.swap = 1; c.msub = 1; c.bn = (M + 15) / 16 * 16; break;
    default: return set_error(SAR_ERR_INVALID_ARG, "gemm: unknown variant");
  }
  if (!c.swap && (N % c.bn || c.bn % 128) && epi == SAR_EPI_SWIGLU)
    return set_error(SAR_ERR_UNSUPPORTED, "gemm: SwiGLU tiles must not straddle N and hold whole gate/up blocks");
  if (c.swap) {
    c.m_tiles = 1;
    c.n_tiles = (N + 127) / 128;
    c.a_box_rows = 128;   // weights
    c.b_box_rows = c.bn;  // tokens
    c.cl = 1;
  } else {
    c.m_tiles = (M + 128 * c.msub - 1) / (128 * c.msub);
    c.n_tiles = (N + c.bn - 1) / c.bn;
    // a CTA pair is a 2-CTA cluster over two token tiles; every other tiling is one CTA
    if (c.pair) {
      c.cl = 2;
      c.m_tiles += c.m_tiles & 1;  // an odd last tile pairs with an all-padding one
    } else {
      c.cl = 1;
    }
    c.a_box_rows = 128;          // tokens
    c.b_box_rows = c.bn / c.cl;  // the weight tile, or this CTA's half of the pair's
  }
  c.m_groups = c.m_tiles / c.cl;
  const int stage_bytes = c.msub * kTileA + (c.pair ? c.bn / 2 : c.bn) * kBK * 2;
  c.stage_bytes = stage_bytes;
  // the in-place residual epilogue of the non-swap tilings adds through TMA reductions
  // (the SwiGLU epilogue stores through TMA too)
  c.tma_out = (!c.swap && ((epi == SAR_EPI_RESIDUAL && in_place) || epi == SAR_EPI_SWIGLU || epi == kEpiRope)) ? 1 : 0;
  // (the rotary epilogue alternates two box pairs per warp)
  const int extra = kBarBytes + 1024 +
                    (c.swap ? (epi == SAR_EPI_SWIGLU ? kSwapXchg : epi == kEpiRope ? kSwapXchgRope : 0)
                            : (c.tma_out ? (epi == kEpiRope ? 2 * kEpiStage : kEpiStage) : 0));
  if (two_ctas && (!c.swap || c.bn > 128))
    return set_error(SAR_ERR_UNSUPPORTED, "gemm: two CTAs per SM only with the swap tiling and M <= 128");
  c.per_sm = two_ctas ? 2 : 1;
  // two per SM: each gets half of the SM's shared memory (less 1 KB the system reserves per CTA)
  const int smem_cap = two_ctas ? (kSmemPerSm / 2 - 1024) : kSmemLimit;
  c.stages = std::min(8, (smem_cap - extra) / stage_bytes);
  if (c.stages < 2) return set_error(SAR_ERR_UNSUPPORTED, "gemm: tile does not fit shared memory");
  c.smem = c.stages * stage_bytes + extra;
  c.splits = 1;
  const long per_kb = c.swap ? kslab_clocks(1, c.bn) : kslab_clocks(c.msub, c.bn, c.pair);
  const long slots = (long)sms * c.per_sm / c.cl;
  const long split_cost = best_split((long)c.m_groups * c.n_tiles, per_kb, &c.splits, slots);
  if (want_sk && (!can_split || c.swap || c.m_groups > slots))
    return set_error(SAR_ERR_UNSUPPORTED,
                     "gemm: stream-K needs a non-swap tiling, the in-place residual epilogue and a cluster per token group");
  // stream-K only on request: on the projections of a 512-row step it measured
  // slower than the best split-K (O 32.1 vs 27.2 us, down 51.7 vs 48.3 us), as
  // its extra partial-tile atomic adds all land at the end of the kernel
  (void)split_cost;
  (void)auto_variant;
  if (want_sk) {
    c.sk = 1;
    c.splits = 1;
  }
  c.kb_per_split = (k_blocks + c.splits - 1) / c.splits;
  c.splits = (k_blocks + c.kb_per_split - 1) / c.kb_per_split;  // no empty K range
  c.grid = c.sk ? (int)(slots * c.cl)
                : std::min(c.m_tiles * c.n_tiles * c.splits, sms * c.per_sm) / c.cl * c.cl;  // refined at launch
  *cfg = c;
  return SAR_OK;
}

int gemm_launch(const GemmCfg& cfg, const CUtensorMap& act_map, const CUtensorMap& w_map, int M, int N,
                int K, int epi, int storage, void* c, const void* residual, int* err, cudaStream_t s,
                const RopeEpi* rope) {
  const void* fn = pick_kernel(storage, epi, cfg.swap != 0, cfg.msub, cfg.pair != 0);
  if (!fn) return set_error(SAR_ERR_INVALID_ARG, "gemm: unknown epilogue");
  if (epi == SAR_EPI_RESIDUAL && residual == nullptr)
    return set_error(SAR_ERR_INVALID_ARG, "gemm: residual epilogue without residual");
  if (epi == kEpiRope &&
      (!rope || !rope->slot || !rope->cs || rope->cs_ld < M || (rope->hd != 64 && rope->hd != 128) || N % 128 ||
       (!cfg.swap && cfg.bn % rope->hd) ||
       N != (rope->qh + 2 * rope->kvh) * rope->hd || rope->page_size <= 0))
    return set_error(SAR_ERR_INVALID_ARG, "gemm: rotary epilogue arguments");
  Params p;
  if (rope) p.rope = *rope;
  p.M = M;
  p.N = N;
  p.K = K;
  p.bn = cfg.bn;
  p.m_tiles = cfg.m_tiles;
  p.n_tiles = cfg.n_tiles;
  p.k_blocks = K / kBK;
  p.splits = cfg.splits;
  p.kb_per_split = cfg.kb_per_split;
  p.sk = cfg.sk;
  if ((cfg.splits > 1 || cfg.sk) && (c != residual || epi != SAR_EPI_RESIDUAL))
    return set_error(SAR_ERR_INVALID_ARG, "gemm: split-K / stream-K needs the residual output in place");
  p.stages = cfg.stages;
  p.stage_bytes = cfg.stage_bytes;
  p.tmem_cols = pow2_at_least(2 * cfg.msub * cfg.bn);
  p.cl = cfg.cl;
  p.m_groups = cfg.m_groups;
  p.c = c;
  p.r = residual;
  p.err = err;
  // (the rotary epilogue's TMA path covers head_dim 128)
  p.tma_out = (cfg.tma_out && !(epi == kEpiRope && rope->hd != 128)) ? 1 : 0;
  CUtensorMap tc_map, kp_map, vp_map;
  std::memset(&tc_map, 0, sizeof(tc_map));
  std::memset(&kp_map, 0, sizeof(kp_map));
  std::memset(&vp_map, 0, sizeof(vp_map));
  if (epi == kEpiRope && p.tma_out) {
    if (!rope->kmap || !rope->vmap) return set_error(SAR_ERR_INVALID_ARG, "gemm: rotary epilogue without page maps");
    kp_map = *rope->kmap;
    vp_map = *rope->vmap;
  }
  if (p.tma_out) {
    int mrc = SAR_OK;
    if (cfg.swap || (epi == SAR_EPI_RESIDUAL && c != residual) ||
        (epi != SAR_EPI_RESIDUAL && epi != SAR_EPI_SWIGLU && epi != kEpiRope))
      return set_error(SAR_ERR_INVALID_ARG, "gemm: TMA epilogue needs the residual output in place, SwiGLU or rotary");
    if (epi == SAR_EPI_RESIDUAL || epi == kEpiRope)
      mrc = make_tmap_f32_box(&tc_map, c, (uint64_t)M, (uint64_t)N, kEpiBox, kEpiBox);
    else  // SwiGLU output [M, N / 2] of the storage type, boxes of 32 rows x 64 columns
      mrc = make_tmap_16(&tc_map, c, (uint64_t)M, (uint64_t)(N / 2), kEpiBox, storage);
    if (mrc != SAR_OK) return mrc;
  }
  if (cfg.cl != (cfg.pair ? 2 : 1) || cfg.m_tiles % cfg.cl || cfg.m_groups * cfg.cl != cfg.m_tiles ||
      cfg.bn % (8 * cfg.cl) || (cfg.pair && (cfg.msub != 1 || cfg.swap)) ||
      cfg.stage_bytes != cfg.msub * kTileA + (cfg.pair ? cfg.bn / 2 : cfg.bn) * kBK * 2)
    return set_error(SAR_ERR_INVALID_ARG, "gemm: inconsistent cluster configuration");
  SAR_TRY(ensure_smem_attr(fn, kSmemLimit, "gemm: set smem attribute"));
  const CUtensorMap& ta = cfg.swap ? w_map : act_map;
  const CUtensorMap& tb = cfg.swap ? act_map : w_map;
  void* args[] = {const_cast<CUtensorMap*>(&ta), const_cast<CUtensorMap*>(&tb), &tc_map, &kp_map, &vp_map, &p};
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[2];
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = (size_t)cfg.smem;
  lc.stream = s;
  lc.attrs = attr;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  lc.numAttrs = 1;
  int grid = cfg.grid;
  if (cfg.cl > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cfg.cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.numAttrs = 2;
    // persistent grid: as many whole clusters as can be resident at once (the
    // SMs of a GPC need not divide into clusters evenly)
    cudaLaunchConfig_t qc = lc;  // the cluster shape alone
    qc.gridDim = dim3(cfg.cl * 64);
    qc.attrs = &attr[1];
    qc.numAttrs = 1;
    int mc = 0;
    SAR_TRY(max_active_clusters(fn, qc, cfg.cl, &mc, "gemm: cluster occupancy"));
    // stream-K: every resident cluster takes a share
    grid = (cfg.sk ? mc : std::min(cfg.m_groups * cfg.n_tiles * cfg.splits, mc)) * cfg.cl;
    if (cfg.sk && mc < cfg.m_groups)
      return set_error(SAR_ERR_UNSUPPORTED, "gemm: stream-K needs a resident cluster per token group");
  }
  lc.gridDim = dim3(grid);
  cudaError_t e = cudaLaunchKernelExC(&lc, fn, args);
  if (e != cudaSuccess) return cuda_error(e, "gemm launch");
  count_launches(1);
  return SAR_OK;
}

}  // namespace sar
