// Prefill-chunk attention on the 5th-generation tensor cores (head_dim 128,
// pages of a multiple of 16 keys).  The chunk's queries attend causally to the keys of the
// prompt's earlier chunks in the paged KV cache and to their own keys, which
// the rotary/append kernel has already written into the pages ("Prefill uses
// FlashAttention-2", SARATHI technique write-up section 3.3; cross-chunk
// attention, same page section 3.1; chunk k re-reads the KV of the k earlier
// chunks, Sarathi-Serve digest section 4).
//
// One CTA = one query tile (up to 128 consecutive rows of one prompt's chunk,
// from the step's tile table, so one launch serves every chunk of a batch)
// of one query head (352 threads):
//   warps 0, 10 TMA producers of K and of V: each 128-key block is 8 runs of
//               16 keys x 2 dim halves (one box each: 16 keys x 64 dims of one
//               page, 128-byte swizzle) into a ring of 3 K and one of 2 V
//               stages; a K stage frees when S_j has been computed (S runs two
//               blocks ahead, so K is fetched three ahead), a V stage after
//               P_j V_j.  Eight lanes issue a block's sixteen boxes, with the
//               pages read from the block table a group of blocks ahead.
//   warp 1      tensor memory (512 columns) and the single MMA-issuing thread:
//               S_j = Q K_j^T (M 128 x N 128 x K 128; the fp32 queries are
//               rounded once to the storage type, as the keys are) into one of three
//               S buffers, two blocks ahead of the softmax (so the next S is
//               ready when a block's softmax ends); then O += P_j V_j with P_j
//               read from tensor memory and V_j as an MN-major operand.
//   warps 2..9  two warps per row quarter (the TMEM lanes a warp may access),
//               each with 64 of the 128 keys of every block: stage the fp32
//               query rows through the (still idle) V stages, scale and round
//               them into Q, then per block the online softmax in base 2 (the two
//               halves exchange their row maxima through shared memory), P
//               (16-bit) written back over S for the next MMA; O is rescaled
//               in tensor memory only when a row's maximum grows by more than
//               2^8 (the stale maximum keeps P <= 256 otherwise); finally
//               O / l is stored.
// With a sliding window of W keys the CTA starts at the block holding its
// first row's oldest visible key, (first position - W + 1), and masks the
// keys each row may not see; a row whose window misses a whole block keeps a
// maximum of -inf there, and its probabilities are then taken as 0.
// When a step has too few query tiles to fill the SMs, the planner splits a
// tile's key blocks over several CTAs: each writes its unnormalised O with the
// row's maximum and sum, and chunk_combine_kernel merges them (the split-K
// form of the decode attention's long contexts).
// Where one-tile CTAs would need more waves of the SMs than pairs of them,
// the planner lists the tiles in pairs and chunk_attn_tc2_kernel (below) runs
// two query tiles of one head per CTA over shared key blocks.
// CTAs run (tile, head) units heads fastest, in the tile table's order (most
// keys first).  Launched right behind decode attention (wait_at_end), the
// kernel starts without waiting for that kernel and only its last CTA waits
// for it before exiting.
// Every wait is bounded; a timeout records SAR_ERR_TIMEOUT.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "tc05.cuh"

namespace sar {

namespace {

constexpr int kD = 128;
constexpr int kBQ = 128;                       // query rows per CTA (TMEM lanes)
constexpr int kBKV = 128;                      // keys per block
constexpr int kRun = 16;                       // keys per TMA box (page sizes are multiples of it)
constexpr int kRunsPerBlock = kBKV / kRun;
constexpr int kThreads = 352;                  // 11 warps
constexpr int kRegion = 128 * 128;             // [128 rows][128 bytes]: 64 dims of 128 rows
constexpr int kQBytes = 2 * kRegion;           // one 16-bit copy of the Q tile (two dim halves)
constexpr int kKVBytes = 2 * kRegion;          // K (or V) of one block
constexpr int kKStages = 3;                    // one per S buffer: S_j's barrier frees K stage j % 3
constexpr int kVStages = 2;                    // one per P.V barrier: o_done[j % 2] frees V stage j % 2
constexpr int kBarOff = kQBytes + (kKStages + kVStages) * kKVBytes;  // after Q, the K stages, the V stages
constexpr int kRedOff = kBarOff + 256;         // softmax exchange: [3][2][128] floats
constexpr int kSmem = 1024 + kRedOff + 3 * 2 * kBQ * 4;
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
static_assert(kVStages * kKVBytes >= kBQ * kD * 4, "the fp32 query rows are staged in the V stages");
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                      // S buffers: S_j in buffer j % 3, issued two blocks ahead
constexpr uint32_t kColS = 128;               // S buffer b at columns [b*128, b*128+128); P overwrites the first 64
static_assert(kKStages == kSBufs, "K stages are freed by the S barriers");
constexpr uint32_t kColO = kSBufs * kColS;     // O at columns [384, 512)
constexpr float kRescale = 8.f;                // log2 of the growth tolerated before rescaling O
static_assert(kBQ == kChunkTileRowsTc, "the step plans tiles of kBQ rows");

struct Bars {
  // a K stage is free again once S_j (buffer j % 3, stage j % 3) has landed,
  // a V stage once P_j V_j has: s_full and o_done serve as the rings' empty
  // barriers
  uint64_t k_full[kKStages], v_full[kVStages];
  uint64_t s_full[kSBufs], p_full[kSBufs];
  uint64_t o_done[2], q_ready, mma_done;  // o_done[j % 2]: P.V of block j; mma_done: once, after every MMA
  uint32_t tmem_slot;
};

// Instruction descriptor, kind::f16: fp32 accumulate, A and B of format fmt,
// A K-major, B K-major (b_mn = 0) or MN-major (1), M = 128, N = 128.
__device__ __forceinline__ uint32_t idesc_128x128(uint32_t fmt, uint32_t b_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn << 16) | ((uint32_t)(128 >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

// 2^x by the SFU's approximate exponential (relative error about 2^-22;
// 2^-inf = 0), ample for a probability rounded to 16 bits next.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, int* err, int site) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, site) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const ChunkAttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  // Q hi, Q lo, then per stage K then V; each a pair of 16 KB dim-half regions
  const uint32_t q_s = sbase;
  auto k_reg = [&](int s) { return sbase + kQBytes + (uint32_t)(s * kKVBytes); };
  auto v_reg = [&](int s) { return sbase + kQBytes + (uint32_t)((kKStages + s) * kKVBytes); };
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // one CTA per (tile, query head), heads fastest: the launch order is the
  // tile table's (most keys first), so the longest tiles start first
  const int tile_i = blockIdx.x / a.qh;
  const int hq = blockIdx.x - tile_i * a.qh;
  const int G = a.qh / a.kvh;
  const int kh = hq / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&bars->v_full[s]), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->p_full[b]), 8);
    }
    mbar_init(smem_u32(&bars->o_done[0]), 1);
    mbar_init(smem_u32(&bars->o_done[1]), 1);
    mbar_init(smem_u32(&bars->q_ready), 8);
    mbar_init(smem_u32(&bars->mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<false>(smem_u32(&bars->tmem_slot), kTmemCols);
    tmem_relinquish<false>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  if (!a.wait_at_end) pdl_wait();
  pdl_launch_dependents();
  // this CTA's tile (the table lists the most keys first)
  const int4 tl = reinterpret_cast<const int4*>(a.tiles)[2 * tile_i];
  const int row0 = tl.x;   // batch row of the tile's first query
  const int pos0 = tl.y;   // its position in the prompt
  const int rows = tl.z;
  const int32_t* bt = a.bt + tl.w;
  const int4 tl2 = reinterpret_cast<const int4*>(a.tiles)[2 * tile_i + 1];
  const int bt_len = tl2.x;
  const int n_keys = pos0 + rows;  // keys of the last row of this tile, inclusive of it
  // blocks [j0, j0 + nb): planned from the block holding the first row's
  // oldest visible key to the last row's, or one share of that range
  const int j0 = tl2.y;
  const int nb = tl2.z - tl2.y;
  const int part = tl2.w;

  if (warp == 0 || warp == 10) {
    // ---------------- producers: warp 0 K, warp 10 V ----------------
    // The whole warp serves one ring: lane 0 waits for a free stage and arms
    // its barrier, lanes 0..7 issue the two boxes of run g = lane, and the
    // page of every run is read from the block table four to eight blocks
    // ahead (lane L holds run L % 8 of block L / 8 of a group of four), so
    // neither the table's latency nor a serial chain of sixteen copy issues
    // sits between a freed stage and its next block.
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->s_full : bars->o_done;
    const int stages = is_k ? kKStages : kVStages;
    if (lane == 0) tma_prefetch_desc(map);
    const int last_run = (n_keys - 1) / kRun;
    bool ok = (n_keys - 1) / a.page_size < bt_len;
    if (!ok && is_k && lane == 0) report(a.err, SAR_ERR_BOUNDS, SITE_CHUNK_BOUNDS, n_keys);
    const int g = lane & 7, sub = lane >> 3;
    // runs past the last key repeat the last one (finite data, masked)
    auto page_of = [&](int jb, int& page, int& off) {  // block jb + sub counts from block j0
      const int key = min((j0 + jb + sub) * kRunsPerBlock + g, last_run) * kRun;
      const int bi = key / a.page_size;
      page = bt[bi];
      off = key - bi * a.page_size;
    };
    int pa = 0, oa = 0, pb = 0, ob = 0;  // this group of four blocks, the next
    if (!is_k && ok) {
      // the V stages hold the fp32 query rows until Q is ready
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&bars->q_ready), 0, a.err, SITE_CHUNK_PIPE);
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    if (ok) {
      page_of(0, pa, oa);
      if (nb > 4) page_of(4, pb, ob);
    }
    for (int j = 0; j < nb && ok; ++j) {
      const int i = j & 3;
      if (i == 0 && j > 0) {
        pa = pb;
        oa = ob;
        if (j + 4 < nb) page_of(j + 4, pb, ob);
      }
      const int s = j % stages;
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((j / stages) & 1) ^ 1), a.err, SITE_CHUNK_PIPE);
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&full[s]);
      const uint32_t dst = is_k ? k_reg(s) : v_reg(s);
      if (lane == 0) mbar_expect_tx(fb, (uint32_t)kKVBytes);
      __syncwarp();
      int page = __shfl_sync(0xffffffffu, pa, (i << 3) | g);
      const int po = __shfl_sync(0xffffffffu, oa, (i << 3) | g);
      if (lane < kRunsPerBlock) {
        if (page < 0 || page >= a.num_pages) {
          report(a.err, SAR_ERR_BOUNDS, SITE_CHUNK_BOUNDS, page);
          page = 0;
        }
        const int row = (page * a.kvh + kh) * a.page_size + po;
        tma_load_2d(dst + g * (kRun * 128), map, 0, row, fb);
        tma_load_2d(dst + kRegion + g * (kRun * 128), map, 64, row, fb);
      }
    }
    // no copy may still be in flight when the CTA leaves
    if (lane == 0) {
      const int first = max(0, nb - stages);
      for (int j = first; j < nb && ok; ++j)
        ok = mbar_wait(smem_u32(&empty[j % stages]), (uint32_t)((j / stages) & 1), a.err, SITE_CHUNK_PIPE);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t fmt = Elem<T>::kMmaFormat;
      const uint32_t id_s = idesc_128x128(fmt, 0), id_pv = idesc_128x128(fmt, 1);
      // descriptors built once: a byte offset b within shared memory moves a
      // descriptor's start-address field (address / 16) by b / 16, so each MMA
      // adds a constant (this thread issues 16 small MMAs per key block and
      // shares its scheduler with two softmax warps)
      const uint64_t dq = sw128_desc(q_s);
      static_assert(kKStages == 3 && kVStages == 2, "one descriptor per stage, chosen by a select");
      const uint64_t dk0 = sw128_desc(k_reg(0)), dk1 = sw128_desc(k_reg(1)), dk2 = sw128_desc(k_reg(2));
      const uint64_t dv0 = sw128_desc_mn(v_reg(0), kRegion, 1024), dv1 = sw128_desc_mn(v_reg(1), kRegion, 1024);
      bool ok = mbar_wait(smem_u32(&bars->q_ready), 0, a.err, SITE_CHUNK_PIPE);
      auto issue_s = [&](int j) -> bool {
        const int s = j % kKStages;
        if (!mbar_wait(smem_u32(&bars->k_full[s]), (uint32_t)((j / kKStages) & 1), a.err, SITE_CHUNK_PIPE))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + (kColS * (uint32_t)(j % kSBufs));
        const uint64_t db = s == 0 ? dk0 : (s == 1 ? dk1 : dk2);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t o = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
          mma_f16<false>(d, dq + o, db + o, id_s, kk != 0);
        }
        mma_commit(smem_u32(&bars->s_full[j % kSBufs]));
        return true;
      };
      // S_0 and S_1, then per block j: S_{j+2} (into the buffer block j - 1's
      // P.V has just been issued from), P_j V_j
      if (ok) ok = issue_s(0);
      if (ok && nb > 1) ok = issue_s(1);
      for (int j = 0; j < nb && ok; ++j) {
        if (j + 2 < nb && !(ok = issue_s(j + 2))) break;
        if (!(ok = mbar_wait(smem_u32(&bars->p_full[j % kSBufs]), (uint32_t)((j / kSBufs) & 1), a.err,
                             SITE_CHUNK_PIPE)))
          break;
        const int s = j % kVStages;
        if (!(ok = mbar_wait(smem_u32(&bars->v_full[s]), (uint32_t)((j / kVStages) & 1), a.err, SITE_CHUNK_PIPE)))
          break;
        tc_fence_after();
        const uint32_t pcol = tmem + (kColS * (uint32_t)(j % kSBufs));
        const uint64_t dvs = s ? dv1 : dv0;
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk) {
          // 16 keys per step: P columns (two keys per 32-bit column), V rows (16 x 128 bytes)
          mma_f16_ts(tmem + kColO, pcol + kk * 8, dvs + (uint64_t)(kk * (16 * 128 / 16)), id_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->o_done[j & 1]));
      }
      // every MMA issued has completed before tensor memory is released
      mma_commit(smem_u32(&bars->mma_done));
      mbar_wait(smem_u32(&bars->mma_done), 0, a.err, SITE_CHUNK_PIPE);
    }
    __syncwarp();
  } else {
    // ---------------- softmax / epilogue ----------------
    // warps 2..9: row quarter qq = warp & 3 (the TMEM lanes this warp may
    // access), column half hf: each row's 128 keys are split over two warps
    // that exchange their partial maxima through shared memory.
    const int qq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = qq * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    const bool valid = r < rows;
    const int pos = pos0 + r;  // this row's position; keys <= pos are visible
    float* red = reinterpret_cast<float*>(smem + kRedOff);  // [2 parities][2 halves][128 rows]
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + qq) : "memory"); };
    {
      // this half of the query row -> scaled by log2(e) / sqrt(d), rounded
      // to 16 bits, swizzled as the MMA reads it (dim half hf is Q region hf).
      // The fp32 rows are first copied into the V stages (idle until Q is
      // ready) with all sixteen 16-byte copies of a thread in flight at once,
      // [128 rows][32 chunks of 16 B], chunk c of row r at slot c ^ (r % 32)
      const float qscale = rsqrtf((float)kD) * 1.4426950408889634f;
      const float* qp = a.q32 + (size_t)(row0 + r) * a.ld32 + (size_t)hq * kD + hf * 64;
      const uint32_t qstg = v_reg(0) + (uint32_t)(r * 512);
      if (valid) {
#pragma unroll
        for (int cc = 0; cc < 16; ++cc)
          cp_async16(qstg + (uint32_t)((((hf * 16 + cc) ^ (r & 31))) << 4), qp + cc * 4, 16);
      }
      cp_async_commit();
      cp_async_wait<0>();  // a thread reads back only its own copies
#pragma unroll 1
      for (int ch = 0; ch < 8; ++ch) {
        float x[8];
        if (valid) {
          const float4 v0 = lds_f4(qstg + (uint32_t)(((hf * 16 + 2 * ch) ^ (r & 31)) << 4));
          const float4 v1 = lds_f4(qstg + (uint32_t)(((hf * 16 + 2 * ch + 1) ^ (r & 31)) << 4));
          x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
          x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        uint32_t qv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) qv[e] = Elem<T>::pack(x[2 * e] * qscale, x[2 * e + 1] * qscale);
        const uint32_t off = (uint32_t)(hf * kRegion + r * 128 + ((ch ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_s + off), "r"(qv[0]), "r"(qv[1]),
                     "r"(qv[2]), "r"(qv[3])
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->q_ready));
    }

    float m_used = -INFINITY, l = 0.f;
    bool alive = true;  // false once a wait gave up: work stops, the pair barriers stay matched
    for (int j = 0; j < nb; ++j) {
      if (alive)
        alive = warp_wait_bar(smem_u32(&bars->s_full[j % kSBufs]), (uint32_t)((j / kSBufs) & 1), a.err, SITE_CHUNK_PIPE);
      tc_fence_after();
      const uint32_t scol = lane_base + (kColS * (uint32_t)(j % kSBufs));
      float sv[64];
      if (alive) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u[16];
          tmem_ld16(scol + hf * 64 + c * 16, u);
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[c * 16 + e] = __uint_as_float(u[e]);
        }
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = 0.f;
      }
      const int key0 = (j0 + j) * kBKV + hf * 64;
      if (key0 + 63 > pos) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key0 + c > pos) sv[c] = -INFINITY;
      }
      if (a.window > 0 && key0 <= pos - a.window) {  // keys at or before pos - W are outside the window
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key0 + c <= pos - a.window) sv[c] = -INFINITY;
      }
      float pm;
      {
        // eight independent chains, then combine
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
        for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
        pm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      // row maximum over both halves (double-buffered by block parity)
      red[((j & 1) * 2 + hf) * kBQ + r] = pm;
      pair_sync();
      const float mx = fmaxf(pm, red[((j & 1) * 2 + (hf ^ 1)) * kBQ + r]);
      const float m_new = fmaxf(m_used, mx);
      // taken on the first block with a visible key (m_used is -inf before it)
      const bool need = m_new > m_used + kRescale;
      const float sc = need ? exp2f(m_used - m_new) : 1.f;  // 0 while m_used is -inf
      // O holds earlier blocks once the row has seen a visible key (a finite
      // maximum, shared by both key halves; a half's own sum l may still be 0
      // when a window masked all of its keys so far): rescale this warp's
      // dimension half once the previous P.V has landed
      if (alive && __any_sync(0xffffffffu, need && m_used != -INFINITY)) {
        // P.V of block j - 1 has landed: o_done[(j - 1) % 2] completes once per
        // two blocks, and the P.V three blocks back is done (S_j followed it),
        // so this parity cannot alias
        alive = warp_wait_bar(smem_u32(&bars->o_done[(j - 1) & 1]), (uint32_t)(((j - 1) >> 1) & 1), a.err,
                              SITE_CHUNK_PIPE);
        if (alive) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t u[16];
            tmem_ld16(lane_base + kColO + hf * 64 + c * 16, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * sc);
            tmem_st16(lane_base + kColO + hf * 64 + c * 16, u);
          }
          tmem_wait_st();
        }
      }
      if (need) {
        l *= sc;
        m_used = m_new;
      }
      // P = 2^(S - m), 16-bit, two keys per column: this half's keys over
      // columns [hf*32, hf*32 + 32) of the S buffer; while no visible key has
      // been seen (a window that starts past this block) every P is 0
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(sv[c * 32 + 2 * e] - mref);
          const float p1 = fast_exp2(sv[c * 32 + 2 * e + 1] - mref);
          ls[e & 7] += p0 + p1;
          u[e] = Elem<T>::pack(p0, p1);
        }
        if (alive) tmem_st16(scol + hf * 32 + c * 16, u);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      if (alive) tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (alive && lane == 0) mbar_arrive(smem_u32(&bars->p_full[j % kSBufs]));
    }
    // ---- O / l -> output row (this warp's 64 dims) ----
    red[(2 * 2 + hf) * kBQ + r] = l;  // row sum over both halves
    pair_sync();
    const float lt = l + red[(2 * 2 + (hf ^ 1)) * kBQ + r];
    // O is final once every MMA has completed: mma_done completes once, after
    // the last P.V (o_done's parity cannot say that: with the last two P.V
    // still in flight, the phase of parity (nb - 1) & 1 two blocks back has
    // already completed)
    if (alive) alive = warp_wait_bar(smem_u32(&bars->mma_done), 0, a.err, SITE_CHUNK_PIPE);
    if (alive && part >= 0) {
      // one share of the tile's keys: O unnormalised, with the row's maximum
      // (base 2) and sum, for chunk_combine_kernel
      tc_fence_after();
      float* pp = a.partials + (((size_t)part * kBQ + r) * a.qh + hq) * (kD + 4);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[16];
        tmem_ld16(lane_base + kColO + hf * 64 + c * 16, u);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(pp + hf * 64 + c * 16);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]), __uint_as_float(u[4 * e + 2]),
                               __uint_as_float(u[4 * e + 3]));
      }
      if (hf == 0) *reinterpret_cast<float2*>(pp + kD) = make_float2(m_used, lt);
    } else if (alive) {
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      T* out = static_cast<T*>(a.out) + (size_t)(row0 + r) * a.ld_out + (size_t)hq * kD + hf * 64;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[16];
        tmem_ld16(lane_base + kColO + hf * 64 + c * 16, u);
        tmem_wait_ld();
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = Elem<T>::pack(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + c * 16);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<false>(tmem, kTmemCols);
  }
  // (run behind the decode attention kernel: the kernels after this one wait
  // for this grid only, so it completes after that one -- its last CTA alone
  // waits, every other CTA leaves its SM to the rest of the grid)
  if (a.wait_at_end && blockIdx.x == gridDim.x - 1) pdl_wait();
}

// ---- two query tiles per CTA ----------------------------------------------
// For launches with more (tile, head) units than the SMs hold at once: one
// CTA takes two query tiles of one head of one prompt (consecutive tiles of a
// chunk, or a chunk's odd last tile with an empty partner), which read the
// same keys.  Each K/V block is loaded once for both, and the two tiles'
// chains interleave on the tensor core: one tile's P.V and next S run while
// the softmax warps work on the other tile.  Tensor memory holds S_A, S_B,
// O_A, O_B (128 columns each, P written back over S); shared memory Q_A, Q_B,
// two K and two V stages.  Per tile the MMA thread issues P_j V_j and then
// S_{j+1} into the same S buffer (the MMAs of one thread run in issue order),
// so the barrier of S_{j+1} also says that P_j V_j has landed: the softmax
// rescales O without a wait of its own.  The later tile's last block is fully
// masked for the earlier one: its P is exactly 0 there, which leaves O and the
// row sum unchanged, so each tile's result is bit for bit the one-tile
// kernel's.  Full causal attention only (no window), whole key ranges.
constexpr int kStages2 = 2;
constexpr int kBarOff2 = 2 * kQBytes + 2 * kStages2 * kKVBytes;  // Q_A, Q_B, K stages, V stages
constexpr int kRedOff2 = kBarOff2 + 256;
// softmax exchange: maxima [tile][block parity][half][128], sums [tile][half][128]
constexpr int kSmem2 = 1024 + kRedOff2 + (8 + 4) * kBQ * 4;
constexpr uint32_t kColO2 = 2 * kColS;  // O_A at [256, 384), O_B at [384, 512)
static_assert(kSmem2 <= 227 * 1024, "shared memory per CTA");
static_assert(kStages2 * kKVBytes >= kBQ * kD * 4, "a tile's fp32 query rows are staged in the K (or the V) stages");

struct Bars2 {
  // K stage j % 2 is free once S_B(j) has landed, V stage j % 2 once P_B(j) V_j
  // has (the tile-A MMAs of a block are issued before tile B's)
  uint64_t k_full[kStages2], v_full[kStages2], k_free[kStages2], v_free[kStages2];
  uint64_t s_full[2], p_full[2];  // per tile: S_x(j) landed (phase j), P_x(j) written (8 warps)
  uint64_t q_ready, mma_done;
  uint32_t tmem_slot;
};
static_assert(sizeof(Bars2) <= 256, "barrier area");

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_tc2_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                          const ChunkAttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto q_reg = [&](int x) { return sbase + (uint32_t)(x * kQBytes); };
  auto k_reg = [&](int s) { return sbase + 2 * kQBytes + (uint32_t)(s * kKVBytes); };
  auto v_reg = [&](int s) { return sbase + 2 * kQBytes + (uint32_t)((kStages2 + s) * kKVBytes); };
  Bars2* bars = reinterpret_cast<Bars2*>(smem + kBarOff2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // one CTA per (tile pair, query head), heads fastest, pairs in the table's
  // order (most keys first)
  const int pair_i = blockIdx.x / a.qh;
  const int hq = blockIdx.x - pair_i * a.qh;
  const int G = a.qh / a.kvh;
  const int kh = hq / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->k_free[s]), 1);
      mbar_init(smem_u32(&bars->v_free[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars->s_full[x]), 1);
      mbar_init(smem_u32(&bars->p_full[x]), 8);
    }
    mbar_init(smem_u32(&bars->q_ready), 8);
    mbar_init(smem_u32(&bars->mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<false>(smem_u32(&bars->tmem_slot), kTmemCols);
    tmem_relinquish<false>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  if (!a.wait_at_end) pdl_wait();
  pdl_launch_dependents();
  // the pair's tiles: A, then B (B's rows may be 0: no second tile)
  const int4* tt = reinterpret_cast<const int4*>(a.tiles) + 4 * pair_i;
  const int4 ta = tt[0], ta2 = tt[1], tb = tt[2], tb2 = tt[3];
  const int32_t* bt = a.bt + ta.w;  // one prompt: one block table
  const int bt_len = ta2.x;
  const int n_keys = max(ta.y + ta.z, tb.y + tb.z);
  const int j0 = min(ta2.y, tb2.y);
  const int nb = max(ta2.z, tb2.z) - j0;

  if (warp == 0 || warp == 10) {
    // ---------------- producers: warp 0 K, warp 10 V ----------------
    // as in the one-tile kernel (lane 0 arms a free stage, lanes 0..7 issue a
    // block's sixteen boxes, pages read a group of four blocks ahead); both
    // rings start once the query rows staged in them have been taken
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_free : bars->v_free;
    if (lane == 0) tma_prefetch_desc(map);
    const int last_run = (n_keys - 1) / kRun;
    bool ok = (n_keys - 1) / a.page_size < bt_len;
    if (!ok && is_k && lane == 0) report(a.err, SAR_ERR_BOUNDS, SITE_CHUNK_BOUNDS, n_keys);
    const int g = lane & 7, sub = lane >> 3;
    auto page_of = [&](int jb, int& page, int& off) {
      const int key = min((j0 + jb + sub) * kRunsPerBlock + g, last_run) * kRun;
      const int bi = key / a.page_size;
      page = bt[bi];
      off = key - bi * a.page_size;
    };
    int pa = 0, oa = 0, pb = 0, ob = 0;
    if (ok) {
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&bars->q_ready), 0, a.err, SITE_CHUNK_PIPE);
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    if (ok) {
      page_of(0, pa, oa);
      if (nb > 4) page_of(4, pb, ob);
    }
    for (int j = 0; j < nb && ok; ++j) {
      const int i = j & 3;
      if (i == 0 && j > 0) {
        pa = pb;
        oa = ob;
        if (j + 4 < nb) page_of(j + 4, pb, ob);
      }
      const int s = j % kStages2;
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&empty[s]), (uint32_t)(((j / kStages2) & 1) ^ 1), a.err, SITE_CHUNK_PIPE);
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&full[s]);
      const uint32_t dst = is_k ? k_reg(s) : v_reg(s);
      if (lane == 0) mbar_expect_tx(fb, (uint32_t)kKVBytes);
      __syncwarp();
      int page = __shfl_sync(0xffffffffu, pa, (i << 3) | g);
      const int po = __shfl_sync(0xffffffffu, oa, (i << 3) | g);
      if (lane < kRunsPerBlock) {
        if (page < 0 || page >= a.num_pages) {
          report(a.err, SAR_ERR_BOUNDS, SITE_CHUNK_BOUNDS, page);
          page = 0;
        }
        const int row = (page * a.kvh + kh) * a.page_size + po;
        tma_load_2d(dst + g * (kRun * 128), map, 0, row, fb);
        tma_load_2d(dst + kRegion + g * (kRun * 128), map, 64, row, fb);
      }
    }
    // no copy may still be in flight when the CTA leaves
    if (lane == 0) {
      const int first = max(0, nb - kStages2);
      for (int j = first; j < nb && ok; ++j)
        ok = mbar_wait(smem_u32(&empty[j % kStages2]), (uint32_t)((j / kStages2) & 1), a.err, SITE_CHUNK_PIPE);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t fmt = Elem<T>::kMmaFormat;
      const uint32_t id_s = idesc_128x128(fmt, 0), id_pv = idesc_128x128(fmt, 1);
      const uint64_t dqa = sw128_desc(q_reg(0)), dqb = sw128_desc(q_reg(1));
      const uint64_t dk0 = sw128_desc(k_reg(0)), dk1 = sw128_desc(k_reg(1));
      const uint64_t dv0 = sw128_desc_mn(v_reg(0), kRegion, 1024), dv1 = sw128_desc_mn(v_reg(1), kRegion, 1024);
      bool ok = mbar_wait(smem_u32(&bars->q_ready), 0, a.err, SITE_CHUNK_PIPE);
      // S_x(j) = Q_x K_j^T into S buffer x; tile B's also frees K stage j % 2
      auto issue_s = [&](int x, int j) -> bool {
        const int s = j % kStages2;
        if (x == 0 && !mbar_wait(smem_u32(&bars->k_full[s]), (uint32_t)((j / kStages2) & 1), a.err, SITE_CHUNK_PIPE))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + kColS * (uint32_t)x;
        const uint64_t db = s ? dk1 : dk0;
        const uint64_t dq = x ? dqb : dqa;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t o = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
          mma_f16<false>(d, dq + o, db + o, id_s, kk != 0);
        }
        mma_commit(smem_u32(&bars->s_full[x]));
        if (x == 1) mma_commit(smem_u32(&bars->k_free[s]));
        return true;
      };
      // O_x += P_x(j) V_j; tile B's also frees V stage j % 2
      auto issue_pv = [&](int x, int j) -> bool {
        if (!mbar_wait(smem_u32(&bars->p_full[x]), (uint32_t)(j & 1), a.err, SITE_CHUNK_PIPE)) return false;
        const int s = j % kStages2;
        if (x == 0 && !mbar_wait(smem_u32(&bars->v_full[s]), (uint32_t)((j / kStages2) & 1), a.err, SITE_CHUNK_PIPE))
          return false;
        tc_fence_after();
        const uint32_t pcol = tmem + kColS * (uint32_t)x;
        const uint32_t dO = tmem + kColO2 + kColS * (uint32_t)x;
        const uint64_t dvs = s ? dv1 : dv0;
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)
          mma_f16_ts(dO, pcol + kk * 8, dvs + (uint64_t)(kk * (16 * 128 / 16)), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
        if (x == 1) mma_commit(smem_u32(&bars->v_free[s]));
        return true;
      };
      if (ok) ok = issue_s(0, 0);
      if (ok) ok = issue_s(1, 0);
      for (int j = 0; j < nb && ok; ++j) {
        if (!(ok = issue_pv(0, j))) break;
        if (j + 1 < nb && !(ok = issue_s(0, j + 1))) break;
        if (!(ok = issue_pv(1, j))) break;
        if (j + 1 < nb && !(ok = issue_s(1, j + 1))) break;
      }
      // every MMA issued has completed before tensor memory is released
      mma_commit(smem_u32(&bars->mma_done));
      mbar_wait(smem_u32(&bars->mma_done), 0, a.err, SITE_CHUNK_PIPE);
    }
    __syncwarp();
  } else {
    // ---------------- softmax / epilogue ----------------
    // warps 2..9 as in the one-tile kernel (row quarter qq, key half hf),
    // each taking tile A then tile B of every block
    const int qq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = qq * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kRedOff2);
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + qq) : "memory"); };
    // tile x's rows, first batch row and this thread's position (selects, not
    // an indexed array, so that they stay in registers)
    auto rows_x = [&](int x) { return x ? tb.z : ta.z; };
    auto row0_x = [&](int x) { return x ? tb.x : ta.x; };
    auto pos_x = [&](int x) { return (x ? tb.y : ta.y) + r; };
    {
      // both tiles' fp32 query rows, A's through the K stages and B's through
      // the V stages (idle until Q is ready), then scaled and rounded into
      // Q_A and Q_B as the one-tile kernel does
      const float qscale = rsqrtf((float)kD) * 1.4426950408889634f;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const uint32_t qstg = (x ? v_reg(0) : k_reg(0)) + (uint32_t)(r * 512);
        if (r < rows_x(x)) {
          const float* qp = a.q32 + (size_t)(row0_x(x) + r) * a.ld32 + (size_t)hq * kD + hf * 64;
#pragma unroll
          for (int cc = 0; cc < 16; ++cc)
            cp_async16(qstg + (uint32_t)((((hf * 16 + cc) ^ (r & 31))) << 4), qp + cc * 4, 16);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
#pragma unroll 1
      for (int x = 0; x < 2; ++x) {
        const uint32_t qstg = (x ? v_reg(0) : k_reg(0)) + (uint32_t)(r * 512);
        const bool valid = r < rows_x(x);
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          float q8[8];
          if (valid) {
            const float4 v0 = lds_f4(qstg + (uint32_t)(((hf * 16 + 2 * ch) ^ (r & 31)) << 4));
            const float4 v1 = lds_f4(qstg + (uint32_t)(((hf * 16 + 2 * ch + 1) ^ (r & 31)) << 4));
            q8[0] = v0.x; q8[1] = v0.y; q8[2] = v0.z; q8[3] = v0.w;
            q8[4] = v1.x; q8[5] = v1.y; q8[6] = v1.z; q8[7] = v1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q8[e] = 0.f;
          }
          uint32_t qv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) qv[e] = Elem<T>::pack(q8[2 * e] * qscale, q8[2 * e + 1] * qscale);
          const uint32_t off = (uint32_t)(hf * kRegion + r * 128 + ((ch ^ (r & 7)) << 4));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_reg(x) + off), "r"(qv[0]), "r"(qv[1]),
                       "r"(qv[2]), "r"(qv[3])
                       : "memory");
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->q_ready));
    }

    float m_a = -INFINITY, l_a = 0.f, m_b = -INFINITY, l_b = 0.f;
    bool alive = true;
    // the online softmax of tile x over block j (the one-tile kernel's steps)
    auto softmax_block = [&](int x, int j, float& m_used, float& l) {
      if (alive) alive = warp_wait_bar(smem_u32(&bars->s_full[x]), (uint32_t)(j & 1), a.err, SITE_CHUNK_PIPE);
      tc_fence_after();
      const uint32_t scol = lane_base + kColS * (uint32_t)x;
      const int pos = pos_x(x);
      float sv[64];
      if (alive) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u[16];
          tmem_ld16(scol + hf * 64 + c * 16, u);
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[c * 16 + e] = __uint_as_float(u[e]);
        }
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = 0.f;
      }
      const int key0 = (j0 + j) * kBKV + hf * 64;
      if (key0 + 63 > pos) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key0 + c > pos) sv[c] = -INFINITY;
      }
      float pm;
      {
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
        for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
        pm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      float* rm = red + ((x * 2 + (j & 1)) * 2) * kBQ;
      rm[hf * kBQ + r] = pm;
      pair_sync();
      const float mx = fmaxf(pm, rm[(hf ^ 1) * kBQ + r]);
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + kRescale;
      const float sc = need ? exp2f(m_used - m_new) : 1.f;
      // P_x(j - 1) V_(j - 1) completed before S_x(j) (issued after it), whose
      // barrier this warp has passed: O_x may be rescaled at once
      if (alive && __any_sync(0xffffffffu, need && m_used != -INFINITY)) {
        const uint32_t ocol = lane_base + kColO2 + kColS * (uint32_t)x;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t u[16];
          tmem_ld16(ocol + hf * 64 + c * 16, u);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * sc);
          tmem_st16(ocol + hf * 64 + c * 16, u);
        }
        tmem_wait_st();
      }
      if (need) {
        l *= sc;
        m_used = m_new;
      }
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(sv[c * 32 + 2 * e] - mref);
          const float p1 = fast_exp2(sv[c * 32 + 2 * e + 1] - mref);
          ls[e & 7] += p0 + p1;
          u[e] = Elem<T>::pack(p0, p1);
        }
        if (alive) tmem_st16(scol + hf * 32 + c * 16, u);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      if (alive) tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (alive && lane == 0) mbar_arrive(smem_u32(&bars->p_full[x]));
    };
    for (int j = 0; j < nb; ++j) {
      softmax_block(0, j, m_a, l_a);
      softmax_block(1, j, m_b, l_b);
    }
    // ---- O / l -> output rows (this warp's 64 dims of each tile) ----
    float* rs = red + 8 * kBQ;
    rs[(0 * 2 + hf) * kBQ + r] = l_a;
    rs[(1 * 2 + hf) * kBQ + r] = l_b;
    pair_sync();
    const float lt_a = l_a + rs[(0 * 2 + (hf ^ 1)) * kBQ + r], lt_b = l_b + rs[(1 * 2 + (hf ^ 1)) * kBQ + r];
    if (alive) alive = warp_wait_bar(smem_u32(&bars->mma_done), 0, a.err, SITE_CHUNK_PIPE);
    if (alive) {
      tc_fence_after();
#pragma unroll 1
      for (int x = 0; x < 2; ++x) {
        const bool valid = r < rows_x(x);
        const float lt = x ? lt_b : lt_a;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        T* out = static_cast<T*>(a.out) + (size_t)(row0_x(x) + r) * a.ld_out + (size_t)hq * kD + hf * 64;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t u[16];
          tmem_ld16(lane_base + kColO2 + kColS * (uint32_t)x + hf * 64 + c * 16, u);
          tmem_wait_ld();
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = Elem<T>::pack(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + c * 16);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<false>(tmem, kTmemCols);
  }
  if (a.wait_at_end && blockIdx.x == gridDim.x - 1) pdl_wait();
}

// Merges the shares of a split tile: out = sum_i O_i 2^(m_i - M) / sum_i l_i 2^(m_i - M)
// per (row, head, dim); a share with no visible key has m = -inf and weighs 0.
template <typename T>
__global__ void chunk_combine_kernel(const float* __restrict__ partials, const int32_t* __restrict__ comb, void* out,
                                     int ld_out, int qh) {
  pdl_wait();
  pdl_launch_dependents();
  const int4 c = reinterpret_cast<const int4*>(comb)[blockIdx.x];  // first row, rows, first slot, slots
  const int r = blockIdx.y, hq = blockIdx.z, d = threadIdx.x;
  if (r >= c.y) return;
  auto rec = [&](int i) { return partials + (((size_t)(c.z + i) * kBQ + r) * qh + hq) * (kD + 4); };
  float M = -INFINITY;
  for (int i = 0; i < c.w; ++i) M = fmaxf(M, rec(i)[kD]);
  float L = 0.f, A = 0.f;
  for (int i = 0; i < c.w; ++i) {
    const float* p = rec(i);
    const float sc = (p[kD] == -INFINITY) ? 0.f : exp2f(p[kD] - M);
    L = fmaf(p[kD + 1], sc, L);
    A = fmaf(p[d], sc, A);
  }
  static_cast<T*>(out)[(size_t)(c.x + r) * ld_out + (size_t)hq * kD + d] = Elem<T>::from(L > 0.f ? A / L : 0.f);
}

template <typename T>
int launch_t(const ChunkAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
  cudaError_t e;
  if (a.dual) {
    const int arc = ensure_smem_attr(reinterpret_cast<const void*>(&chunk_attn_tc2_kernel<T>), kSmem2,
                                     "chunk attention (tcgen05, two tiles) attribute");
    if (arc != SAR_OK) return arc;
    e = launch_pdl(chunk_attn_tc2_kernel<T>, dim3(a.n_tiles / 2 * a.qh), dim3(kThreads), (size_t)kSmem2, s, tmk,
                   tmv, a);
  } else {
    const int arc = ensure_smem_attr(reinterpret_cast<const void*>(&chunk_attn_tc_kernel<T>), kSmem,
                                     "chunk attention (tcgen05) attribute");
    if (arc != SAR_OK) return arc;
    e = launch_pdl(chunk_attn_tc_kernel<T>, dim3(a.n_tiles * a.qh), dim3(kThreads), (size_t)kSmem, s, tmk, tmv, a);
  }
  if (e != cudaSuccess) return cuda_error(e, "chunk attention (tcgen05) launch");
  count_launches(1);
  if (a.n_comb > 0) {
    e = launch_pdl(chunk_combine_kernel<T>, dim3(a.n_comb, kBQ, a.qh), dim3(kD), 0, s, a.partials, a.comb, a.out,
                   a.ld_out, a.qh);
    if (e != cudaSuccess) return cuda_error(e, "chunk combine launch");
    count_launches(1);
  }
  return SAR_OK;
}

}  // namespace

bool chunk_attention_tc_supported(const ChunkAttnArgs& a) {
  return a.d == kD && a.page_size % kRun == 0 && a.qh % a.kvh == 0 && a.window >= 0;
}

int launch_chunk_attention_tc(const ChunkAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              cudaStream_t s) {
  if (a.n_tiles <= 0) return SAR_OK;
  if (!chunk_attention_tc_supported(a))
    return set_error(SAR_ERR_UNSUPPORTED, "chunk attention (tcgen05): head_dim 128, pages of a multiple of 16 keys");
  if ((reinterpret_cast<uintptr_t>(a.q32) & 15) || (a.ld32 & 3) || (reinterpret_cast<uintptr_t>(a.out) & 15) ||
      (a.ld_out & 7))
    return set_error(SAR_ERR_INVALID_ARG, "chunk attention (tcgen05): misaligned query or output rows");
  if (a.n_comb > 0 && (!a.partials || !a.comb || (reinterpret_cast<uintptr_t>(a.partials) & 15)))
    return set_error(SAR_ERR_INVALID_ARG, "chunk attention (tcgen05): split tiles without a partials buffer");
  if (a.dual && (a.n_tiles % 2 || a.n_comb > 0 || a.window > 0))
    return set_error(SAR_ERR_INVALID_ARG, "chunk attention (tcgen05): tile pairs need an even table, no splits, no window");
  return a.storage == SAR_STORAGE_BF16 ? launch_t<__nv_bfloat16>(a, tmk, tmv, s) : launch_t<__half>(a, tmk, tmv, s);
}

}  // namespace sar
