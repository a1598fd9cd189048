// Paged decode attention: every decode row's query heads against that
// request's own paged K/V history (the "Decode uses PagedAttention" half of
// the split, SARATHI technique write-up section 3.3; reading notes part 2
// section 3: "each decode looks up its own history KV").
//
// HBM-bound (about 4 flops per byte), so the design is about streaming pages
// with as few instructions per byte as possible:
//   * one CTA = (work item, KV head); a work item is a range of a decode's
//     keys (long contexts are split so every SM has work, then merged);
//   * each of the 4 warps owns a private ring of 16-key blocks; one lane
//     fills a block with 2-D TMA tensor loads of the page (64-dimension boxes,
//     128-byte swizzle, so the ldmatrix reads below are bank-conflict free);
//   * the query heads of one GQA group (up to 8) are the rows of a 16-row MMA
//     tile: S = Q K^T and O += P V run on warp-level tensor-core MMAs
//     (m16n8k16, fp32 accumulate), 48 per 16-key block; the fp32 queries enter
//     as a high and a low 16-bit part so the scores keep fp32-like precision;
//   * online softmax in base 2 on the accumulator fragments; the 4 warps'
//     (max, sum, acc) are merged in shared memory; split items write
//     unnormalised partials that decode_combine_kernel merges;
//   * with a sliding window the host plans each decode's ranges from the
//     16-key block holding its oldest visible key; keys below that key are
//     masked (every block still holds at least one visible key).
#include <cuda.h>
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace sar {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;    // per-warp ring depth (16-key blocks)
constexpr int kBlockKeys = 16;
constexpr int kMaxGroup = 8;  // query heads per KV head (rows of the MMA tile that are real)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (Elem<T>::kMmaFormat == 1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Byte offset of (key row, 16-byte chunk over the whole head_dim) inside one
// TMA-filled block: 64-dimension halves of 16 rows x 128 bytes, each written
// with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t blk_off(int row, int chunk) {
  const int h = chunk >> 3, c = chunk & 7;
  return (uint32_t)(h * (kBlockKeys * 128) + row * 128 + ((c ^ (row & 7)) << 4));
}

// COMPUTED = false: work items come from the host-planned list `a.items`.
// COMPUTED = true: CTA x covers split (x % max_splits) of decode (x / max_splits)
// with fixed `split_keys` ranges and a padded [n_decode][bt_stride] block table.
template <typename T, int D, bool COMPUTED = false>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       DecodeAttnArgs a) {
  constexpr int HALVES = D / 64;
  constexpr int BLK_BYTES = HALVES * kBlockKeys * 128;  // K (or V) of one 16-key block
  constexpr int STAGE_BYTES = 2 * BLK_BYTES;
  constexpr int NT = D / 8;                             // output n-tiles of 8 dimensions
  constexpr int KT = D / 16;                            // k-steps over head_dim

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * kStages * STAGE_BYTES;
  // after the key loop each warp's own ring holds its [row][D + 2] merge record
  static_assert(kMaxGroup * (D + 2) * 4 <= kStages * STAGE_BYTES, "merge record must fit the ring");
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * STAGE_BYTES) + warp * kStages;
  pdl_wait();
  pdl_launch_dependents();

  int b, kbeg, kend, part, btlen;
  int wlo = 0;  // oldest key inside the sliding window
  const int* bt;
  if constexpr (COMPUTED) {
    b = blockIdx.x / a.max_splits;
    const int sidx = blockIdx.x - b * a.max_splits;
    const int nk = a.ctx_lens[b] + 1;
    if (nk < 1 || nk > a.max_splits * a.split_keys) {
      if (threadIdx.x == 0 && sidx == 0) report(a.err, SAR_ERR_BOUNDS, SITE_DECODE_BOUNDS, nk);
      return;
    }
    kbeg = sidx * a.split_keys;
    if (kbeg >= nk) return;
    kend = min(nk, kbeg + a.split_keys);
    part = nk > a.split_keys ? b * a.max_splits + sidx : -1;
    bt = a.bt + (size_t)b * a.bt_stride;
    btlen = a.bt_stride;
  } else {
    // planned items, KV head fastest, so the launch order is the plan's order
    // (full key ranges first, the shorter remainders last, for a short drain)
    const int4 item = reinterpret_cast<const int4*>(a.items)[blockIdx.x / a.kvh];
    b = item.x;
    kbeg = item.y;
    kend = item.z;
    part = item.w;
    bt = a.bt + a.bt_off[b];
    btlen = a.bt_len[b];
    if (a.window > 0) wlo = max(0, a.nkeys[b] - a.window);
  }
  const int kh = COMPUTED ? (int)blockIdx.y : (int)(blockIdx.x % a.kvh);
  const int G = a.qh / a.kvh;
  const int nblk = (kend - kbeg + kBlockKeys - 1) / kBlockKeys;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncwarp();

  // Issue block `j` of this CTA's range into stage s (lane 0 only).
  // Page of this CTA's block j (-1 past the block table).
  auto page_of = [&](int j) -> int {
    const int bi = (kbeg + j * kBlockKeys) / a.page_size;
    return (bi < btlen) ? bt[bi] : -1;
  };
  // Issue block `j` (its page looked up beforehand) into stage s (lane 0 only).
  auto issue = [&](int j, int s, int page) -> bool {
    const int key0 = kbeg + j * kBlockKeys;
    const int bi = key0 / a.page_size;
    if (page < 0 || page >= a.num_pages) {
      report(a.err, SAR_ERR_BOUNDS, SITE_DECODE_BOUNDS, key0);
      return false;
    }
    const int row = (page * a.kvh + kh) * a.page_size + (key0 - bi * a.page_size);
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t dst = smem_u32(ring + s * STAGE_BYTES);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, STAGE_BYTES);
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
      tma_load_2d(dst + h * kBlockKeys * 128, &tmk, h * 64, row, bar);
      tma_load_2d(dst + BLK_BYTES + h * kBlockKeys * 128, &tmv, h * 64, row, bar);
    }
    return true;
  };

  // first pages in flight before the query loads, so their latencies overlap;
  // the block-table entry of the next block to issue is read one block ahead
  const int my_n = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
  bool ok = true;
  int issued = 0, consumed = 0;
  int next_page = -1;
  if (lane == 0) {
    int first[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) first[i] = i < my_n ? page_of(warp + i * kWarps) : -1;
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      if (i < my_n && ok) {
        ok = issue(warp + i * kWarps, i, first[i]);
        if (ok) ++issued;
      }
    }
    if (kStages < my_n) next_page = page_of(warp + kStages * kWarps);
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;

  // ---- query fragments: rows = the group's heads (zero rows pad to 16), split hi + lo ----
  const int g = lane >> 2, c4 = lane & 3;
  const float qscale = rsqrtf((float)D) * 1.4426950408889634f;  // softmax in base 2
  uint32_t qh[KT][2], ql[KT][2];  // registers a0 and a2 of the A fragment; a1, a3 (rows 8..15) are zero
#pragma unroll
  for (int kk = 0; kk < KT; ++kk) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int col = kk * 16 + r * 8 + 2 * c4;
      float x0 = 0.f, x1 = 0.f;
      if (g < G) {
        if (a.q32) {
          const float* qp = a.q32 + (size_t)b * a.ld32 + (size_t)(kh * G + g) * D + col;
          x0 = qp[0] * qscale;
          x1 = qp[1] * qscale;
        } else {
          const T* qp = static_cast<const T*>(a.qkv) + (size_t)b * a.ld + (size_t)(kh * G + g) * D + col;
          x0 = Elem<T>::to(qp[0]) * qscale;
          x1 = Elem<T>::to(qp[1]) * qscale;
        }
      }
      const uint32_t hi = Elem<T>::pack(x0, x1);
      qh[kk][r] = hi;
      ql[kk][r] = Elem<T>::pack(x0 - Elem<T>::lo(hi), x1 - Elem<T>::hi(hi));
    }
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_part = 0.f;  // for query row g (this lane's share of the sum)


  for (int i = 0; i < my_n && ok; ++i) {
    const int s = i % kStages;
    const uint32_t par = (uint32_t)((i / kStages) & 1);
    int got = 0;
    if (lane == 0) got = mbar_wait(smem_u32(&bars[s]), par, a.err, SITE_DECODE_PIPE) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got) {
      ok = false;
      break;
    }
    ++consumed;
    const int j = warp + i * kWarps;
    const int nk = min(kBlockKeys, kend - (kbeg + j * kBlockKeys));
    const int nlo = wlo - (kbeg + j * kBlockKeys);  // keys of this block below it are outside the window
    const uint32_t kb = smem_u32(ring + s * STAGE_BYTES);
    const uint32_t vb = kb + BLK_BYTES;
    const int mi = lane >> 3;

    // ---- S = Q K^T: 16 rows x 16 keys ----
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < KT; kk += 2) {
#pragma unroll
      for (int jn = 0; jn < 2; ++jn) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + blk_off(jn * 8 + (lane & 7), kk * 2 + mi), b0, b1, b2, b3);
        mma16816<T>(sc[jn], qh[kk][0], 0u, qh[kk][1], 0u, b0, b1);
        mma16816<T>(sc[jn], ql[kk][0], 0u, ql[kk][1], 0u, b0, b1);
        mma16816<T>(sc[jn], qh[kk + 1][0], 0u, qh[kk + 1][1], 0u, b2, b3);
        mma16816<T>(sc[jn], ql[kk + 1][0], 0u, ql[kk + 1][1], 0u, b2, b3);
      }
    }
    // ---- online softmax for row g over keys jn*8 + 2*c4 + e ----
    float mx = -INFINITY;
#pragma unroll
    for (int jn = 0; jn < 2; ++jn)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kk = jn * 8 + 2 * c4 + e;
        if (kk >= nk || kk < nlo) sc[jn][e] = -INFINITY;
        mx = fmaxf(mx, sc[jn][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m_run, mx);  // finite: every block has at least one key
    const float alpha = exp2f(m_run - mn);
    m_run = mn;
    const float p00 = exp2f(sc[0][0] - mn), p01 = exp2f(sc[0][1] - mn);
    const float p10 = exp2f(sc[1][0] - mn), p11 = exp2f(sc[1][1] - mn);
    l_part = l_part * alpha + (p00 + p01 + p10 + p11);
    const uint32_t pa0 = Elem<T>::pack(p00, p01), pa2 = Elem<T>::pack(p10, p11);
    // ---- O = O * alpha + P V ----
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= alpha;
      o[n][1] *= alpha;
    }
#pragma unroll
    for (int n = 0; n < NT; n += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + blk_off((mi & 1) * 8 + (lane & 7), n + (mi >> 1)), b0, b1, b2, b3);
      mma16816<T>(o[n], pa0, 0u, pa2, 0u, b0, b1);
      mma16816<T>(o[n + 1], pa0, 0u, pa2, 0u, b2, b3);
    }
    __syncwarp();
    if (i + kStages < my_n) {
      int r = 1;
      if (lane == 0) {
        r = issue(warp + (i + kStages) * kWarps, s, next_page) ? 1 : 0;
        issued += r;
        if (i + kStages + 1 < my_n) next_page = page_of(warp + (i + kStages + 1) * kWarps);
      }
      if (!__shfl_sync(0xffffffffu, r, 0)) ok = false;
    }
  }
  // never leave with copies in flight: wait (bounded) for any not consumed
  if (lane == 0) {
    for (int i = consumed; i < issued; ++i)
      mbar_wait(smem_u32(&bars[i % kStages]), (uint32_t)((i / kStages) & 1), a.err, SITE_DECODE_PIPE);
  }
  __syncwarp();

  // ---- per-warp row state into shared memory, then merge the 4 warps ----
  float lsum = l_part;
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  float* my = reinterpret_cast<float*>(ring);
  if (g < G) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      my[g * (D + 2) + n * 8 + 2 * c4] = o[n][0];
      my[g * (D + 2) + n * 8 + 2 * c4 + 1] = o[n][1];
    }
    if (c4 == 0) {
      my[g * (D + 2) + D] = m_run;
      my[g * (D + 2) + D + 1] = lsum;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, dd = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + w * kStages * STAGE_BYTES)[h * (D + 2) + D]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* src = reinterpret_cast<const float*>(smem + w * kStages * STAGE_BYTES) + h * (D + 2);
      const float sc = (src[D] == -INFINITY) ? 0.f : exp2f(src[D] - M);
      L = fmaf(src[D + 1], sc, L);
      A = fmaf(src[dd], sc, A);
    }
    const int hq = kh * G + h;
    if (part < 0) {
      static_cast<T*>(a.out)[(size_t)b * a.ld_out + (size_t)hq * D + dd] = Elem<T>::from(A / L);
    } else {
      float* pp = a.partials + ((size_t)part * a.qh + hq) * (D + 2);
      pp[dd] = A;
      if (dd == 0) {
        pp[D] = M;
        pp[D + 1] = L;
      }
    }
  }
}

// Merges the split partial results of each decode: out = sum_i A_i 2^(m_i - M) / sum_i L_i 2^(m_i - M).
template <typename T, int D, bool COMPUTED = false>
__global__ void decode_combine_kernel(DecodeAttnArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int hq = blockIdx.y;
  int cnt, p0;
  if constexpr (COMPUTED) {
    cnt = (a.ctx_lens[b] + a.split_keys) / a.split_keys;  // ceil((ctx + 1) / split)
    if (cnt > a.max_splits || cnt < 1) return;           // flagged by the attention kernel
    p0 = b * a.max_splits;
  } else {
    cnt = a.parts_count[b];
    p0 = a.parts_begin[b];
  }
  if (cnt <= 1) return;
  const int dd = threadIdx.x;
  // partials four at a time, their loads in flight together, merged online
  float M = -INFINITY, L = 0.f, A = 0.f;
  for (int i0 = 0; i0 < cnt; i0 += 4) {
    float pm[4], pl[4], pa[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool v = i0 + u < cnt;
      const float* pp = a.partials + ((size_t)(p0 + (v ? i0 + u : 0)) * a.qh + hq) * (D + 2);
      pm[u] = v ? pp[D] : -INFINITY;
      pl[u] = v ? pp[D + 1] : 0.f;
      pa[u] = v ? pp[dd] : 0.f;
    }
    const float mn = fmaxf(fmaxf(M, fmaxf(pm[0], pm[1])), fmaxf(pm[2], pm[3]));
    const float rs = M == -INFINITY ? 0.f : exp2f(M - mn);
    L *= rs;
    A *= rs;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float sc = pm[u] == -INFINITY ? 0.f : exp2f(pm[u] - mn);
      L = fmaf(pl[u], sc, L);
      A = fmaf(pa[u], sc, A);
    }
    M = mn;
  }
  static_cast<T*>(a.out)[(size_t)b * a.ld_out + (size_t)hq * D + dd] = Elem<T>::from(A / L);
}

template <typename T, int D, bool COMPUTED = false>
int launch_impl(const DecodeAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
  constexpr int STAGE_BYTES = 2 * (D / 64) * kBlockKeys * 128;
  const size_t smem = 1024 + (size_t)kWarps * kStages * STAGE_BYTES + (size_t)kWarps * kStages * 8;
  const int arc = ensure_smem_attr(reinterpret_cast<const void*>(&decode_attn_kernel<T, D, COMPUTED>), (int)smem,
                                   "decode attention attribute");
  if (arc != SAR_OK) return arc;
  const int n_ctas = COMPUTED ? a.n_decode * a.max_splits : a.n_items;
  const dim3 grid = COMPUTED ? dim3(n_ctas, a.kvh) : dim3(n_ctas * a.kvh);
  launch_pdl(decode_attn_kernel<T, D, COMPUTED>, grid, dim3(kWarps * 32), smem, s, tmk, tmv, a);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "decode attention launch");
  if (a.partials && !a.defer_combine) {
    launch_pdl(decode_combine_kernel<T, D, COMPUTED>, dim3(a.n_decode, a.qh), dim3(D), 0, s, a);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "decode combine launch");
  }
  return SAR_OK;
}

template <bool COMPUTED>
int dispatch(const DecodeAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
  const bool bf = a.storage == SAR_STORAGE_BF16;
  if (a.d == 128) return bf ? launch_impl<__nv_bfloat16, 128, COMPUTED>(a, tmk, tmv, s)
                            : launch_impl<__half, 128, COMPUTED>(a, tmk, tmv, s);
  if (a.d == 64) return bf ? launch_impl<__nv_bfloat16, 64, COMPUTED>(a, tmk, tmv, s)
                           : launch_impl<__half, 64, COMPUTED>(a, tmk, tmv, s);
  return set_error(SAR_ERR_UNSUPPORTED, "decode attention: head_dim must be 64 or 128");
}

}  // namespace

int make_kv_tmap(CUtensorMap* map, const void* pages, int num_pages, int kvh, int page_size, int head_dim,
                 int storage) {
  // rows = (page, head, slot) triples, columns = head_dim; boxes of 16 slots x 64 dimensions
  return make_tmap_16(map, pages, (uint64_t)num_pages * kvh * page_size, head_dim, kBlockKeys, storage);
}

int launch_decode_combine(const DecodeAttnArgs& a, cudaStream_t s) {
  if (a.n_items <= 0 || !a.partials) return SAR_OK;
  const bool bf = a.storage == SAR_STORAGE_BF16;
  if (a.d == 128)
    launch_pdl(bf ? decode_combine_kernel<__nv_bfloat16, 128> : decode_combine_kernel<__half, 128>,
               dim3(a.n_decode, a.qh), dim3(128), 0, s, a);
  else if (a.d == 64)
    launch_pdl(bf ? decode_combine_kernel<__nv_bfloat16, 64> : decode_combine_kernel<__half, 64>,
               dim3(a.n_decode, a.qh), dim3(64), 0, s, a);
  else
    return set_error(SAR_ERR_UNSUPPORTED, "decode combine: head_dim must be 64 or 128");
  count_launches(1);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SAR_OK : cuda_error(e, "decode combine launch");
}

int launch_decode_attention(const DecodeAttnArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                            cudaStream_t s) {
  if (a.n_items <= 0) return SAR_OK;
  const int G = a.qh / a.kvh;
  if (a.qh % a.kvh || G > kMaxGroup || (a.d != 64 && a.d != 128) || a.page_size % kBlockKeys)
    return set_error(SAR_ERR_UNSUPPORTED, "decode attention: head_dim 64/128, group <= 8, page % 16");
  return dispatch<false>(a, tmk, tmv, s);
}

}  // namespace sar

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs while another
// component is capturing a CUDA graph on the same stream, runtimes that hand
// out a fixed memory budget up front and own every allocation, or hosts that
// forbid allocation on the serving path.  This variant keeps the split
// partial results in a file-scope device array of fixed size instead of the
// model's workspace, and plans the key splits on the device instead of
// shipping a host-planned list, so it needs neither a device allocation nor a
// pinned staging buffer.  The array exists on every GPU that loads the
// library, until the process exits.
// ---------------------------------------------------------------------------

namespace sar {
namespace {

constexpr size_t kStaticScratchFloats = size_t(2) << 20;  // 8 MiB of fp32 partials
static __device__ __align__(256) float g_decode_scratch[kStaticScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_addr[256] = {};  // per device: device address of g_decode_scratch

}  // namespace
}  // namespace sar

extern "C" int sar_decode_attention_noalloc(const void* q, int32_t q_stride, const void* k_pages,
                                            const void* v_pages, int32_t num_pages, int32_t page_size,
                                            int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                            int32_t n_decode, const int32_t* ctx_lens, int32_t max_ctx,
                                            const int32_t* block_tables, int32_t bt_stride, void* out,
                                            int32_t out_stride, int32_t storage, int32_t* err_flag,
                                            void* stream) {
  using namespace sar;
  if (!q || !k_pages || !v_pages || !ctx_lens || !block_tables || !out)
    return set_error(SAR_ERR_INVALID_ARG, "decode_attention_noalloc: null pointer");
  if (n_decode <= 0 || max_ctx < 0 || num_pages <= 0 || bt_stride <= 0 || n_kv_heads <= 0 || page_size <= 0 ||
      n_q_heads % n_kv_heads || (int64_t)(max_ctx / page_size + 1) > bt_stride)
    return set_error(SAR_ERR_INVALID_ARG, "decode_attention_noalloc: bad sizes or block table too short");
  const bool q_f32 = (storage & SAR_Q_F32) != 0;  // query rows in fp32 (q_stride in floats)
  storage &= ~SAR_Q_F32;
  if ((head_dim != 64 && head_dim != 128) || page_size % kBlockKeys || n_q_heads / n_kv_heads > 8 ||
      q_stride < n_q_heads * head_dim || out_stride < n_q_heads * head_dim)
    return set_error(SAR_ERR_UNSUPPORTED, "decode_attention_noalloc: shape not supported");
  if (storage != SAR_STORAGE_F16 && storage != SAR_STORAGE_BF16)
    return set_error(SAR_ERR_INVALID_ARG, "decode_attention_noalloc: bad storage");
  // split length: the smallest power of two in [256, 4096] keys whose partials
  // fit the static array; longer contexts are always split (so use the array)
  const int64_t per_split = (int64_t)n_decode * n_q_heads * (head_dim + 2);
  auto need = [&](int64_t sp) {
    const int64_t ns = ((int64_t)max_ctx + sp) / sp;  // ceil((max_ctx + 1) / sp)
    return ns > 1 ? ns * per_split : 0;
  };
  int64_t split = 256;
  while (split < 4096 && need(split) > (int64_t)kStaticScratchFloats) split *= 2;
  if (need(split) > (int64_t)kStaticScratchFloats)
    return set_error(SAR_ERR_INVALID_ARG, "decode_attention_noalloc: partials exceed the 8 MiB static scratch");
  const int64_t max_splits = ((int64_t)max_ctx + split) / split;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "decode_attention_noalloc: current device");
  if (dev < 0 || dev >= 256) return set_error(SAR_ERR_UNSUPPORTED, "decode_attention_noalloc: device index");
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_decode_scratch);  // once per device, with it current
      if (e != cudaSuccess) return cuda_error(e, "decode_attention_noalloc: scratch symbol address");
      g_scratch_addr[dev] = static_cast<float*>(p);
    }
    scratch = g_scratch_addr[dev];
  }
  DecodeAttnArgs a{};
  a.qkv = q;
  if (q_f32) {
    a.q32 = static_cast<const float*>(q);
    a.ld32 = q_stride;
  }
  a.out = out;
  a.k_cache = k_pages;
  a.v_cache = v_pages;
  a.bt = block_tables;
  a.partials = max_splits > 1 ? scratch : nullptr;
  a.n_decode = n_decode;
  a.ld = q_stride;
  a.ld_out = out_stride;
  a.qh = n_q_heads;
  a.kvh = n_kv_heads;
  a.d = head_dim;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.storage = storage;
  a.err = err_flag;
  a.ctx_lens = ctx_lens;
  a.split_keys = (int)split;
  a.max_splits = (int)max_splits;
  a.bt_stride = bt_stride;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tmk, tmv;  // host-side descriptors of the caller's pages (no device memory)
  int rc = make_kv_tmap(&tmk, k_pages, num_pages, n_kv_heads, page_size, head_dim, storage);
  if (rc == SAR_OK) rc = make_kv_tmap(&tmv, v_pages, num_pages, n_kv_heads, page_size, head_dim, storage);
  if (rc != SAR_OK) return rc;
  return dispatch<true>(a, tmk, tmv, s);
}
