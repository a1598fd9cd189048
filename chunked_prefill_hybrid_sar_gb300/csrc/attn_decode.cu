// Paged decode attention: every decode row's query heads against that
// request's own paged K/V history (the "Decode uses PagedAttention" half of
// the split, SARATHI technique write-up section 3.3; reading notes part 2
// section 3: "each decode looks up its own history KV").
//
// HBM-bound (about 4 flops per byte), so the design is about streaming pages:
//   * one CTA = (work item, KV head); a work item is a range of a decode's
//     keys (long contexts are split so every SM has work, then merged);
//   * the query heads of one GQA group share every K/V byte that is loaded;
//   * each of the 4 warps owns a private 2-deep ring of 16-key blocks
//     (K and V, 2 x 4 KB at head_dim 128) filled by cp.async.bulk straight
//     from the page (one contiguous run per block) -- no page gather, no
//     register staging;
//   * a lane owns head_dim/32 consecutive dimensions; the 16 x group partial
//     dot products are reduced with a halving butterfly (15.5 shuffles per
//     head per block instead of 80), softmax runs online in base 2;
//   * the 4 warps' (max, sum, acc) are merged in shared memory; split items
//     write unnormalised partials that decode_combine_kernel merges.
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace sar {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 2;   // per-warp ring depth (16-key blocks); 3 CTAs fit an SM
constexpr int kBlockKeys = 16;

// One halving step of the butterfly: the NV >> STEP values in v[] are split
// in two, the lane keeps the half chosen by its bit `16 >> STEP` and adds the
// partner lane's copy of that half.
template <int NV, int STEP>
__device__ __forceinline__ void butterfly_step(float (&v)[NV], int lane) {
  constexpr int mask = 16 >> STEP;
  constexpr int half = (NV >> STEP) / 2;
  const bool upper = (lane & mask) != 0;
#pragma unroll
  for (int j = 0; j < half; ++j) {
    const float send = upper ? v[j] : v[j + half];
    const float keep = upper ? v[j + half] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
  }
}

// COMPUTED = false: work items come from the host-planned list `a.items`.
// COMPUTED = true: CTA x covers split (x % max_splits) of decode (x / max_splits)
// with fixed `split_keys` ranges and a padded [n_decode][bt_stride] block table.
template <typename T, int D, int GP, bool COMPUTED = false>
__global__ void __launch_bounds__(kWarps * 32, GP >= 8 ? 2 : 3) decode_attn_kernel(DecodeAttnArgs a) {
  constexpr int DPL = D / 32;            // dimensions per lane
  constexpr int NV = kBlockKeys * GP;    // partial dots per block: 16 keys x GP heads
  constexpr int NVL = NV >= 32 ? NV / 32 : 1;
  constexpr int BLK_BYTES = kBlockKeys * D * 2;

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // layout: [warp][stage][K | V] blocks, then p buffers, merge area, barriers
  uint8_t* ring = smem + warp * kStages * 2 * BLK_BYTES;
  float* pbuf = reinterpret_cast<float*>(smem + kWarps * kStages * 2 * BLK_BYTES) + warp * NV;
  float* mrg = reinterpret_cast<float*>(smem + kWarps * kStages * 2 * BLK_BYTES) + kWarps * NV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(mrg + kWarps * GP * (D + 2)) + warp * kStages;

  int b, kbeg, kend, part, btlen;
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
    const int4 item = reinterpret_cast<const int4*>(a.items)[blockIdx.x];
    b = item.x;
    kbeg = item.y;
    kend = item.z;
    part = item.w;
    bt = a.bt + a.bt_off[b];
    btlen = a.bt_len[b];
  }
  const int kh = blockIdx.y;
  const int G = a.qh / a.kvh;
  const int nblk = (kend - kbeg + kBlockKeys - 1) / kBlockKeys;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Issue block `j` of this CTA's range into stage s (lane 0 only).
  auto issue = [&](int j, int s) -> bool {
    const int key0 = kbeg + j * kBlockKeys;
    const int bi = key0 / a.page_size;
    int page = (bi < btlen) ? bt[bi] : -1;
    if (page < 0 || page >= a.num_pages) {
      report(a.err, SAR_ERR_BOUNDS, SITE_DECODE_BOUNDS, key0);
      return false;
    }
    const int off = key0 - bi * a.page_size;
    const size_t elem = (((size_t)page * a.kvh + kh) * a.page_size + off) * D;
    const uint32_t bar = smem_u32(&bars[s]);
    uint8_t* dst = ring + s * 2 * BLK_BYTES;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, 2 * BLK_BYTES);
    bulk_g2s(smem_u32(dst), static_cast<const T*>(a.k_cache) + elem, BLK_BYTES, bar);
    bulk_g2s(smem_u32(dst + BLK_BYTES), static_cast<const T*>(a.v_cache) + elem, BLK_BYTES, bar);
    return true;
  };

  // query heads of this KV head, pre-scaled so that softmax runs in base 2
  const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
  float q[GP][DPL];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
#pragma unroll
    for (int e = 0; e < DPL; ++e) q[h][e] = 0.f;
    if (h < G) {
      if (a.q32) {
        const float* qp = a.q32 + (size_t)b * a.ld32 + (size_t)(kh * G + h) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) q[h][e] = qp[e] * qscale;
      } else {
        const T* qp = static_cast<const T*>(a.qkv) + (size_t)b * a.ld + (size_t)(kh * G + h) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) q[h][e] = Elem<T>::to(qp[e]) * qscale;
      }
    }
  }

  float m_run[GP], acc[GP][DPL];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    m_run[h] = -INFINITY;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
  }
  float l_part = 0.f;  // this lane's share of its own head's denominator

  // my blocks: j = warp, warp + 4, ...
  const int my_n = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
  bool ok = true;
  int issued = 0, consumed = 0;  // blocks put in flight / taken out (lane 0's view)
  if (lane == 0) {
    for (int i = 0; i < kStages && i < my_n && ok; ++i) {
      ok = issue(warp + i * kWarps, i);
      if (ok) ++issued;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;

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
    const int key0 = kbeg + j * kBlockKeys;
    const int nk = min(kBlockKeys, kend - key0);
    const uint8_t* kb = ring + s * 2 * BLK_BYTES;
    const uint8_t* vb = kb + BLK_BYTES;

    // ---- scores: partial dots over this lane's dims, then butterfly ----
    float v[NV];
#pragma unroll
    for (int k = 0; k < kBlockKeys; ++k) {
      float kf[DPL];
      if constexpr (DPL == 4) {
        const uint2 kv = *reinterpret_cast<const uint2*>(kb + (k * D + lane * 4) * 2);
        kf[0] = Elem<T>::lo(kv.x); kf[1] = Elem<T>::hi(kv.x); kf[2] = Elem<T>::lo(kv.y); kf[3] = Elem<T>::hi(kv.y);
      } else {
        const uint32_t kv = *reinterpret_cast<const uint32_t*>(kb + (k * D + lane * 2) * 2);
        kf[0] = Elem<T>::lo(kv); kf[1] = Elem<T>::hi(kv);
      }
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) d = fmaf(q[h][e], kf[e], d);
        v[h * kBlockKeys + k] = d;
      }
    }
    butterfly_step<NV, 0>(v, lane);
    butterfly_step<NV, 1>(v, lane);
    butterfly_step<NV, 2>(v, lane);
    butterfly_step<NV, 3>(v, lane);
    if constexpr (NV >= 32) {
      butterfly_step<NV, 4>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    }
    // lane now holds scores of indices [base, base + NVL): index = head*16 + key
    const int base = NV >= 32 ? lane * NVL : (lane >> 1);
    const int myh = base / kBlockKeys;
    float bmax = -INFINITY;
#pragma unroll
    for (int t = 0; t < NVL; ++t) {
      const int key = (base + t) % kBlockKeys;
      if (key >= nk) v[t] = -INFINITY;
      bmax = fmaxf(bmax, v[t]);
    }
    // lanes of one head: a contiguous group of 16/NVL lanes (NV >= 32), or all (NV == 16)
    constexpr int GROUP = NV >= 32 ? kBlockKeys / NVL : 32;
#pragma unroll
    for (int o = (NV >= 32 ? 1 : 2); o < GROUP; o <<= 1)
      bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
    float alpha[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      const int src = NV >= 32 ? h * GROUP : 0;
      const float bm = __shfl_sync(0xffffffffu, bmax, src);
      const float mn = fmaxf(m_run[h], bm);
      alpha[h] = exp2f(m_run[h] - mn);
      m_run[h] = mn;
    }
    float psum = 0.f;
    float mh = m_run[0], am = alpha[0];
#pragma unroll
    for (int h = 1; h < GP; ++h)
      if (h == myh) {
        mh = m_run[h];
        am = alpha[h];
      }
#pragma unroll
    for (int t = 0; t < NVL; ++t) {
      const float p = exp2f(v[t] - mh);
      psum += p;
      const int idx = base + t;
      pbuf[(idx % kBlockKeys) * GP + idx / kBlockKeys] = p;  // [key][head]
    }
    if (NV < 32 && (lane & 1)) psum = 0.f;  // lane pairs hold the same value
    l_part = l_part * am + psum;
    __syncwarp();

    // ---- acc = acc * alpha + P V ----
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] *= alpha[h];
#pragma unroll 4
    for (int k = 0; k < nk; ++k) {
      float vf[DPL];
      if constexpr (DPL == 4) {
        const uint2 vv = *reinterpret_cast<const uint2*>(vb + (k * D + lane * 4) * 2);
        vf[0] = Elem<T>::lo(vv.x); vf[1] = Elem<T>::hi(vv.x); vf[2] = Elem<T>::lo(vv.y); vf[3] = Elem<T>::hi(vv.y);
      } else {
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(vb + (k * D + lane * 2) * 2);
        vf[0] = Elem<T>::lo(vv); vf[1] = Elem<T>::hi(vv);
      }
      float p[GP];
      if constexpr (GP >= 4) {
#pragma unroll
        for (int h = 0; h < GP; h += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(&pbuf[k * GP + h]);
          p[h] = p4.x; p[h + 1] = p4.y; p[h + 2] = p4.z; p[h + 3] = p4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < GP; ++h) p[h] = pbuf[k * GP + h];
      }
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(p[h], vf[e], acc[h][e]);
    }
    __syncwarp();
    // refill this stage with block i + kStages
    if (i + kStages < my_n) {
      int r = 1;
      if (lane == 0) {
        r = issue(warp + (i + kStages) * kWarps, s) ? 1 : 0;
        issued += r;
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

  // ---- per-warp denominators, then merge the 4 warps ----
  float lsum = l_part;
  {
    constexpr int GROUP = NV >= 32 ? kBlockKeys / NVL : 32;
#pragma unroll
    for (int o = 1; o < GROUP; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  }
  float* my = mrg + warp * GP * (D + 2);
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    constexpr int GROUP = NV >= 32 ? kBlockKeys / NVL : 32;
    const float lh = __shfl_sync(0xffffffffu, lsum, NV >= 32 ? h * GROUP : 0);
#pragma unroll
    for (int e = 0; e < DPL; ++e) my[h * (D + 2) + lane * DPL + e] = acc[h][e];
    if (lane == 0) {
      my[h * (D + 2) + D] = m_run[h];
      my[h * (D + 2) + D + 1] = lh;
    }
  }
  __syncthreads();
  // 128 threads: thread t handles (head, dim) pairs
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, dd = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg[w * GP * (D + 2) + h * (D + 2) + D]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* src = mrg + w * GP * (D + 2) + h * (D + 2);
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
  float M = -INFINITY;
  for (int i = 0; i < cnt; ++i) M = fmaxf(M, a.partials[((size_t)(p0 + i) * a.qh + hq) * (D + 2) + D]);
  float L = 0.f, A = 0.f;
  for (int i = 0; i < cnt; ++i) {
    const float* pp = a.partials + ((size_t)(p0 + i) * a.qh + hq) * (D + 2);
    const float sc = exp2f(pp[D] - M);
    L = fmaf(pp[D + 1], sc, L);
    A = fmaf(pp[dd], sc, A);
  }
  static_cast<T*>(a.out)[(size_t)b * a.ld_out + (size_t)hq * D + dd] = Elem<T>::from(A / L);
}

template <typename T, int D, int GP, bool COMPUTED = false>
int launch_impl(const DecodeAttnArgs& a, cudaStream_t s) {
  constexpr int NV = kBlockKeys * GP;
  const size_t smem = (size_t)kWarps * kStages * 2 * kBlockKeys * D * 2 + (size_t)kWarps * NV * 4 +
                      (size_t)kWarps * GP * (D + 2) * 4 + (size_t)kWarps * kStages * 8 + 16;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_attn_kernel<T, D, GP, COMPUTED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_error(e, "decode attention attribute");
    attr = true;
  }
  const int n_ctas = COMPUTED ? a.n_decode * a.max_splits : a.n_items;
  decode_attn_kernel<T, D, GP, COMPUTED><<<dim3(n_ctas, a.kvh), kWarps * 32, smem, s>>>(a);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "decode attention launch");
  if (a.partials) {
    decode_combine_kernel<T, D, COMPUTED><<<dim3(a.n_decode, a.qh), D, 0, s>>>(a);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "decode combine launch");
  }
  return SAR_OK;
}

}  // namespace

int launch_decode_attention(const DecodeAttnArgs& a, cudaStream_t s) {
  if (a.n_items <= 0) return SAR_OK;
  const int G = a.qh / a.kvh;
  if (a.qh % a.kvh || G > 8 || (a.d != 64 && a.d != 128) || a.page_size % kBlockKeys)
    return set_error(SAR_ERR_UNSUPPORTED, "decode attention: head_dim 64/128, group <= 8, page % 16");
  const int GP = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
#define SAR_DEC(DD, GG)                                                             \
  if (a.d == DD && GP == GG)                                                         \
    return a.storage == SAR_STORAGE_BF16 ? launch_impl<__nv_bfloat16, DD, GG>(a, s) \
                                         : launch_impl<__half, DD, GG>(a, s);
  SAR_DEC(128, 1) SAR_DEC(128, 2) SAR_DEC(128, 4) SAR_DEC(128, 8)
  SAR_DEC(64, 1) SAR_DEC(64, 2) SAR_DEC(64, 4) SAR_DEC(64, 8)
#undef SAR_DEC
  return set_error(SAR_ERR_UNSUPPORTED, "decode attention: no kernel for this shape");
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
  const int G = n_q_heads / n_kv_heads;
  const int GP = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
#define SAR_DEC_NA(DD, GG)                                                                 \
  if (head_dim == DD && GP == GG)                                                          \
    return storage == SAR_STORAGE_BF16 ? launch_impl<__nv_bfloat16, DD, GG, true>(a, s) \
                                       : launch_impl<__half, DD, GG, true>(a, s);
  SAR_DEC_NA(128, 1) SAR_DEC_NA(128, 2) SAR_DEC_NA(128, 4) SAR_DEC_NA(128, 8)
  SAR_DEC_NA(64, 1) SAR_DEC_NA(64, 2) SAR_DEC_NA(64, 4) SAR_DEC_NA(64, 8)
#undef SAR_DEC_NA
  return set_error(SAR_ERR_UNSUPPORTED, "decode_attention_noalloc: no kernel for this shape");
}
