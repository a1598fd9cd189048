// Row-wise kernels of the hybrid step: RMSNorm, rotary embedding fused with
// the KV-page append, embedding gather and greedy argmax.  All are HBM-bound
// and read/write each byte once with 16-byte accesses where the layout allows.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace sar {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float t = (l < nw) ? red[l] : 0.f;
  t = warp_sum(t);
  __syncthreads();
  return t;
}

// y[r] = x[src(r)] * rsqrt(mean(x^2) + eps) * gain, fp32 reduction.  The
// normalisation ahead of attention and FFN, and the final norm ahead of the
// LM head ("insert an explicit sync before LayerNorm", SARATHI technique
// write-up, section 6.1).
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                              const __nv_bfloat16* __restrict__ g,
                                                              __nv_bfloat16* __restrict__ y,
                                                              int hidden, float eps,
                                                              const int32_t* __restrict__ ridx) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int src = ridx ? ridx[r] : r;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)src * hidden);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)r * hidden);
  const int nv = hidden >> 3;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo(w[e]), b = bf16hi(w[e]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)hidden + eps);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const uint4 v = xr[i];
    const uint4 gv = gr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_bf16(bf16lo(w[e]) * inv * bf16lo(gw[e]), bf16hi(w[e]) * inv * bf16hi(gw[e]));
    yr[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void embed_kernel(const int32_t* __restrict__ tok, const __nv_bfloat16* __restrict__ table,
                             __nv_bfloat16* __restrict__ out, int hidden, int vocab, int* err) {
  const int r = blockIdx.x;
  const int t = tok[r];
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)r * hidden);
  const int nv = hidden >> 3;
  if (t < 0 || t >= vocab) {
    if (threadIdx.x == 0) report(err, SAR_ERR_BOUNDS, SITE_EMBED_BOUNDS, t);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(table + (size_t)t * hidden);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = src[i];
}

// Rotary embedding of the q and k heads of one row at its absolute position
// (a chunk keeps numbering from its start position: "maintain an independent
// position_id for each chunk", SARATHI technique write-up, section 6.1), then
// the rotated k and the v of that row are written into the row's page slot.
// The angle pos * theta_i is formed and reduced modulo 2*pi in double
// precision once per (row, frequency), so long positions keep fp32 accuracy.
__global__ void rope_append_kernel(RopeArgs a) {
  __shared__ float cs[64], sn[64];
  const int r = blockIdx.x;
  const int pos = a.pos[r];
  const int slot = a.slot[r];
  const int half = a.d >> 1;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    double ang = (double)pos * a.inv_freq[i];
    const double two_pi = 6.283185307179586476925286766559;
    ang -= two_pi * rint(ang * (1.0 / two_pi));
    float s, c;
    sincosf((float)ang, &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
  __syncthreads();
  const int page = slot / a.page_size;
  const int off = slot - page * a.page_size;
  const bool slot_ok = slot >= 0 && page < a.num_pages;
  if (!slot_ok && threadIdx.x == 0) report(a.err, SAR_ERR_BOUNDS, SITE_ROPE_BOUNDS, slot);
  const int width = (a.qh + 2 * a.kvh) * a.d;
  __nv_bfloat16* row = a.qkv + (size_t)r * width;
  const int n_pairs = (a.qh + a.kvh) * half;
  for (int idx = threadIdx.x; idx < n_pairs; idx += blockDim.x) {
    const int h = idx / half;
    const int i = idx - h * half;
    __nv_bfloat16* base = row + h * a.d;
    const float x1 = __bfloat162float(base[i]);
    const float x2 = __bfloat162float(base[i + half]);
    const float c = cs[i], s = sn[i];
    const __nv_bfloat16 y1 = __float2bfloat16_rn(x1 * c - x2 * s);
    const __nv_bfloat16 y2 = __float2bfloat16_rn(x2 * c + x1 * s);
    base[i] = y1;
    base[i + half] = y2;
    if (h >= a.qh && slot_ok) {
      const int kh = h - a.qh;
      __nv_bfloat16* kc = a.k_cache + (((size_t)page * a.kvh + kh) * a.page_size + off) * a.d;
      kc[i] = y1;
      kc[i + half] = y2;
    }
  }
  if (slot_ok) {
    const __nv_bfloat16* vrow = row + (a.qh + a.kvh) * a.d;
    const int nv = a.kvh * a.d;
    for (int idx = threadIdx.x; idx < nv; idx += blockDim.x) {
      const int kh = idx / a.d;
      const int j = idx - kh * a.d;
      a.v_cache[(((size_t)page * a.kvh + kh) * a.page_size + off) * a.d + j] = vrow[idx];
    }
  }
}

// Greedy sampling: lowest index among the maxima of each row.
__global__ void __launch_bounds__(1024) argmax_kernel(const float* __restrict__ logits, int vocab,
                                                     int32_t* __restrict__ out) {
  __shared__ float bv[32];
  __shared__ int bi[32];
  const float* row = logits + (size_t)blockIdx.x * vocab;
  float best = -FLT_MAX;
  int besti = 0x7fffffff;
  for (int i = threadIdx.x; i < vocab; i += blockDim.x) {
    const float v = row[i];
    if (v > best) {
      best = v;
      besti = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, best, o);
    const int j = __shfl_xor_sync(0xffffffffu, besti, o);
    if (v > best || (v == best && j < besti)) {
      best = v;
      besti = j;
    }
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    bv[w] = best;
    bi[w] = besti;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    best = l < nw ? bv[l] : -FLT_MAX;
    besti = l < nw ? bi[l] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v = __shfl_xor_sync(0xffffffffu, best, o);
      const int j = __shfl_xor_sync(0xffffffffu, besti, o);
      if (v > best || (v == best && j < besti)) {
        best = v;
        besti = j;
      }
    }
    if (l == 0) out[blockIdx.x] = besti;
  }
}

}  // namespace

int launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* gain, __nv_bfloat16* y, int rows,
                   int hidden, float eps, const int32_t* row_index, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  if (hidden % 8) return set_error(SAR_ERR_UNSUPPORTED, "rmsnorm: hidden must be a multiple of 8");
  rmsnorm_kernel<<<rows, kNormThreads, 0, s>>>(x, gain, y, hidden, eps, row_index);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "rmsnorm launch");
}

int launch_embed(const int32_t* tokens, const __nv_bfloat16* table, __nv_bfloat16* out, int rows,
                 int hidden, int vocab, int* err, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  embed_kernel<<<rows, 256, 0, s>>>(tokens, table, out, hidden, vocab, err);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "embed launch");
}

int launch_rope_append(const RopeArgs& a, cudaStream_t s) {
  if (a.M <= 0) return SAR_OK;
  if (a.d > 128 || a.d % 2) return set_error(SAR_ERR_UNSUPPORTED, "rope: head_dim > 128");
  rope_append_kernel<<<a.M, 256, 0, s>>>(a);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "rope launch");
}

int launch_argmax(const float* logits, int rows, int vocab, int32_t* out, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  argmax_kernel<<<rows, 1024, 0, s>>>(logits, vocab, out);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "argmax launch");
}

}  // namespace sar
