// Row-wise kernels of the hybrid step: RMSNorm (the step's first one also
// stacks the input rows or embeds the token ids into the fp32 residual stream,
// writes the step's rotary table and clears the logits rows), bf16 -> fp32 and
// weight conversion, greedy argmax.  All are HBM-bound and read/write each
// byte once with 16-byte accesses where the layout allows.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sar {

namespace {

constexpr int kNormThreads = 256;
constexpr int kNormMaxVec = 8;  // hidden <= 8 * 4 * 256 = 8192

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

// y[r] = x[src(r)] * rsqrt(mean(x^2) + eps) * gain with x the fp32 residual
// stream, fp32 reduction, y in the storage type T.  The normalisation ahead of
// attention and FFN, and the final norm ahead of the LM head ("insert an
// explicit sync before LayerNorm", SARATHI technique write-up, section 6.1).
//
// SRC selects where row r comes from: kSrcResidual reads the fp32 stream;
// kSrcRows (bf16 rows of the stacked batch) and kSrcTokens (embedding rows of
// token ids, storage type) are the step's first norm, which also writes the
// row into the fp32 stream `h`.  `zero` (optional): floats [0, zero_n) are
// cleared, split evenly over the blocks (the LM head's split-K accumulator,
// cleared by the step's first kernel).
enum { kSrcResidual = 0, kSrcRows = 1, kSrcTokens = 2 };

struct NormArgs {
  const float* x;         // kSrcResidual
  const void* in;         // kSrcRows: bf16 [rows, hidden]; kSrcTokens: int32 ids
  const void* table;      // kSrcTokens: [vocab, hidden] storage type
  float* h;               // kSrcRows / kSrcTokens: fp32 copy of the input row
  const float* g;
  void* y;
  const int32_t* ridx;    // kSrcResidual: optional source row per output row
  float* zero;
  size_t zero_n;
  float* zero2;           // a second region to clear (a split-K accumulator of the next GEMM)
  size_t zero2_n;
  // kSrcRows / kSrcTokens, optional: the step's rotary table, (cos, sin) of
  // pos[r] * inv_freq[i], i < half_d, at float2 index ((i / 2) * cs_ld + r) * 2
  // + i % 2 (frequency pairs major, rows adjacent)
  const int32_t* pos;
  const double* inv_freq;
  float2* cs;
  int half_d, cs_ld;
  int hidden, vocab;
  float eps;
  int* err;
};

template <typename T, int SRC>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const NormArgs a) {
  const int nv = a.hidden >> 2;
  // the gains are weights, not the previous kernel's output: fetch them while
  // that kernel drains
  const float4* gr = reinterpret_cast<const float4*>(a.g);
  float4 gv[kNormMaxVec];
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    if (i < nv) gv[k] = __ldg(gr + i);
  }
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[32];
  const int r = blockIdx.x;
  float4 v[kNormMaxVec];
  bool ok = true;
  if constexpr (SRC == kSrcResidual) {
    const int src = a.ridx ? a.ridx[r] : r;
    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)src * a.hidden);
#pragma unroll
    for (int k = 0; k < kNormMaxVec; ++k) {
      const int i = threadIdx.x + k * kNormThreads;
      if (i < nv) v[k] = xr[i];
    }
  } else {
    const uint2* sr;
    if constexpr (SRC == kSrcRows) {
      sr = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.in) + (size_t)r * a.hidden);
    } else {
      const int t = static_cast<const int32_t*>(a.in)[r];
      ok = t >= 0 && t < a.vocab;
      if (!ok && threadIdx.x == 0) report(a.err, SAR_ERR_BOUNDS, SITE_EMBED_BOUNDS, t);
      sr = reinterpret_cast<const uint2*>(static_cast<const T*>(a.table) + (size_t)(ok ? t : 0) * a.hidden);
    }
    // the row's loads first, then the rotary table (its double-precision
    // steps overlap their latency), then the fp32 copy of the row
    uint2 u[kNormMaxVec];
#pragma unroll
    for (int k = 0; k < kNormMaxVec; ++k) {
      const int i = threadIdx.x + k * kNormThreads;
      if (i < nv) u[k] = sr[i];
    }
    if (a.cs) {
      // the angle pos * theta_i is formed and reduced modulo 2*pi in double
      // precision, so long positions keep fp32 accuracy
      const double p = (double)a.pos[r];
      for (int i = threadIdx.x; i < a.half_d; i += kNormThreads) {
        double ang = p * a.inv_freq[i];
        const double two_pi = 6.283185307179586476925286766559;
        ang -= two_pi * rint(ang * (1.0 / two_pi));
        float sn, cn;
        sincosf((float)ang, &sn, &cn);
        a.cs[((size_t)(i >> 1) * a.cs_ld + r) * 2 + (i & 1)] = make_float2(cn, sn);
      }
    }
    float4* hr = reinterpret_cast<float4*>(a.h + (size_t)r * a.hidden);
#pragma unroll
    for (int k = 0; k < kNormMaxVec; ++k) {
      const int i = threadIdx.x + k * kNormThreads;
      if (i < nv) {
        if constexpr (SRC == kSrcRows)
          v[k] = make_float4(bf16lo(u[k].x), bf16hi(u[k].x), bf16lo(u[k].y), bf16hi(u[k].y));
        else
          v[k] = make_float4(Elem<T>::lo(u[k].x), Elem<T>::hi(u[k].x), Elem<T>::lo(u[k].y), Elem<T>::hi(u[k].y));
        if (!ok) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        hr[i] = v[k];
      }
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    if (i < nv) {
      ss = fmaf(v[k].x, v[k].x, ss);
      ss = fmaf(v[k].y, v[k].y, ss);
      ss = fmaf(v[k].z, v[k].z, ss);
      ss = fmaf(v[k].w, v[k].w, ss);
    }
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)a.hidden + a.eps);
  uint2* yr = reinterpret_cast<uint2*>(static_cast<T*>(a.y) + (size_t)r * a.hidden);
#pragma unroll
  for (int k = 0; k < kNormMaxVec; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    if (i < nv) {
      yr[i] = make_uint2(Elem<T>::pack(v[k].x * inv * gv[k].x, v[k].y * inv * gv[k].y),
                         Elem<T>::pack(v[k].z * inv * gv[k].z, v[k].w * inv * gv[k].w));
    }
  }
  // block r clears its share of each region, a multiple of 4 floats (16-byte stores)
  auto clear = [&](float* z, size_t n) {
    const size_t per = ((n + gridDim.x - 1) / gridDim.x + 3) & ~(size_t)3;
    const size_t z0 = per * r, z1 = min(n, z0 + per);
    if (z0 < z1) {
      const size_t n4 = (z1 - z0) >> 2;
      float4* z4 = reinterpret_cast<float4*>(z + z0);
      for (size_t i = threadIdx.x; i < n4; i += kNormThreads) z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (size_t i = z0 + 4 * n4 + threadIdx.x; i < z1; i += kNormThreads) z[i] = 0.f;
    }
  };
  if (a.zero) clear(a.zero, a.zero_n);
  if (a.zero2) clear(a.zero2, a.zero2_n);
}

// The rotary embedding and KV-page append for rows whose QKV projection was
// accumulated split-K into fp32 (the small-row steps): per row, q and k heads
// are rotated in place (dim i with i + hd/2, the (cos, sin) table of the
// row's position), and k and v are rounded once into the row's page slot --
// what the fused QKV epilogue does for larger steps.  One block per row.
template <typename T>
__global__ void rope_append_kernel(float* qkv, int ld, RopeEpi rp, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const int half = rp.hd >> 1, hq4 = half >> 2;  // 4 pairs per item
  const int heads = rp.qh + 2 * rp.kvh;
  const int sl = rp.slot[r];
  const int page = sl >= 0 ? sl / rp.page_size : -1;
  const int off = sl - page * rp.page_size;
  const bool slot_ok = sl >= 0 && page < rp.num_pages;
  if (!slot_ok && threadIdx.x == 0) report(err, SAR_ERR_BOUNDS, SITE_ROPE_BOUNDS, r);
  float* row = qkv + (size_t)r * ld;
  const float4* cs4 = reinterpret_cast<const float4*>(rp.cs) + r;  // pair i of this row at cs4[i * cs_ld]
  for (int it = threadIdx.x; it < heads * hq4; it += blockDim.x) {
    const int head = it / hq4, i = (it - head * hq4) * 4;
    const bool is_v = head >= rp.qh + rp.kvh, is_k = !is_v && head >= rp.qh;
    float4* p1 = reinterpret_cast<float4*>(row + head * rp.hd + i);
    float4* p2 = reinterpret_cast<float4*>(row + head * rp.hd + half + i);
    float4 a = *p1, b = *p2;
    if (!is_v) {
      const float4 c01 = cs4[(size_t)(i >> 1) * rp.cs_ld], c23 = cs4[(size_t)((i >> 1) + 1) * rp.cs_ld];  // (cos, sin) of i..i+3
      const float c[4] = {c01.x, c01.z, c23.x, c23.z}, sn[4] = {c01.y, c01.w, c23.y, c23.w};
      const float x1[4] = {a.x, a.y, a.z, a.w}, x2[4] = {b.x, b.y, b.z, b.w};
      float y1[4], y2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        y1[e] = x1[e] * c[e] - x2[e] * sn[e];
        y2[e] = x2[e] * c[e] + x1[e] * sn[e];
      }
      a = make_float4(y1[0], y1[1], y1[2], y1[3]);
      b = make_float4(y2[0], y2[1], y2[2], y2[3]);
      *p1 = a;
      *p2 = b;
    }
    if ((is_k || is_v) && slot_ok) {
      const int kh = head - rp.qh - (is_v ? rp.kvh : 0);
      T* dst = static_cast<T*>(is_v ? rp.v_cache : rp.k_cache) + (((size_t)page * rp.kvh + kh) * rp.page_size + off) * rp.hd;
      *reinterpret_cast<uint2*>(dst + i) = make_uint2(Elem<T>::pack(a.x, a.y), Elem<T>::pack(a.z, a.w));
      *reinterpret_cast<uint2*>(dst + half + i) = make_uint2(Elem<T>::pack(b.x, b.y), Elem<T>::pack(b.z, b.w));
    }
  }
}

// silu(gate) * up from the gate/up projection accumulated split-K into fp32
// (the packed layout: 64-row gate and up blocks interleaved), rounded once to
// the storage type; what the fused SwiGLU epilogue does for larger steps.
template <typename T>
__global__ void swiglu_finish_kernel(const float* __restrict__ gu, T* __restrict__ act, int rows, int F) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t n4 = (size_t)rows * F / 4;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n4; q += (size_t)gridDim.x * blockDim.x) {
    const size_t o = q * 4;
    const size_t r = o / F;
    const int f = (int)(o - r * F);
    const int blk = f >> 6, j = f & 63;
    const float* src = gu + r * 2 * (size_t)F + (size_t)blk * 128 + j;
    const float4 g = *reinterpret_cast<const float4*>(src);
    const float4 u = *reinterpret_cast<const float4*>(src + 64);
    auto sl = [](float x) { return silu(x); };
    *reinterpret_cast<uint2*>(act + o) =
        make_uint2(Elem<T>::pack(sl(g.x) * u.x, sl(g.y) * u.y), Elem<T>::pack(sl(g.z) * u.z, sl(g.w) * u.w));
  }
}

// Embedding rows of the storage type into the fp32 residual stream.
template <typename T>
__global__ void embed_kernel(const int32_t* __restrict__ tok, const T* __restrict__ table,
                             float* __restrict__ out, int hidden, int vocab, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const int t = tok[r];
  float4* dst = reinterpret_cast<float4*>(out + (size_t)r * hidden);
  const int nv = hidden >> 2;
  if (t < 0 || t >= vocab) {
    if (threadIdx.x == 0) report(err, SAR_ERR_BOUNDS, SITE_EMBED_BOUNDS, t);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const uint2* src = reinterpret_cast<const uint2*>(table + (size_t)t * hidden);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const uint2 v = src[i];
    dst[i] = make_float4(Elem<T>::lo(v.x), Elem<T>::hi(v.x), Elem<T>::lo(v.y), Elem<T>::hi(v.y));
  }
}

// bf16 -> fp32 (input rows into the residual stream, norm gains), 8 values
// (16 bytes in, 32 out) per thread; n is a multiple of 8.
__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst, size_t n8) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 v = reinterpret_cast<const uint4*>(src)[i];
  float4* d = reinterpret_cast<float4*>(dst) + 2 * i;
  d[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
  d[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
}

// bf16 weight rows -> storage type T, row r of the source landing on row
// map(r) of the destination: identity, or the gate/up interleave (64-row
// blocks, gate first when `up` is 0).
template <typename T>
__global__ void convert_rows_kernel(const __nv_bfloat16* __restrict__ src, T* __restrict__ dst, int rows,
                                    int cols, int interleave, int up) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const int dr = interleave ? (r / 64) * 128 + up * 64 + (r % 64) : r;
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src + (size_t)r * cols);
  uint32_t* d = reinterpret_cast<uint32_t*>(dst + (size_t)dr * cols);
  for (int i = threadIdx.x; i < (cols >> 1); i += blockDim.x) {
    const uint32_t v = s[i];
    d[i] = Elem<T>::pack(bf16lo(v), bf16hi(v));
  }
}

// Greedy sampling: lowest index among the maxima of each row.
__global__ void __launch_bounds__(1024) argmax_kernel(const float* __restrict__ logits, int vocab,
                                                     int32_t* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float bv[32];
  __shared__ int bi[32];
  const float* row = logits + (size_t)blockIdx.x * vocab;
  float best = -FLT_MAX;
  int besti = 0x7fffffff;
  // each thread scans its entries in increasing index order (so the first of
  // equal maxima stays); rows whose start is 16-byte aligned are read as
  // float4, eight loads in flight per thread
  int tail = 0;
  if ((vocab & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = vocab >> 2;
    constexpr int kU = 8;
    for (int base = 0; base < n4; base += kU * (int)blockDim.x) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * (int)blockDim.x + (int)threadIdx.x;
        v[u] = i < n4 ? __ldg(r4 + i) : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = 4 * (base + u * (int)blockDim.x + (int)threadIdx.x);
        if (v[u].x > best) { best = v[u].x; besti = i; }
        if (v[u].y > best) { best = v[u].y; besti = i + 1; }
        if (v[u].z > best) { best = v[u].z; besti = i + 2; }
        if (v[u].w > best) { best = v[u].w; besti = i + 3; }
      }
    }
    tail = vocab;  // nothing left
  }
  for (int i = tail + (int)threadIdx.x; i < vocab; i += blockDim.x) {
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

int launch_rmsnorm(const float* x, const float* gain, void* y, int rows, int hidden, float eps,
                   const int32_t* row_index, int storage, cudaStream_t s, float* zero, size_t zero_n) {
  if (rows <= 0) return SAR_OK;
  if (hidden % 4 || hidden > 4 * kNormThreads * kNormMaxVec)
    return set_error(SAR_ERR_UNSUPPORTED, "rmsnorm: hidden must be a multiple of 4 and at most 8192");
  NormArgs a = {};
  a.x = x;
  a.g = gain;
  a.y = y;
  a.ridx = row_index;
  a.hidden = hidden;
  a.eps = eps;
  a.zero = zero;
  a.zero_n = zero_n;
  cudaError_t e = storage == SAR_STORAGE_BF16
                      ? launch_pdl(rmsnorm_kernel<__nv_bfloat16, kSrcResidual>, dim3(rows), dim3(kNormThreads), 0, s, a)
                      : launch_pdl(rmsnorm_kernel<__half, kSrcResidual>, dim3(rows), dim3(kNormThreads), 0, s, a);
  if (e != cudaSuccess) return cuda_error(e, "rmsnorm launch");
  count_launches(1);
  return SAR_OK;
}

int launch_input_norm(int in_kind, const void* in, const void* table, int vocab, float* h, const float* gain,
                      void* y, int rows, int hidden, float eps, int storage, int* err, cudaStream_t s,
                      float* zero, size_t zero_n, const int32_t* pos, const double* inv_freq, float2* cs,
                      int half_d, int cs_ld, float* zero2, size_t zero2_n) {
  if (rows <= 0) return SAR_OK;
  if (hidden % 4 || hidden > 4 * kNormThreads * kNormMaxVec)
    return set_error(SAR_ERR_UNSUPPORTED, "rmsnorm: hidden must be a multiple of 4 and at most 8192");
  NormArgs a = {};
  a.in = in;
  a.table = table;
  a.h = h;
  a.g = gain;
  a.y = y;
  a.hidden = hidden;
  a.vocab = vocab;
  a.eps = eps;
  a.err = err;
  a.zero = zero;
  a.zero_n = zero_n;
  a.zero2 = zero2;
  a.zero2_n = zero2_n;
  a.pos = pos;
  a.inv_freq = inv_freq;
  a.cs = cs;
  a.half_d = half_d;
  a.cs_ld = cs_ld;
  if (cs && (cs_ld < rows || half_d % 2)) return set_error(SAR_ERR_INVALID_ARG, "input norm: rotary table stride");
  const bool bf = storage == SAR_STORAGE_BF16;
  const dim3 g(rows), b(kNormThreads);
  cudaError_t e;
  if (in_kind == SAR_IN_TOKENS)
    e = bf ? launch_pdl(rmsnorm_kernel<__nv_bfloat16, kSrcTokens>, g, b, 0, s, a)
           : launch_pdl(rmsnorm_kernel<__half, kSrcTokens>, g, b, 0, s, a);
  else
    e = bf ? launch_pdl(rmsnorm_kernel<__nv_bfloat16, kSrcRows>, g, b, 0, s, a)
           : launch_pdl(rmsnorm_kernel<__half, kSrcRows>, g, b, 0, s, a);
  if (e != cudaSuccess) return cuda_error(e, "input norm launch");
  count_launches(1);
  return SAR_OK;
}

int launch_rope_append(float* qkv, int ld, int rows, const RopeEpi& rp, int storage, int* err, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  if ((rp.hd != 64 && rp.hd != 128) || ld != (rp.qh + 2 * rp.kvh) * rp.hd || !rp.slot || !rp.cs || rp.cs_ld < rows)
    return set_error(SAR_ERR_INVALID_ARG, "rope/append: bad arguments");
  cudaError_t e = storage == SAR_STORAGE_BF16
                      ? launch_pdl(rope_append_kernel<__nv_bfloat16>, dim3(rows), dim3(256), 0, s, qkv, ld, rp, err)
                      : launch_pdl(rope_append_kernel<__half>, dim3(rows), dim3(256), 0, s, qkv, ld, rp, err);
  if (e != cudaSuccess) return cuda_error(e, "rope/append launch");
  count_launches(1);
  return SAR_OK;
}

int launch_swiglu_finish(const float* gu, void* act, int rows, int F, int storage, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  if (F % 64) return set_error(SAR_ERR_INVALID_ARG, "swiglu: F must be a multiple of 64");
  const size_t n4 = (size_t)rows * F / 4;
  const int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)num_sms() * 8);
  cudaError_t e = storage == SAR_STORAGE_BF16
                      ? launch_pdl(swiglu_finish_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s, gu,
                                   static_cast<__nv_bfloat16*>(act), rows, F)
                      : launch_pdl(swiglu_finish_kernel<__half>, dim3(blocks), dim3(256), 0, s, gu,
                                   static_cast<__half*>(act), rows, F);
  if (e != cudaSuccess) return cuda_error(e, "swiglu launch");
  count_launches(1);
  return SAR_OK;
}

int launch_embed(const int32_t* tokens, const void* table, float* out, int rows, int hidden, int vocab,
                 int storage, int* err, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  if (storage == SAR_STORAGE_BF16)
    launch_pdl(embed_kernel<__nv_bfloat16>, dim3(rows), dim3(256), 0, s, tokens, static_cast<const __nv_bfloat16*>(table), out, hidden,
                                                     vocab, err);
  else
    launch_pdl(embed_kernel<__half>, dim3(rows), dim3(256), 0, s, tokens, static_cast<const __half*>(table), out, hidden, vocab, err);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "embed launch");
}

int launch_bf16_to_f32(const void* src, float* dst, size_t n, cudaStream_t s) {
  if (n == 0) return SAR_OK;
  if (n % 8) return set_error(SAR_ERR_UNSUPPORTED, "bf16 to fp32: length must be a multiple of 8");
  const size_t n8 = n / 8;
  launch_pdl(bf16_to_f32_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src), dst, n8);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "bf16 to fp32 launch");
}

int launch_convert_rows(const void* src, void* dst, int rows, int cols, int interleave, int up, int storage,
                        cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  if (cols % 2) return set_error(SAR_ERR_UNSUPPORTED, "convert: odd row width");
  const __nv_bfloat16* sp = static_cast<const __nv_bfloat16*>(src);
  if (storage == SAR_STORAGE_BF16)
    launch_pdl(convert_rows_kernel<__nv_bfloat16>, dim3(rows), dim3(256), 0, s, sp, static_cast<__nv_bfloat16*>(dst), rows, cols,
                                                           interleave, up);
  else
    launch_pdl(convert_rows_kernel<__half>, dim3(rows), dim3(256), 0, s, sp, static_cast<__half*>(dst), rows, cols, interleave, up);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "convert launch");
}

int launch_argmax(const float* logits, int rows, int vocab, int32_t* out, cudaStream_t s) {
  if (rows <= 0) return SAR_OK;
  launch_pdl(argmax_kernel, dim3(rows), dim3(1024), 0, s, logits, vocab, out);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "argmax launch");
}

// The bounded-wait path on its own: one thread initialises a barrier that
// expects two arrivals, arrives `arrivals` times and waits for the phase with
// mbar_wait's limit set to `limit_ns`.  With fewer than two arrivals the phase
// never completes, so the wait runs out, records SAR_ERR_TIMEOUT in `err` and
// the kernel returns; nothing else is in flight.
__global__ void wait_check_kernel(uint64_t limit_ns, int arrivals, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 2);
  fence_mbar_init();
  for (int i = 0; i < arrivals; ++i) mbar_arrive(b);
  mbar_wait(b, 0, err, SITE_WAIT_CHECK, limit_ns);
}

int launch_wait_check(uint64_t limit_ns, int arrivals, int* err, cudaStream_t s) {
  wait_check_kernel<<<1, 32, 0, s>>>(limit_ns, arrivals, err);
  count_launches(1);
  return cuda_error(cudaGetLastError(), "wait check launch");
}

}  // namespace sar
