// Prefill-chunk attention: the chunk's queries (rows [0, Lp) of the stacked
// batch) attend causally to the keys of the prompt's earlier chunks, held in
// the paged KV cache, and to their own keys, which the rotary/append kernel
// has already written into the pages ("Prefill uses FlashAttention-2",
// SARATHI technique write-up section 3.3; cross-chunk attention must stay
// correct, same page section 3.1).  Chunk k re-reads the KV of the k earlier
// chunks -- the N(N-1)/2 re-read of the Sarathi-Serve digest, section 4.
//
// One launch serves every chunk of a batch: CTA x takes tile x of the step's
// tile table (up to 64 consecutive rows of one prompt's chunk).
//
// Tiled online-softmax attention on warp-level 16-bit MMAs (m16n8k16, fp32
// accumulate; the fp32 queries enter as a high and a low 16-bit part, so the
// scores are as precise as the 16-bit keys allow): a CTA owns 64 query rows of
// one query head (16 per warp); K/V
// tiles of 64 keys are gathered page by page with 16-byte cp.async into an
// XOR-swizzled shared layout (conflict-free ldmatrix), double buffered.
// Keys past the causal limit are zero-filled and masked.  With a sliding
// window of W keys the CTA starts at the tile holding its first row's oldest
// visible key and masks, per row, the keys at or before (position - W).
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace sar {

namespace {

constexpr int kBQ = 64;      // query rows per CTA
constexpr int kBKV = 64;     // keys per tile
constexpr int kThreads = 128;
static_assert(kBQ == kChunkTileRows, "the step plans tiles of kBQ rows");

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
// D += A . B on a 16x8x16 tile, fp32 accumulate; A and B both of the storage type T.
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

// byte offset of (row, 16-byte chunk) in a [rows][D] bf16 tile, chunks XOR-swizzled by row % 8
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) chunk_attn_kernel(ChunkAttnArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int TILE = kBKV * D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sq = smem;                     // [2][64][D]: q split into a high and a low part
  uint8_t* skv = smem + 2 * kBQ * D * 2;  // [2 stages][K | V][64][D]

  const int hq = blockIdx.y;
  const int G = a.qh / a.kvh;
  const int kh = hq / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tile (the table lists the most keys first)
  const int* tl = a.tiles + 8 * blockIdx.x;
  const int row0 = tl[0], pos0 = tl[1], nq = tl[2];
  const int32_t* bt = a.bt + tl[3];
  const int bt_len = tl[4];
  const int last_pos = pos0 + nq - 1;        // latest query position in this CTA
  const int n_tiles = last_pos / kBKV + 1;
  const int t0 = a.window > 0 ? max(0, pos0 - a.window + 1) / kBKV : 0;  // first key tile in any window
  const uint32_t sq_u = smem_u32(sq), skv_u = smem_u32(skv);
  const uint32_t sql_u = sq_u + kBQ * D * 2;

  // ---- Q tile from fp32 rows, split q = hi + lo in the storage type so that
  // the scores keep about twice the storage precision (rows past the chunk are zero)
  for (int c = threadIdx.x; c < kBQ * CH; c += kThreads) {
    const int r = c / CH, ch = c % CH;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < nq) {
      const float4* src = reinterpret_cast<const float4*>(a.q32 + (size_t)(row0 + r) * a.ld32 + (size_t)hq * D + ch * 8);
      const float4 x0 = src[0], x1 = src[1];
      f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w; f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hi[e] = Elem<T>::pack(f[2 * e], f[2 * e + 1]);
      lo[e] = Elem<T>::pack(f[2 * e] - Elem<T>::lo(hi[e]), f[2 * e + 1] - Elem<T>::hi(hi[e]));
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sq_u + swz<D>(r, ch)), "r"(hi[0]), "r"(hi[1]),
                 "r"(hi[2]), "r"(hi[3]) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sql_u + swz<D>(r, ch)), "r"(lo[0]), "r"(lo[1]),
                 "r"(lo[2]), "r"(lo[3]) : "memory");
  }
  auto load_kv = [&](int t, int stage) {
    const uint32_t kbase = skv_u + stage * 2 * TILE;
    const uint32_t vbase = kbase + TILE;
    for (int c = threadIdx.x; c < kBKV * CH; c += kThreads) {
      const int r = c / CH, ch = c % CH;
      const int pos = t * kBKV + r;
      const int bi = pos / a.page_size;
      bool ok = pos <= last_pos && bi < bt_len;
      int page = ok ? bt[bi] : 0;
      if (ok && (page < 0 || page >= a.num_pages)) {
        report(a.err, SAR_ERR_BOUNDS, SITE_CHUNK_BOUNDS, pos);
        ok = false;
        page = 0;
      }
      const size_t elem = (((size_t)page * a.kvh + kh) * a.page_size + (pos - bi * a.page_size)) * D + ch * 8;
      const T* ks = static_cast<const T*>(a.k_cache) + (ok ? elem : 0);
      const T* vs = static_cast<const T*>(a.v_cache) + (ok ? elem : 0);
      cp_async16(kbase + swz<D>(r, ch), ks, ok ? 16 : 0);
      cp_async16(vbase + swz<D>(r, ch), vs, ok ? 16 : 0);
    }
  };
  load_kv(t0, t0 & 1);
  cp_async_commit();

  const float sl2 = rsqrtf((float)D) * 1.4426950408889634f;
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int r_lo = warp * 16 + (lane >> 2);  // this thread's two query rows in the tile
  const int qpos0 = pos0 + r_lo;
  const int qpos1 = qpos0 + 8;
  // oldest visible key of each row (keys below it are masked)
  const int klo0 = a.window > 0 ? qpos0 - a.window + 1 : 0;
  const int klo1 = a.window > 0 ? qpos1 - a.window + 1 : 0;

  for (int t = t0; t < n_tiles; ++t) {
    if (t + 1 < n_tiles) load_kv(t + 1, (t + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kbase = skv_u + (t & 1) * 2 * TILE;
    const uint32_t vbase = kbase + TILE;

    // ---- S = Q K^T (16 x 64 per warp) ----
    float s[kBKV / 8][4];
#pragma unroll
    for (int j = 0; j < kBKV / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      const int mi = lane >> 3;
      const int qrow = warp * 16 + (mi & 1) * 8 + (lane & 7);
      uint32_t qh0[4], qh1[4], ql0[4], ql1[4];
      ldsm_x4(sq_u + swz<D>(qrow, kk * 2 + (mi >> 1)), qh0[0], qh0[1], qh0[2], qh0[3]);
      ldsm_x4(sq_u + swz<D>(qrow, kk * 2 + 2 + (mi >> 1)), qh1[0], qh1[1], qh1[2], qh1[3]);
      ldsm_x4(sql_u + swz<D>(qrow, kk * 2 + (mi >> 1)), ql0[0], ql0[1], ql0[2], ql0[3]);
      ldsm_x4(sql_u + swz<D>(qrow, kk * 2 + 2 + (mi >> 1)), ql1[0], ql1[1], ql1[2], ql1[3]);
#pragma unroll
      for (int j = 0; j < kBKV / 8; ++j) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz<D>(j * 8 + (lane & 7), kk * 2 + mi), b0, b1, b2, b3);
        mma16816<T>(s[j], qh0[0], qh0[1], qh0[2], qh0[3], b0, b1);
        mma16816<T>(s[j], ql0[0], ql0[1], ql0[2], ql0[3], b0, b1);
        mma16816<T>(s[j], qh1[0], qh1[1], qh1[2], qh1[3], b2, b3);
        mma16816<T>(s[j], ql1[0], ql1[1], ql1[2], ql1[3], b2, b3);
      }
    }
    // ---- causal (and window) mask + online softmax (base 2) ----
    const int kpos0 = t * kBKV + 2 * (lane & 3);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < kBKV / 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kp = kpos0 + j * 8 + e;
        s[j][e] = (kp <= qpos0 && kp >= klo0) ? s[j][e] * sl2 : -INFINITY;
        s[j][2 + e] = (kp <= qpos1 && kp >= klo1) ? s[j][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pf[kBKV / 16][4];
#pragma unroll
    for (int j = 0; j < kBKV / 8; ++j) {
      const float p0 = exp2f(s[j][0] - ref0), p1 = exp2f(s[j][1] - ref0);
      const float p2 = exp2f(s[j][2] - ref1), p3 = exp2f(s[j][3] - ref1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      pf[j >> 1][(j & 1) * 2 + 0] = Elem<T>::pack(p0, p1);
      pf[j >> 1][(j & 1) * 2 + 1] = Elem<T>::pack(p2, p3);
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
    }
    // ---- O += P V ----
#pragma unroll
    for (int kt = 0; kt < kBKV / 16; ++kt) {
#pragma unroll
      for (int j = 0; j < D / 8; j += 2) {
        uint32_t b0, b1, b2, b3;
        const int mi = lane >> 3;
        ldsm_x4_t(vbase + swz<D>(kt * 16 + (mi & 1) * 8 + (lane & 7), j + (mi >> 1)), b0, b1, b2, b3);
        mma16816<T>(o[j], pf[kt][0], pf[kt][1], pf[kt][2], pf[kt][3], b0, b1);
        mma16816<T>(o[j + 1], pf[kt][0], pf[kt][1], pf[kt][2], pf[kt][3], b2, b3);
      }
    }
    __syncthreads();  // stage (t & 1) is refilled at iteration t + 1
  }

  // ---- normalise and store ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int orow0 = row0 + r_lo, orow1 = orow0 + 8;
#pragma unroll
  T* out = static_cast<T*>(a.out);
  for (int j = 0; j < D / 8; ++j) {
    const int col = hq * D + j * 8 + 2 * (lane & 3);
    if (r_lo < nq)
      *reinterpret_cast<uint32_t*>(out + (size_t)orow0 * a.ld_out + col) = Elem<T>::pack(o[j][0] * inv0, o[j][1] * inv0);
    if (r_lo + 8 < nq)
      *reinterpret_cast<uint32_t*>(out + (size_t)orow1 * a.ld_out + col) = Elem<T>::pack(o[j][2] * inv1, o[j][3] * inv1);
  }
}

template <typename T, int D>
int launch_impl(const ChunkAttnArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)2 * kBQ * D * 2 + (size_t)2 * 2 * kBKV * D * 2;
  const int arc = ensure_smem_attr(reinterpret_cast<const void*>(&chunk_attn_kernel<T, D>), (int)smem,
                                   "chunk attention attribute");
  if (arc != SAR_OK) return arc;
  dim3 grid(a.n_tiles, a.qh);
  cudaError_t e = launch_pdl(chunk_attn_kernel<T, D>, grid, dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return cuda_error(e, "chunk attention launch");
  count_launches(1);
  return SAR_OK;
}

}  // namespace

int launch_chunk_attention(const ChunkAttnArgs& a, cudaStream_t s) {
  if (a.n_tiles <= 0) return SAR_OK;
  if (a.qh % a.kvh) return set_error(SAR_ERR_UNSUPPORTED, "chunk attention: qh % kvh");
  const bool bf = a.storage == SAR_STORAGE_BF16;
  if (a.d == 128) return bf ? launch_impl<__nv_bfloat16, 128>(a, s) : launch_impl<__half, 128>(a, s);
  if (a.d == 64) return bf ? launch_impl<__nv_bfloat16, 64>(a, s) : launch_impl<__half, 64>(a, s);
  return set_error(SAR_ERR_UNSUPPORTED, "chunk attention: head_dim must be 64 or 128");
}

}  // namespace sar
