// Shared device helpers: bf16 packing, warp reductions, mbarrier / TMA / bulk
// copy wrappers with bounded waits, and the device error flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sar.h"

namespace sar {

// Device error record: [0] = first status code, [1] = site id, [2] = detail.
struct DevErr {
  int* flag;
};

// Sites reported in DevErr[1] when a wait gives up or a bounds check fires.
enum ErrSite {
  SITE_GEMM_PRODUCER = 1,
  SITE_GEMM_MMA = 2,
  SITE_GEMM_EPILOGUE = 3,
  SITE_DECODE_PIPE = 10,
  SITE_DECODE_BOUNDS = 11,
  SITE_CHUNK_BOUNDS = 20,
  SITE_CHUNK_PIPE = 21,
  SITE_ROPE_BOUNDS = 30,
  SITE_EMBED_BOUNDS = 40,
  SITE_WAIT_CHECK = 50,
};

// A wait that has not finished after this long gives up (normal waits take
// microseconds; a stuck pipeline must return rather than hold the GPU).  The
// step's kernels use this default; mbar_wait takes the limit as an argument.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void report(int* err, int code, int site, int detail) {
  if (err == nullptr) return;
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = site;
    err[2] = detail;
  }
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// silu(x) = x / (1 + e^-x) with the approximate exponential and divide: the
// result is rounded to 16 bits next, so their few-ulp fp32 errors never show,
// and an IEEE divide per element would take the epilogue warps' issue slots
// (which they share with the MMA-issuing warp).  For x below about -88 the
// denominator overflows and the approximate divide gives 0, the limit.  Every
// kernel that forms silu(gate) * up uses this one definition.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- bf16 helpers ----------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- warp reductions -------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// A waiting thread may be suspended up to this long per try (it resumes as
// soon as the phase completes), so polling warps take fewer issue slots.
constexpr uint32_t kTryWaitSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kTryWaitSuspendNs)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns (about; checked every 32 tries), records SAR_ERR_TIMEOUT at `site`
// and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err, int site,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      report(err, SAR_ERR_TIMEOUT, site, (int)parity);
      return false;
    }
  }
}

// ---- TMA / bulk copies -----------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Prefetch one tile of a tensor map into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(c0), "r"(c1)
               : "memory");
}

// Programmatic dependent launch.  pdl_wait(): until the previous kernel of the
// stream has completed and its writes are visible (returns at once for a
// kernel launched normally); nothing global that a previous kernel writes or
// reads may be touched before it.  pdl_launch_dependents(): the next kernel
// may start launching once every CTA of this one has called it or exited.
// Shared -> global tile reduction: adds the box at [src] (the tensor map's
// layout and swizzle) into the tensor at (c0, c1); element-wise atomic.
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(tmap), "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
// Shared -> global tile store of the box at [src] into the tensor at (c0, c1).
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(tmap), "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// All but the newest group have finished reading their shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Every committed group has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group has completed (its global writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Untiled bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---- cp.async (16 bytes, zero-fill when src_bytes == 0) ---------------------

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace sar

#include <cuda_fp16.h>

namespace sar {

// ---- storage element traits --------------------------------------------------
// The step stores activations, weights and the KV cache in one 16-bit type T
// (fp16 or bf16) and accumulates in fp32.  Elem<T> converts packed pairs.
template <typename T>
struct Elem;

template <>
struct Elem<__half> {
  static constexpr uint32_t kMmaFormat = 0;  // tcgen05 kind::f16 operand format: F16
  __device__ static __forceinline__ float lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
  }
  __device__ static __forceinline__ float hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
  }
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ __half from(float a) { return __float2half_rn(a); }
  __device__ static __forceinline__ float to(__half a) { return __half2float(a); }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr uint32_t kMmaFormat = 1;  // BF16
  __device__ static __forceinline__ float lo(uint32_t v) { return __uint_as_float(v << 16); }
  __device__ static __forceinline__ float hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ __nv_bfloat16 from(float a) { return __float2bfloat16_rn(a); }
  __device__ static __forceinline__ float to(__nv_bfloat16 a) { return __bfloat162float(a); }
};

}  // namespace sar
