// common.cuh -- device helpers shared by the codec and attention kernels
// (sm_103a): packed float32x2 arithmetic, bf16 unpacking, the MUFU log2,
// directed-rounding FMA, mbarrier waits with a bounded spin, and TMA loads.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lynx {

constexpr int kD = 128;            // channels per head supported by the kernels
constexpr float kEps = 1e-6f;      // epsilon of both normalisations
constexpr unsigned kFull = 0xffffffffu;

// --------------------------------------------------------------- f32x2

// Packed pair of floats; the arithmetic below maps to the sm_100 float2
// intrinsics, whose per-lane behaviour is that of the scalar _rn intrinsics
// (one IEEE rounding, never contracted into a fused multiply-add).
using f2 = float2;

__device__ __forceinline__ f2 add2(f2 a, f2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ f2 sub2(f2 a, f2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ f2 mul2(f2 a, f2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }

// --------------------------------------------------------------- scalar

__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// fma rounded toward -inf (one rounding).
__device__ __forceinline__ float fma_rm(float a, float b, float c) {
  float r;
  asm("fma.rm.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bf16x2 word -> two floats (exact).
__device__ __forceinline__ f2 bf2_to_f2(uint32_t w) {
  f2 r;
  r.x = __uint_as_float(w << 16);
  r.y = __uint_as_float(w & 0xffff0000u);
  return r;
}
// two floats -> bf16x2 word, round to nearest even (x in the low half).
__device__ __forceinline__ uint32_t f2_to_bf2(float x, float y) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
  return r;
}

// (lo(w) - c, hi(w) - c) for the two bf16 halves of w: each half converted
// exactly to f32, then one round-to-nearest subtraction.
__device__ __forceinline__ f2 bf2_sub_f32(uint32_t w, f2 c) {
  f2 r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
      " sub.rn.f32.bf16 %0, lo, %3;\n sub.rn.f32.bf16 %1, hi, %4;\n}"
      : "=f"(r.x), "=f"(r.y) : "r"(w), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Streaming 16-byte global load that bypasses L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ void stg_stream(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// --------------------------------------------------------------- paging

// Bits of the per-file device flag words (read through lynx_device_errors).
constexpr unsigned kFlagWaitTimeout = 1u;   // a bounded wait gave up
constexpr unsigned kFlagBadBlock = 2u;      // a block-table entry was out of range
constexpr unsigned kFlagBadToken = 4u;      // a draft token was outside the vocabulary
constexpr unsigned kFlagIndexCheck = 8u;    // checked build: an index check failed

// The checked build (compiled with -DLYNX_CHECKED) verifies the index
// arithmetic of every kernel at the points where it addresses global memory
// (TMA coordinates, bulk-copy offsets, block and row indices) against the
// extents that the call's shapes give.  An index outside [0, n) is recorded in
// *flag (bit kFlagIndexCheck, read through lynx_device_errors) and replaced by
// 0, so a bad index gives wrong numbers, never a stray access.  In the
// regular build the check compiles to nothing.
#ifdef LYNX_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ int64_t checked_index(int64_t i, int64_t n, unsigned int* flag) {
  if constexpr (kChecked) {
    if (i < 0 || i >= n) {
      atomicOr(flag, kFlagIndexCheck);
      return 0;
    }
  }
  return i;
}

// Physical page block of logical block blk = (b*NB + p)*H + h.  Without a
// block table the streams are dense and the two coincide; with one, row
// b*NB + p of the table names the physical page, whose H head blocks are
// contiguous.  An entry outside [0, nphys) is replaced by 0 and reported in
// *flag, so a bad table gives wrong numbers, never a stray access.
__device__ __forceinline__ int64_t phys_block(const int32_t* bt, int64_t nphys, int64_t blk,
                                              int H, unsigned int* flag) {
  if (!bt) return blk;
  const int64_t h = blk % H, row = blk / H;
  int64_t pg = __ldg(bt + row);
  if (pg < 0 || pg >= nphys) {
    atomicOr(flag, kFlagBadBlock);
    pg = 0;
  }
  return pg * H + h;
}

// --------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(phase) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false if the phase did not complete within kWaitNs (the
// caller then records the timeout and returns instead of hanging).
constexpr uint64_t kWaitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, phase))
    if (global_ns() - t0 > kWaitNs) return false;
  return true;
}

// --------------------------------------------------------------- TMA

// 2D tiled bulk tensor load global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// 1D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace lynx
