// variants.cu -- the comparison points of "Lynx: Progressive Speculative KV
// Cache Transfer for Disaggregated LLM Inference" (technical review):
//
//  * the linear INT-B quantizer of Prerequisites Eq. 4 (the INT8 / INT4
//    baselines of the pages' tables), one scale and zero point per token and
//    KV head over its 128 channels;
//  * other Anchor/Residual bit splits (Concrete Improvement Suggestions,
//    items 4-5: 3+5, 5+3, 6+2): a re-split of the 4+4 streams into a k-bit
//    Anchor and an (8-k)-bit Residual of the same signed 8-bit code, the
//    inverse join, and the Anchor-only decode of a k-bit Anchor.
//
// All of it is streaming work, one pass over HBM: a warp per token row for
// INT-B (lane = 4 channels), a thread per (token, group of 8 channels) for
// the bit splits.  Grids are sized in whole waves of the SMs.
#include "common.cuh"
#include "internal.h"
#include "lynx.h"

namespace lynx {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ----------------------------------------------------------------- INT-B

// One token row of 128 BF16 channels per half-warp, 8 channels a lane (one
// 16-byte load), so a warp instruction serves two rows and the per-row work
// (min / max reduction, scale, reciprocal) spreads over 256 elements; R rows
// in flight per half-warp.
template <int BITS>
__global__ void __launch_bounds__(kThreads) int_encode_kernel(const uint8_t* __restrict__ x,
                                                              const int64_t rows,
                                                              uint8_t* __restrict__ codes,
                                                              float2* __restrict__ meta) {
  constexpr int R = 4;
  constexpr int qmax = (1 << BITS) - 1;
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const int64_t half = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 4;
  const int64_t nhalves = ((int64_t)gridDim.x * kThreads) >> 4;
  // both halves of a warp iterate the same number of times (rows are
  // assigned in whole warps), so the shuffles below always see 32 lanes
  const int64_t base0 = (half & ~1ll) * R;
  for (int64_t r0 = base0; r0 < rows; r0 += nhalves * R) {
    const int64_t myr0 = r0 + (half & 1) * R;
    uint4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
      v[i] = myr0 + i < rows ? ldg_stream(x + (myr0 + i) * 256 + hl * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int64_t row = myr0 + i;
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      // row minimum and maximum on bf16 pairs (exact), then the half-warp
      uint32_t mn2 = bf2_min(bf2_min(w[0], w[1]), bf2_min(w[2], w[3]));
      uint32_t mx2 = bf2_max(bf2_max(w[0], w[1]), bf2_max(w[2], w[3]));
#pragma unroll
      for (int o = 8; o; o >>= 1) {                // within the half-warp
        mn2 = bf2_min(mn2, __shfl_xor_sync(kFull, mn2, o));
        mx2 = bf2_max(mx2, __shfl_xor_sync(kFull, mx2, o));
      }
      float lo = fminf(bf16_lo(mn2), bf16_hi(mn2));
      float hi = fmaxf(bf16_lo(mx2), bf16_hi(mx2));
      if (row >= rows) continue;
      lo = __fadd_rn(lo, 0.0f);  // a zero extreme counts as +0
      hi = __fadd_rn(hi, 0.0f);
      const float S = __fdiv_rn(__fsub_rn(hi, lo), (float)qmax);
      const float rs = S > 0.0f ? __frcp_rn(S) : 0.0f;
      uint32_t q[8];
      const f2 lo2 = make_float2(lo, lo);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // (x - lo) rs per lane: the differences as a packed pair, the products
        // scalar __fmul_rn (never contracted into the add that follows); then
        // round to nearest even on the FMA pipe: for 0 <= y < 2^22 the bits of
        // y + 1.5 * 2^23 hold round(y) above 0x4B400000
        const f2 d = sub2(bf2_to_f2(w[j]), lo2);
        const f2 y = make_float2(__fmul_rn(d.x, rs), __fmul_rn(d.y, rs));
        const f2 t = add2(y, make_float2(12582912.0f, 12582912.0f));
        const int c0 = (int)__float_as_uint(t.x) - 0x4B400000, c1 = (int)__float_as_uint(t.y) - 0x4B400000;
        q[2 * j] = (uint32_t)(c0 < 0 ? 0 : c0 > qmax ? qmax : c0);
        q[2 * j + 1] = (uint32_t)(c1 < 0 ? 0 : c1 > qmax ? qmax : c1);
      }
      if constexpr (BITS == 8) {
        *reinterpret_cast<uint2*>(codes + row * 128 + hl * 8) =
            make_uint2(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24),
                       q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24));
      } else {
        *reinterpret_cast<uint32_t*>(codes + row * 64 + hl * 4) =
            q[0] | (q[1] << 4) | (q[2] << 8) | (q[3] << 12) | (q[4] << 16) | (q[5] << 20) |
            (q[6] << 24) | (q[7] << 28);
      }
      if (hl == 0) meta[row] = make_float2(lo, S);
    }
  }
}

template <int BITS, bool BF16OUT>
__global__ void __launch_bounds__(kThreads) int_decode_kernel(const uint8_t* __restrict__ codes,
                                                              const float2* __restrict__ meta,
                                                              const int64_t rows,
                                                              void* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t row = warp; row < rows; row += nwarps) {
    uint32_t q[4];
    if constexpr (BITS == 8) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(codes + row * 128 + lane * 4));
      q[0] = w & 0xff; q[1] = (w >> 8) & 0xff; q[2] = (w >> 16) & 0xff; q[3] = w >> 24;
    } else {
      const uint32_t w = __ldg(reinterpret_cast<const uint16_t*>(codes + row * 64 + lane * 2));
      q[0] = w & 0xf; q[1] = (w >> 4) & 0xf; q[2] = (w >> 8) & 0xf; q[3] = (w >> 12) & 0xf;
    }
    const float2 m = __ldg(meta + row);
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = __fmaf_rn((float)q[j], m.y, m.x);
    if constexpr (BF16OUT) {
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(out) + row * 256 + lane * 8) =
          make_uint2(f2_to_bf2(y[0], y[1]), f2_to_bf2(y[2], y[3]));
    } else {
      *reinterpret_cast<float4*>(static_cast<uint8_t*>(out) + row * 512 + lane * 16) =
          make_float4(y[0], y[1], y[2], y[3]);
    }
  }
}

// ---------------------------------------------------------- bit splits

// One thread per 4 consecutive groups (32 channels of one token row): the
// k-bit fields of the 8 codes' top bits of a group fill K bytes, the low 8-K
// bits 8-K bytes (channel j at bits j*w .. j*w + w - 1, little-endian), so 4
// groups are K and 8-K whole 32-bit words.
// Four W-bit fields held in the low bits of the four bytes of x, packed
// into the low 4W bits: byte pairs into 16-bit lanes, then the two lanes.
template <int W>
__device__ __forceinline__ uint32_t pack4(uint32_t x) {
  const uint32_t y = (x & 0x00ff00ffu) | ((x & 0xff00ff00u) >> (8 - W));
  return (y & 0x0000ffffu) | ((y & 0xffff0000u) >> (16 - 2 * W));
}

// n words from shared to global memory, 16 bytes an instruction where the
// destination allows (it does for every tile start: see the caller).
__device__ __forceinline__ void copy_out_words(const uint32_t* s, uint32_t* g, int n) {
  const int n4 = n >> 2;
  for (int j = threadIdx.x; j < n4; j += kThreads)
    reinterpret_cast<uint4*>(g)[j] = reinterpret_cast<const uint4*>(s)[j];
  for (int j = (n4 << 2) + threadIdx.x; j < n; j += kThreads) g[j] = s[j];
}

// A thread packs one quad (4 groups of 8 channels) into K words of the
// k-bit stream and 8-K words of the (8-k)-bit stream.  The words of a tile
// of kThreads quads are contiguous in each stream, so they are staged in
// shared memory and written out as whole 16-byte stores: written straight
// from the threads, every store instruction would hit K (or 8-K) partial
// sectors per 128 bytes.
template <int K>
__global__ void __launch_bounds__(kThreads) split_bits_kernel(const uint8_t* __restrict__ anchor,
                                                              const uint8_t* __restrict__ residual,
                                                              const int64_t groups,
                                                              uint8_t* __restrict__ ak,
                                                              uint8_t* __restrict__ rk) {
  constexpr int RW = 8 - K;
  constexpr uint32_t kMaskA = 0x01010101u * ((1u << K) - 1u);
  constexpr uint32_t kMaskR = 0x01010101u * ((1u << RW) - 1u);
  __shared__ __align__(16) uint32_t stage[kThreads * 8];
  uint32_t* sa = stage;                  // [kThreads][K]
  uint32_t* sr = stage + kThreads * K;   // [kThreads][8-K]
  const int64_t quads = groups / 4;
  const int64_t ntiles = (quads + kThreads - 1) / kThreads;
  for (int64_t ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
    const int64_t q0 = ti * kThreads, qi = q0 + threadIdx.x;
    const int nq = (int)(quads - q0 < kThreads ? quads - q0 : kThreads);
    if (qi < quads) {
      const uint4 a4 = __ldg(reinterpret_cast<const uint4*>(anchor) + qi);
      const uint4 r4 = __ldg(reinterpret_cast<const uint4*>(residual) + qi);
      const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w}, rw[4] = {r4.x, r4.y, r4.z, r4.w};
      // the four groups' k-bit (and 8-k bit) fields as one bit stream each, in
      // 32-bit words: group q's 8 fields fill bits 8K q .. 8K q + 8K - 1
      uint32_t oa[K], orr[RW];
      uint64_t acc_a = 0, acc_r = 0;
      int na = 0, nr = 0, ia = 0, ir = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // 8-bit codes of channels 0-3 (E) and 4-7 (O) of the group
        const uint32_t E = ((aw[q] << 4) & 0xf0f0f0f0u) | (rw[q] & 0x0f0f0f0fu);
        const uint32_t O = (aw[q] & 0xf0f0f0f0u) | ((rw[q] >> 4) & 0x0f0f0f0fu);
        const uint64_t fa = (uint64_t)pack4<K>((E >> RW) & kMaskA) |
                            ((uint64_t)pack4<K>((O >> RW) & kMaskA) << (4 * K));
        const uint64_t fr = (uint64_t)pack4<RW>(E & kMaskR) |
                            ((uint64_t)pack4<RW>(O & kMaskR) << (4 * RW));
        acc_a |= fa << na;
        na += 8 * K;
        while (na >= 32) {
          oa[ia++] = (uint32_t)acc_a;
          acc_a >>= 32;
          na -= 32;
        }
        acc_r |= fr << nr;
        nr += 8 * RW;
        while (nr >= 32) {
          orr[ir++] = (uint32_t)acc_r;
          acc_r >>= 32;
          nr -= 32;
        }
      }
#pragma unroll
      for (int i = 0; i < K; ++i) sa[threadIdx.x * K + i] = oa[i];
#pragma unroll
      for (int i = 0; i < RW; ++i) sr[threadIdx.x * RW + i] = orr[i];
    }
    __syncthreads();
    // tile ti starts at word q0*K (q0*(8-K)): byte offsets that are
    // multiples of 4 * kThreads, so 16-byte aligned
    copy_out_words(sa, reinterpret_cast<uint32_t*>(ak) + q0 * K, nq * K);
    copy_out_words(sr, reinterpret_cast<uint32_t*>(rk) + q0 * RW, nq * RW);
    __syncthreads();   // the stage is refilled by the next tile
  }
}

template <int K>
__global__ void __launch_bounds__(kThreads) join_bits_kernel(const uint8_t* __restrict__ ak,
                                                             const uint8_t* __restrict__ rk,
                                                             const int64_t groups,
                                                             uint32_t* __restrict__ anchor,
                                                             uint32_t* __restrict__ residual) {
  constexpr int RW = 8 - K;
  const int64_t quads = groups / 4;
  for (int64_t qi = (int64_t)blockIdx.x * kThreads + threadIdx.x; qi < quads;
       qi += (int64_t)gridDim.x * kThreads) {
    uint32_t ia[K], ir[RW];
#pragma unroll
    for (int i = 0; i < K; ++i) ia[i] = __ldg(reinterpret_cast<const uint32_t*>(ak) + qi * K + i);
#pragma unroll
    for (int i = 0; i < RW; ++i) ir[i] = __ldg(reinterpret_cast<const uint32_t*>(rk) + qi * RW + i);
    uint32_t a[4], r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint64_t fa = 0, fr = 0;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int byte = q * K + i;
        fa |= (uint64_t)((ia[byte >> 2] >> (8 * (byte & 3))) & 0xffu) << (8 * i);
      }
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        const int byte = q * RW + i;
        fr |= (uint64_t)((ir[byte >> 2] >> (8 * (byte & 3))) & 0xffu) << (8 * i);
      }
      uint32_t wa = 0, wr = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t q8 = ((uint32_t)(fa >> (j * K)) & ((1u << K) - 1u)) << RW |
                            ((uint32_t)(fr >> (j * RW)) & ((1u << RW) - 1u));
        const int sh = 8 * (j & 3) + ((j & 4) ? 4 : 0);  // byte j&3, high nibble for j >= 4
        wa |= (q8 >> 4) << sh;
        wr |= (q8 & 15u) << sh;
      }
      a[q] = wa;
      r[q] = wr;
    }
    reinterpret_cast<uint4*>(anchor)[qi] = make_uint4(a[0], a[1], a[2], a[3]);
    reinterpret_cast<uint4*>(residual)[qi] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// Anchor-only decode of a K-bit Anchor, the same reconstruction as the 4+4
// Anchor decoder with the bucket point I = 2^(8-K) V + 2^(7-K) - 1.  One
// persistent kernel: a CTA walks units of up to 256 tokens (a page block, or
// one half of a 512-token page), whose K-bit codes (unit x 16 K bytes) and
// metadata rows (for a half page: the gamma rows and the mu and sigma rows of
// its chunks) arrive in shared memory by bulk asynchronous copies, one stage
// ahead of the unit being decoded.  Thread (slot, G) of 256 decodes a run of
// unit/16 tokens (inside one chunk) of channels 8G..8G+7.  The K bytes of (token t, group G) start at byte (16 t + G) K of
// the block and lie in two consecutive 32-bit words ((o mod 4) + K <= 8: o
// is even when K = 6); the word after a block's last code is still inside
// the stage (its metadata follows), and the shift drops its bytes.
constexpr int kBitsStages = 2;
constexpr int kBitsUnit = 256;   // most tokens of a decode unit

// Set by a kernel of this file whose bounded wait on a stage gave up (it
// then returns early).  Read through read_variant_wait_timeout(); never reset.
__device__ unsigned int g_variant_wait_timeout = 0;

template <int K>
__host__ __device__ constexpr size_t bits_table_bytes() { return (size_t)(1 << K) * 32 * 4; }

template <int K, bool BF16OUT>
__global__ void __launch_bounds__(kThreads, 2)
decode_anchor_bits_kernel(const uint8_t* __restrict__ ak, const float* __restrict__ meta,
                          const int64_t nblk, const int64_t NB, const int H, const int64_t L,
                          const int P, const int C, void* __restrict__ out,
                          const __grid_constant__ ExpandTable tab) {
  static_assert(K >= 3 && K <= 6, "the K bytes of a code fit two 32-bit words");
  constexpr int NCODE = 1 << K;
  extern __shared__ __align__(16) uint8_t smem[];
  // the signed value of every K-bit Anchor code a (two's complement): S X(I)
  // with V = S > 0 ? a : -a - 1 and I = 2^(8-K) V + 2^(7-K) - 1; one copy a
  // lane (row a, column lane), so that every lane reads its own bank
  float* xk = reinterpret_cast<float*>(smem);
  const int U = P < kBitsUnit ? P : kBitsUnit;    // tokens of a unit
  const int parts = P / U;
  const int64_t nunit = nblk * parts;
  const uint32_t code_bytes = (uint32_t)U * 16 * K;
  const int NC = U / C, blk_meta_rows = 2 + 2 * (P / C);
  const uint32_t meta_bytes = (uint32_t)(2 + 2 * NC) * kD * 4;
  const uint32_t stage_bytes = code_bytes + meta_bytes;
  uint8_t* stages = smem + bits_table_bytes<K>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + kBitsStages * stage_bytes);
  const int tid = threadIdx.x, lane = tid & 31, G = tid & 15, slot = tid >> 4;
  const int run = U >> 4, t0 = slot * run, chunk = t0 / C;
  const int64_t ostride = (int64_t)H * kD;

  for (int i = tid; i < NCODE * 32; i += kThreads) {
    const int a = (i >> 5) >= NCODE / 2 ? (i >> 5) - NCODE : (i >> 5);
    const float m = tab.x[(1 << (8 - K)) * (a >= 0 ? a : -a - 1) + (1 << (7 - K)) - 1];
    xk[i] = a >= 0 ? m : -m;
  }
  if (tid == 0) {
    for (int i = 0; i < kBitsStages; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const float* xl = xk + lane;

  auto issue = [&](int64_t un, int stage) {
    un = checked_index(un, nunit, &g_variant_wait_timeout);
    const int64_t blk = un / parts, part = un % parts;
    uint8_t* st = stages + stage * stage_bytes;
    mbar_expect_tx(&bars[stage], stage_bytes);
    bulk_load(st, ak + un * code_bytes, code_bytes, &bars[stage]);
    const float* mb = meta + blk * (int64_t)blk_meta_rows * kD;
    if (parts == 1) {
      bulk_load(st + code_bytes, mb, meta_bytes, &bars[stage]);
    } else {  // gamma rows, then the unit's mu rows and sigma rows
      const uint32_t rows = (uint32_t)NC * kD * 4;
      bulk_load(st + code_bytes, mb, 2 * kD * 4, &bars[stage]);
      bulk_load(st + code_bytes + 2 * kD * 4, mb + (2 + part * NC) * kD, rows, &bars[stage]);
      bulk_load(st + code_bytes + 2 * kD * 4 + rows, mb + (2 + P / C + part * NC) * kD, rows,
                &bars[stage]);
    }
  };
  if (tid == 0)
    for (int i = 0; i < kBitsStages; ++i) {
      const int64_t un = blockIdx.x + (int64_t)i * gridDim.x;
      if (un < nunit) issue(un, i);
    }

  int it = 0;
  for (int64_t un = blockIdx.x; un < nunit; un += gridDim.x, ++it) {
    const int stage = it % kBitsStages;
    const uint32_t phase = (uint32_t)(it / kBitsStages) & 1u;
    const bool ok = mbar_wait(&bars[stage], phase);
    const uint8_t* st = stages + stage * stage_bytes;
    const float* mrow = reinterpret_cast<const float*>(st + code_bytes) + 8 * G;
    f2 gm[4], gs[4], mu[4], sg[4];
    auto row8 = [&](const float* r, f2 (&v)[4], bool eps) {
      const float4 u0 = reinterpret_cast<const float4*>(r)[0];
      const float4 u1 = reinterpret_cast<const float4*>(r)[1];
      v[0] = make_float2(u0.x, u0.y);
      v[1] = make_float2(u0.z, u0.w);
      v[2] = make_float2(u1.x, u1.y);
      v[3] = make_float2(u1.z, u1.w);
      if (eps) {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = add2(v[j], make_float2(kEps, kEps));
      }
    };
    row8(mrow, gm, false);
    row8(mrow + kD, gs, true);
    row8(mrow + (2 + chunk) * kD, mu, false);
    row8(mrow + (2 + NC + chunk) * kD, sg, true);
    const int64_t blk = un / parts, part = un % parts;
    const int64_t h = blk % H, rest = blk / H;
    const int64_t p = rest % NB, b = rest / NB;
    const int64_t row0 = checked_index(b * L + p * P + part * U + t0, nblk / H * P - run + 1,
                                       &g_variant_wait_timeout);
    const int64_t orow0 = (row0 * H + h) * kD + 8 * G;
#pragma unroll 4
    for (int r = 0; r < run; ++r) {
      const uint32_t o = (uint32_t)((t0 + r) * 16 + G) * K;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(st) + (o >> 2);
      const uint64_t fa = (((uint64_t)w[1] << 32) | w[0]) >> (8 * (o & 3));
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = xl[((uint32_t)(fa >> (j * K)) & (NCODE - 1u)) * 32u];
      f2 y[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        y[j] = fma2(fma2(make_float2(v[2 * j], v[2 * j + 1]), sg[j], mu[j]), gs[j], gm[j]);
      char* ob = reinterpret_cast<char*>(out);
      const int64_t oe = orow0 + (int64_t)r * ostride;
      if constexpr (BF16OUT) {
        stg_stream(ob + oe * 2, make_uint4(f2_to_bf2(y[0].x, y[0].y), f2_to_bf2(y[1].x, y[1].y),
                                           f2_to_bf2(y[2].x, y[2].y), f2_to_bf2(y[3].x, y[3].y)));
      } else {
        stg_stream(ob + oe * 4, make_uint4(__float_as_uint(y[0].x), __float_as_uint(y[0].y),
                                           __float_as_uint(y[1].x), __float_as_uint(y[1].y)));
        stg_stream(ob + oe * 4 + 16, make_uint4(__float_as_uint(y[2].x), __float_as_uint(y[2].y),
                                                __float_as_uint(y[3].x), __float_as_uint(y[3].y)));
      }
    }

    if (!__syncthreads_and(ok)) {
      // a stage never arrived: record it and stop this CTA (bounded waits)
      if (tid == 0) {
        atomicOr(&g_variant_wait_timeout, kFlagWaitTimeout);
        for (int i = 0; i < kBitsStages; ++i) (void)mbar_wait(&bars[i], phase);
      }
      return;
    }
    // every thread is done with this stage: refill it kBitsStages units ahead
    if (tid == 0) {
      const int64_t nxt = un + (int64_t)kBitsStages * gridDim.x;
      if (nxt < nunit) {
        fence_proxy_async();
        issue(nxt, stage);
      }
    }
  }
}

// ---------------------------------------------------------- Appendix A.1

// One CTA per page block, one thread per (16-token chunk k, group G of 8
// channels): P threads.  A thread reads its chunk's 16 rows of 16 bytes
// twice: once for the maxima, once (from L1/L2) for the codes, which keeps
// its registers, and so the warps an SM holds, at twice what keeping the
// rows would allow.  The page maximum of |x| (exact, on bf16 pairs) combines
// the chunks' maxima through shared memory.  The chunk maximum of |x'| = |x| rm
// is rn(max|x| rm): rounding is monotone.  |Q| comes from the encoder's fast
// rounding, run on pairs of channels, with the host thresholds of Eq. 7
// (|Q| = #{k : a >= thr[k]}) deciding inside its window, or from a binary
// search over the thresholds for alpha < 1.  The codes leave as one 32-bit
// word per stream and token: byte j holds channel 8G + j in the low nibble
// and 8G + j + 4 in the high one.
constexpr int kA1Chunk = 16;

// prmt.b32 in its default mode: a selector digit of 8 or more replicates
// the sign bit of the byte it names.
__device__ __forceinline__ uint32_t a1_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// |Q| = Round(Y(a)) of Eq. 7.  FAST (alpha >= 1): the encoder's Stage-3 fast
// path per lane (t = rn(alpha a + 1), MUFU lg2, s = rd(lg2(t) c16 + C0): the
// code in byte 2, its distance to the rounding boundary in the low 16 bits),
// the same operations whose window the exhaustive self-check verifies, with
// the threshold deciding inside the window; otherwise a binary search over
// the thresholds.
constexpr float kA1C0 = 8388608.0f + 32768.0f + (float)kAmbiguityK;
template <bool FAST>
__device__ __forceinline__ int a1_round(float a, float alpha, float c16, const float* thr) {
  if constexpr (FAST) {
    const float t = __fmaf_rn(alpha, a, 1.0f);
    const uint32_t bits = __float_as_uint(fma_rm(lg2_approx(t), c16, kA1C0));
    int I = (int)((bits >> 16) & 0xffu);
    if ((bits & 0xffffu) < 2u * kAmbiguityK) {
      const int b = I > 0 ? I - 1 : 0;
      I = b + (a >= thr[b] ? 1 : 0);
    }
    return I;
  } else {
    int I = 0;                                     // #{k < 127 : a >= thr[k]}
#pragma unroll
    for (int step = 64; step; step >>= 1)
      if (I + step <= 127 && a >= thr[I + step - 1]) I += step;
    return I;
  }
}

template <bool FAST>
__global__ void __launch_bounds__(512)
a1_encode_kernel(const uint8_t* __restrict__ kv, const int64_t NB, const int H, const int64_t L,
                 const int P, uint32_t* __restrict__ anchor, uint32_t* __restrict__ residual,
                 float* __restrict__ meta, const __grid_constant__ CompanderTable tab) {
  __shared__ float thr[128];
  __shared__ uint4 pmx[32][16];                  // [chunk][group]: bf16x2 maxima of |x|
  const int tid = threadIdx.x, G = tid & 15, k = tid >> 4;
  const int64_t blk = blockIdx.x;
  const int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);
  for (int i = tid; i < 128; i += P) thr[i] = tab.thr[i];   // P >= 64 threads
  const uint8_t* src = kv + ((b * L + p * P + k * kA1Chunk) * H + h) * 256 + 16 * G;
  // pass 1: the chunk maxima only; pass 2 reads the rows again (from L1/L2)
  // rather than holding them, to keep registers low
  uint32_t cm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int t = 0; t < kA1Chunk; ++t) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)t * H * 256));
    cm[0] = bf2_max(cm[0], v.x & 0x7fff7fffu);
    cm[1] = bf2_max(cm[1], v.y & 0x7fff7fffu);
    cm[2] = bf2_max(cm[2], v.z & 0x7fff7fffu);
    cm[3] = bf2_max(cm[3], v.w & 0x7fff7fffu);
  }
  pmx[k][G] = make_uint4(cm[0], cm[1], cm[2], cm[3]);
  __syncthreads();
  uint32_t pm[4] = {0u, 0u, 0u, 0u};
  for (int c = 0; c < P / kA1Chunk; ++c) {
    const uint4 v = pmx[c][G];
    pm[0] = bf2_max(pm[0], v.x);
    pm[1] = bf2_max(pm[1], v.y);
    pm[2] = bf2_max(pm[2], v.z);
    pm[3] = bf2_max(pm[3], v.w);
  }
  // per channel pair j: page max m, rm = 1/m, chunk max mi, rmi = 1/mi
  const int NCk = P / kA1Chunk;
  float* mrow = meta + blk * (int64_t)(1 + NCk) * kD + 8 * G;
  f2 rm2[4], rmi2[4];
  float mv[8], miv[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const f2 m = bf2_to_f2(pm[j]), cx = bf2_to_f2(cm[j]);
    rm2[j] = make_float2(m.x > 0.0f ? __frcp_rn(m.x) : 0.0f, m.y > 0.0f ? __frcp_rn(m.y) : 0.0f);
    // an infinite input makes rm 0 and this product NaN; the chunk's finite
    // values then give 0
    const float m0 = fmaxf(__fmul_rn(cx.x, rm2[j].x), 0.0f);
    const float m1 = fmaxf(__fmul_rn(cx.y, rm2[j].y), 0.0f);
    rmi2[j] = make_float2(m0 > 0.0f ? __frcp_rn(m0) : 0.0f, m1 > 0.0f ? __frcp_rn(m1) : 0.0f);
    mv[2 * j] = m.x;
    mv[2 * j + 1] = m.y;
    miv[2 * j] = m0;
    miv[2 * j + 1] = m1;
  }
  if (k == 0) {
    reinterpret_cast<float4*>(mrow)[0] = make_float4(mv[0], mv[1], mv[2], mv[3]);
    reinterpret_cast<float4*>(mrow)[1] = make_float4(mv[4], mv[5], mv[6], mv[7]);
  }
  reinterpret_cast<float4*>(mrow + (1 + k) * kD)[0] = make_float4(miv[0], miv[1], miv[2], miv[3]);
  reinterpret_cast<float4*>(mrow + (1 + k) * kD)[1] = make_float4(miv[4], miv[5], miv[6], miv[7]);

  const f2 alpha2 = make_float2(tab.alpha, tab.alpha), c16_2 = make_float2(tab.c16, tab.c16);
  uint32_t* arow = anchor + (blk * P + k * kA1Chunk) * 16 + G;
  uint32_t* rrow = residual + (blk * P + k * kA1Chunk) * 16 + G;
#pragma unroll 4
  for (int t = 0; t < kA1Chunk; ++t) {
    const uint4 wt = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)t * H * 256));
    const uint32_t wj[4] = {wt.x, wt.y, wt.z, wt.w};
    uint32_t bits[8], sbits[8];
    float av[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const f2 xpp = mul2(mul2(bf2_to_f2(wj[j]), rm2[j]), rmi2[j]);
      sbits[2 * j] = __float_as_uint(xpp.x);
      sbits[2 * j + 1] = __float_as_uint(xpp.y);
      // |x''| <= 1 up to rounding; a NaN (only) fails the test and codes as 0
      float a0 = fabsf(xpp.x), a1 = fabsf(xpp.y);
      a0 = a0 <= 2.0f ? a0 : 0.0f;
      a1 = a1 <= 2.0f ? a1 : 0.0f;
      av[2 * j] = a0;
      av[2 * j + 1] = a1;
      if constexpr (FAST) {
        const f2 tt = __ffma2_rn(alpha2, make_float2(a0, a1), make_float2(1.0f, 1.0f));
        const f2 s = __ffma2_rd(make_float2(lg2_approx(tt.x), lg2_approx(tt.y)), c16_2,
                                make_float2(kA1C0, kA1C0));
        bits[2 * j] = __float_as_uint(s.x);
        bits[2 * j + 1] = __float_as_uint(s.y);
      } else {
        bits[2 * j] = (uint32_t)a1_round<false>(a0, tab.alpha, tab.c16, thr) << 16;
        bits[2 * j + 1] = (uint32_t)a1_round<false>(a1, tab.alpha, tab.c16, thr) << 16;
      }
    }
    if constexpr (FAST) {
      // a 16-bit-lane minimum over the words, then one test of the low half
      const uint32_t d01 = __vminu2(bits[0], bits[1]), d23 = __vminu2(bits[2], bits[3]);
      const uint32_t d45 = __vminu2(bits[4], bits[5]), d67 = __vminu2(bits[6], bits[7]);
      const uint32_t dmin = __vminu2(__vminu2(d01, d23), __vminu2(d45, d67));
      if ((dmin & 0xffffu) < 2u * kAmbiguityK) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((bits[i] & 0xffffu) < 2u * kAmbiguityK) {
            const int I = (int)((bits[i] >> 16) & 0xffu), bb = I > 0 ? I - 1 : 0;
            bits[i] = (bits[i] & 0xff00ffffu) | ((uint32_t)(bb + (av[i] >= thr[bb] ? 1 : 0)) << 16);
          }
      }
    }
    // |Q| bytes of channels 0-3 and 4-7, negated where x'' < 0 (two's complement)
    const uint32_t i01 = a1_prmt(bits[0], bits[1], 0x0062u), i23 = a1_prmt(bits[2], bits[3], 0x0062u);
    const uint32_t i45 = a1_prmt(bits[4], bits[5], 0x0062u), i67 = a1_prmt(bits[6], bits[7], 0x0062u);
    const uint32_t s01 = a1_prmt(sbits[0], sbits[1], 0x00fbu), s23 = a1_prmt(sbits[2], sbits[3], 0x00fbu);
    const uint32_t s45 = a1_prmt(sbits[4], sbits[5], 0x00fbu), s67 = a1_prmt(sbits[6], sbits[7], 0x00fbu);
    const uint32_t I0 = a1_prmt(i01, i23, 0x5410u), S0 = a1_prmt(s01, s23, 0x5410u);
    const uint32_t I1 = a1_prmt(i45, i67, 0x5410u), S1 = a1_prmt(s45, s67, 0x5410u);
    const uint32_t W0 = __vsub4(I0 ^ S0, S0), W1 = __vsub4(I1 ^ S1, S1);
    arow[t * 16] = ((W0 >> 4) & 0x0f0f0f0fu) | (W1 & 0xf0f0f0f0u);
    rrow[t * 16] = (W0 & 0x0f0f0f0fu) | ((W1 << 4) & 0xf0f0f0f0u);
  }
}

// Decode of the A.1 variant, persistent, like the 4+4 decoders: a block's
// Anchor and Residual codes and its metadata rows (m, then m_i per 16-token
// chunk) arrive in shared memory by bulk asynchronous copies, one stage
// ahead; thread (slot, G) of 256 decodes a run of page/16 tokens (one chunk
// or part of one, two chunks at page 512) of channels 8G..8G+7.  The 8-bit code of a channel, Anchor nibble
// above Residual nibble (Residual 7 in Anchor-only mode), read as an int8 is
// Q; a lane-replicated table over that byte gives sgn(Q) X(min(|Q|, 127)).
constexpr int kA1Stages = 2;
constexpr size_t kA1Table = 256 * 32 * 4;

template <bool FULL, bool BF16OUT>
__global__ void __launch_bounds__(kThreads, 2)
a1_decode_kernel(const uint8_t* __restrict__ anchor, const uint8_t* __restrict__ residual,
                 const float* __restrict__ meta, const int64_t nblk, const int64_t NB,
                 const int H, const int64_t L, const int P, void* __restrict__ out,
                 const __grid_constant__ ExpandTable tab) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xq = reinterpret_cast<float*>(smem);     // [byte][lane]
  const uint32_t code_bytes = (uint32_t)P * (kD / 2);
  const int NCk = P / kA1Chunk;
  const uint32_t meta_bytes = (uint32_t)(1 + NCk) * kD * 4;
  const uint32_t stage_bytes = code_bytes * (FULL ? 2 : 1) + meta_bytes;
  uint8_t* stages = smem + kA1Table;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + kA1Stages * stage_bytes);
  const int tid = threadIdx.x, lane = tid & 31, G = tid & 15, slot = tid >> 4;
  const int run = P >> 4, t0 = slot * run, chunk = t0 / kA1Chunk;
  const int64_t ostride = (int64_t)H * kD;

  for (int i = tid; i < 256 * 32; i += kThreads) {
    const int Q = (int)(int8_t)(uint8_t)(i >> 5);
    const int I = Q < 0 ? (-Q > 127 ? 127 : -Q) : Q;
    xq[i] = Q < 0 ? -tab.x[I] : tab.x[I];
  }
  if (tid == 0) {
    for (int i = 0; i < kA1Stages; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const uint32_t tbase = smem_u32(xq) + (uint32_t)lane * 4u;
  // table value of byte POS of w
  auto lut = [&](uint32_t w, int pos) -> float {
    float v;
    const uint32_t addr = tbase + (((w >> (8 * pos)) & 0xffu) << 7);
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
  };

  auto issue = [&](int64_t blk, int stage) {
    uint8_t* st = stages + stage * stage_bytes;
    mbar_expect_tx(&bars[stage], stage_bytes);
    bulk_load(st, anchor + blk * code_bytes, code_bytes, &bars[stage]);
    if constexpr (FULL) bulk_load(st + code_bytes, residual + blk * code_bytes, code_bytes, &bars[stage]);
    bulk_load(st + code_bytes * (FULL ? 2 : 1), meta + blk * (int64_t)(1 + NCk) * kD, meta_bytes,
              &bars[stage]);
  };
  if (tid == 0)
    for (int i = 0; i < kA1Stages; ++i) {
      const int64_t blk = blockIdx.x + (int64_t)i * gridDim.x;
      if (blk < nblk) issue(blk, i);
    }

  int it = 0;
  for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++it) {
    const int stage = it % kA1Stages;
    const uint32_t phase = (uint32_t)(it / kA1Stages) & 1u;
    const bool ok = mbar_wait(&bars[stage], phase);
    const uint8_t* st = stages + stage * stage_bytes;
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(st) + t0 * 16 + G;
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(st + code_bytes) + t0 * 16 + G;
    const float* mrow = reinterpret_cast<const float*>(st + code_bytes * (FULL ? 2 : 1)) + 8 * G;
    f2 m2[4], mi2[4];
    {
      const float4 u0 = reinterpret_cast<const float4*>(mrow)[0];
      const float4 u1 = reinterpret_cast<const float4*>(mrow)[1];
      const float4 v0 = reinterpret_cast<const float4*>(mrow + (1 + chunk) * kD)[0];
      const float4 v1 = reinterpret_cast<const float4*>(mrow + (1 + chunk) * kD)[1];
      m2[0] = make_float2(u0.x, u0.y); m2[1] = make_float2(u0.z, u0.w);
      m2[2] = make_float2(u1.x, u1.y); m2[3] = make_float2(u1.z, u1.w);
      mi2[0] = make_float2(v0.x, v0.y); mi2[1] = make_float2(v0.z, v0.w);
      mi2[2] = make_float2(v1.x, v1.y); mi2[3] = make_float2(v1.z, v1.w);
    }
    const int64_t h = blk % H, rest = blk / H;
    const int64_t p = rest % NB, b = rest / NB;
    const int64_t orow0 = ((b * L + p * P + t0) * H + h) * kD + 8 * G;
    // a run lies in one chunk up to pages of 256 and spans two at 512: the
    // chunk factors are reloaded at each 16-token boundary
    for (int r0 = 0; r0 < run; r0 += kA1Chunk) {
      if (r0 > 0) {
        const float* crow = mrow + (1 + (t0 + r0) / kA1Chunk) * kD;
        const float4 v0 = reinterpret_cast<const float4*>(crow)[0];
        const float4 v1 = reinterpret_cast<const float4*>(crow)[1];
        mi2[0] = make_float2(v0.x, v0.y); mi2[1] = make_float2(v0.z, v0.w);
        mi2[2] = make_float2(v1.x, v1.y); mi2[3] = make_float2(v1.z, v1.w);
      }
      const int r1 = run < r0 + kA1Chunk ? run : r0 + kA1Chunk;
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
      const uint32_t a = aw[r * 16], rr = FULL ? rw[r * 16] : 0x77777777u;
      const uint32_t E = ((a << 4) & 0xf0f0f0f0u) | (rr & 0x0f0f0f0fu);  // codes of ch 0-3
      const uint32_t O = (a & 0xf0f0f0f0u) | ((rr >> 4) & 0x0f0f0f0fu);  // codes of ch 4-7
      const f2 v[4] = {make_float2(lut(E, 0), lut(E, 1)), make_float2(lut(E, 2), lut(E, 3)),
                       make_float2(lut(O, 0), lut(O, 1)), make_float2(lut(O, 2), lut(O, 3))};
      f2 y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = mul2(mul2(v[k], mi2[k]), m2[k]);
      char* ob = reinterpret_cast<char*>(out);
      const int64_t oe = orow0 + (int64_t)r * ostride;
      if constexpr (BF16OUT) {
        stg_stream(ob + oe * 2, make_uint4(f2_to_bf2(y[0].x, y[0].y), f2_to_bf2(y[1].x, y[1].y),
                                           f2_to_bf2(y[2].x, y[2].y), f2_to_bf2(y[3].x, y[3].y)));
      } else {
        stg_stream(ob + oe * 4, make_uint4(__float_as_uint(y[0].x), __float_as_uint(y[0].y),
                                           __float_as_uint(y[1].x), __float_as_uint(y[1].y)));
        stg_stream(ob + oe * 4 + 16, make_uint4(__float_as_uint(y[2].x), __float_as_uint(y[2].y),
                                                __float_as_uint(y[3].x), __float_as_uint(y[3].y)));
      }
    }
    }

    if (!__syncthreads_and(ok)) {
      // a stage never arrived: record it and stop this CTA (bounded waits)
      if (tid == 0) {
        atomicOr(&g_variant_wait_timeout, kFlagWaitTimeout);
        for (int i = 0; i < kA1Stages; ++i) (void)mbar_wait(&bars[i], phase);
      }
      return;
    }
    if (tid == 0) {
      const int64_t nxt = blk + (int64_t)kA1Stages * gridDim.x;
      if (nxt < nblk) {
        fence_proxy_async();
        issue(nxt, stage);
      }
    }
  }
}

unsigned grid_for(int64_t work_items, int per_block) {
  const int64_t waves = (int64_t)sm_count() * 8;  // 8 CTAs of 256 threads per SM
  const int64_t need = (work_items + per_block - 1) / per_block;
  return (unsigned)(need < waves ? (need > 0 ? need : 1) : waves);
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

cudaError_t read_variant_wait_timeout(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_variant_wait_timeout, sizeof(unsigned int));
}

template <int K, bool BF16OUT>
static cudaError_t run_decode_bits(const uint8_t* ak, const float* meta, const Shape& s,
                                   const ExpandTable& tab, void* out, cudaStream_t stream) {
  auto fn = decode_anchor_bits_kernel<K, BF16OUT>;
  const int U = s.page < kBitsUnit ? s.page : kBitsUnit;
  const size_t stage = (size_t)U * 16 * K + (size_t)(2 + 2 * (U / s.C)) * kD * 4;
  const size_t smem = bits_table_bytes<K>() + kBitsStages * stage + kBitsStages * 8;
  constexpr size_t kMaxSmem = bits_table_bytes<K>() + kBitsStages * (256 * 16 * K + 34 * kD * 4) + 64;
  static thread_local int configured_dev = -1;
  static thread_local size_t last_smem = 0;
  static thread_local int per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
    last_smem = 0;
  }
  if (smem != last_smem) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
    last_smem = smem;
  }
  const int64_t nblk = s.blocks();
  int64_t grid = (int64_t)sm_count() * per_sm;
  if (grid > nblk * (s.page / U)) grid = nblk * (s.page / U);
  fn<<<(unsigned)grid, kThreads, smem, stream>>>(ak, meta, nblk, s.NB(), s.H, s.L, s.page, s.C,
                                                 out, tab);
  return cudaGetLastError();
}

cudaError_t launch_decode_anchor_bits(const void* ak, const float* meta, const Shape& s, int k,
                                      const ExpandTable& tab, void* out, bool bf16_out,
                                      cudaStream_t stream) {
  if (s.blocks() == 0) return cudaSuccess;
  const uint8_t* a = static_cast<const uint8_t*>(ak);
#define LYNX_DAB(KK)                                                                      \
  if (k == KK)                                                                            \
    return bf16_out ? run_decode_bits<KK, true>(a, meta, s, tab, out, stream)             \
                    : run_decode_bits<KK, false>(a, meta, s, tab, out, stream);
  LYNX_DAB(3)
  LYNX_DAB(4)
  LYNX_DAB(5)
  LYNX_DAB(6)
#undef LYNX_DAB
  return cudaErrorInvalidValue;
}

cudaError_t launch_a1_encode(const void* kv, const Shape& s, const CompanderTable& tab,
                             void* anchor, void* residual, float* meta, cudaStream_t stream) {
  const int64_t nblk = s.blocks();
  if (nblk > 0x7fffffff) return cudaErrorInvalidValue;
  auto fn = tab.alpha >= kMinEncodeAlpha ? a1_encode_kernel<true> : a1_encode_kernel<false>;
  fn<<<(unsigned)nblk, (unsigned)s.page, 0, stream>>>(
      static_cast<const uint8_t*>(kv), s.NB(), s.H, s.L, s.page, static_cast<uint32_t*>(anchor),
      static_cast<uint32_t*>(residual), meta, tab);
  return cudaGetLastError();
}

template <bool FULL, bool BF16OUT>
static cudaError_t run_a1_decode(const uint8_t* a, const uint8_t* r, const float* meta,
                                 const Shape& s, const ExpandTable& tab, void* out,
                                 cudaStream_t stream) {
  auto fn = a1_decode_kernel<FULL, BF16OUT>;
  const size_t stage = (size_t)s.page * (kD / 2) * (FULL ? 2 : 1) +
                       (size_t)(1 + s.page / kA1Chunk) * kD * 4;
  const size_t smem = kA1Table + kA1Stages * stage + kA1Stages * 8;
  constexpr size_t kMaxSmem = kA1Table + kA1Stages * (512 * 64 * 2 + 33 * kD * 4) + 64;
  static thread_local int configured_dev = -1;
  static thread_local size_t last_smem = 0;
  static thread_local int per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
    last_smem = 0;
  }
  if (smem != last_smem) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
    last_smem = smem;
  }
  const int64_t nblk = s.blocks();
  int64_t grid = (int64_t)sm_count() * per_sm;
  if (grid > nblk) grid = nblk;
  fn<<<(unsigned)grid, kThreads, smem, stream>>>(a, r, meta, nblk, s.NB(), s.H, s.L, s.page,
                                                 out, tab);
  return cudaGetLastError();
}

cudaError_t launch_a1_decode(const void* anchor, const void* residual, const float* meta,
                             const Shape& s, const ExpandTable& tab, void* out, bool bf16_out,
                             cudaStream_t stream) {
  if (s.blocks() == 0) return cudaSuccess;
  const uint8_t* a = static_cast<const uint8_t*>(anchor);
  const uint8_t* r = static_cast<const uint8_t*>(residual);
  if (r)
    return bf16_out ? run_a1_decode<true, true>(a, r, meta, s, tab, out, stream)
                    : run_a1_decode<true, false>(a, r, meta, s, tab, out, stream);
  return bf16_out ? run_a1_decode<false, true>(a, nullptr, meta, s, tab, out, stream)
                  : run_a1_decode<false, false>(a, nullptr, meta, s, tab, out, stream);
}

}  // namespace lynx

using namespace lynx;

extern "C" {

int lynx_int_encode(const void* kv, int64_t rows, int D, int bits, void* codes, float* meta,
                    void* stream) {
  if (D != kD) return report_error(LYNX_EUNSUPPORTED, "only D = 128 is built");
  if (bits != 4 && bits != 8) return report_error(LYNX_EUNSUPPORTED, "bits must be 4 or 8");
  if (rows < 0) return report_error(LYNX_ESHAPE, "rows must be >= 0");
  if (rows == 0) return LYNX_OK;
  if (!kv || !codes || !meta) return report_error(LYNX_EINVAL, "null pointer");
  if (!aligned(kv, 16) || !aligned(codes, 16) || !aligned(meta, 16))
    return report_error(LYNX_EINVAL, "pointer not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = grid_for((rows + 7) / 8, kThreads / 32);  // 2 halves x 4 rows a warp
  if (bits == 8)
    int_encode_kernel<8><<<grid, kThreads, 0, st>>>(static_cast<const uint8_t*>(kv), rows,
                                                    static_cast<uint8_t*>(codes),
                                                    reinterpret_cast<float2*>(meta));
  else
    int_encode_kernel<4><<<grid, kThreads, 0, st>>>(static_cast<const uint8_t*>(kv), rows,
                                                    static_cast<uint8_t*>(codes),
                                                    reinterpret_cast<float2*>(meta));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_error(LYNX_ECUDA, cudaGetErrorString(e));
  return LYNX_OK;
}

int lynx_int_decode(const void* codes, const float* meta, int64_t rows, int D, int bits,
                    void* out, int out_dtype, void* stream) {
  if (D != kD) return report_error(LYNX_EUNSUPPORTED, "only D = 128 is built");
  if (bits != 4 && bits != 8) return report_error(LYNX_EUNSUPPORTED, "bits must be 4 or 8");
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return report_error(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  if (rows < 0) return report_error(LYNX_ESHAPE, "rows must be >= 0");
  if (rows == 0) return LYNX_OK;
  if (!codes || !meta || !out) return report_error(LYNX_EINVAL, "null pointer");
  if (!aligned(codes, 16) || !aligned(meta, 16) || !aligned(out, 16))
    return report_error(LYNX_EINVAL, "pointer not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = grid_for(rows, kThreads / 32);
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  const float2* m = reinterpret_cast<const float2*>(meta);
  const bool b16 = out_dtype == LYNX_OUT_BF16;
  if (bits == 8 && b16) int_decode_kernel<8, true><<<grid, kThreads, 0, st>>>(c, m, rows, out);
  if (bits == 8 && !b16) int_decode_kernel<8, false><<<grid, kThreads, 0, st>>>(c, m, rows, out);
  if (bits == 4 && b16) int_decode_kernel<4, true><<<grid, kThreads, 0, st>>>(c, m, rows, out);
  if (bits == 4 && !b16) int_decode_kernel<4, false><<<grid, kThreads, 0, st>>>(c, m, rows, out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_error(LYNX_ECUDA, cudaGetErrorString(e));
  return LYNX_OK;
}

int lynx_split_bits(const void* anchor, const void* residual, int64_t rows, int D, int k,
                    void* anchor_k, void* residual_k, void* stream) {
  if (D != kD) return report_error(LYNX_EUNSUPPORTED, "only D = 128 is built");
  if (k < 3 || k > 6) return report_error(LYNX_EUNSUPPORTED, "k must be 3, 4, 5 or 6");
  if (rows < 0) return report_error(LYNX_ESHAPE, "rows must be >= 0");
  if (rows == 0) return LYNX_OK;
  if (!anchor || !residual || !anchor_k || !residual_k)
    return report_error(LYNX_EINVAL, "null pointer");
  if (!aligned(anchor, 16) || !aligned(residual, 16) || !aligned(anchor_k, 16) ||
      !aligned(residual_k, 16))
    return report_error(LYNX_EINVAL, "pointer not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t groups = rows * (kD / 8);
  const unsigned grid = grid_for(groups / 4, kThreads);
  const uint8_t* a = static_cast<const uint8_t*>(anchor);
  const uint8_t* r = static_cast<const uint8_t*>(residual);
  uint8_t* ao = static_cast<uint8_t*>(anchor_k);
  uint8_t* ro = static_cast<uint8_t*>(residual_k);
  if (k == 3) split_bits_kernel<3><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 4) split_bits_kernel<4><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 5) split_bits_kernel<5><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 6) split_bits_kernel<6><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_error(LYNX_ECUDA, cudaGetErrorString(e));
  return LYNX_OK;
}

int lynx_join_bits(const void* anchor_k, const void* residual_k, int64_t rows, int D, int k,
                   void* anchor, void* residual, void* stream) {
  if (D != kD) return report_error(LYNX_EUNSUPPORTED, "only D = 128 is built");
  if (k < 3 || k > 6) return report_error(LYNX_EUNSUPPORTED, "k must be 3, 4, 5 or 6");
  if (rows < 0) return report_error(LYNX_ESHAPE, "rows must be >= 0");
  if (rows == 0) return LYNX_OK;
  if (!anchor || !residual || !anchor_k || !residual_k)
    return report_error(LYNX_EINVAL, "null pointer");
  if (!aligned(anchor, 16) || !aligned(residual, 16) || !aligned(anchor_k, 16) ||
      !aligned(residual_k, 16))
    return report_error(LYNX_EINVAL, "pointer not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t groups = rows * (kD / 8);
  const unsigned grid = grid_for(groups / 4, kThreads);
  const uint8_t* a = static_cast<const uint8_t*>(anchor_k);
  const uint8_t* r = static_cast<const uint8_t*>(residual_k);
  uint32_t* ao = static_cast<uint32_t*>(anchor);
  uint32_t* ro = static_cast<uint32_t*>(residual);
  if (k == 3) join_bits_kernel<3><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 4) join_bits_kernel<4><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 5) join_bits_kernel<5><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  if (k == 6) join_bits_kernel<6><<<grid, kThreads, 0, st>>>(a, r, groups, ao, ro);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_error(LYNX_ECUDA, cudaGetErrorString(e));
  return LYNX_OK;
}

}  // extern "C"
