// decode.cu -- the two decoders of "Lynx: Progressive Speculative KV Cache
// Transfer for Disaggregated LLM Inference" (technical review, Mechanism 2:
// Anchor Phase "Q_approx = dequant(Q_anc, gamma, mu, sigma)" and Residual
// Phase "Q_full = dequant(Q_anc + Q_res)"; Worked Example Eq. 14-15).
//
// One persistent kernel per (mode, output type).  A CTA walks page blocks;
// thread (slot, g) of 256 decodes a run of page/16 consecutive tokens of the
// block (always inside one chunk) for channels 8g..8g+7, so each thread loads
// its chunk's mu, sigma and the page's gamma once per block.
//
// Reconstruction of one element (identical in both modes once v is known):
//   v = S * X(I), X(I) = ((1+alpha)^(I/127) - 1)/alpha rounded to float32,
//   n = fma(v, sigma + eps, mu),  x = fma(n, gamma_scale + eps, gamma_min).
// Full: Q8 = Anchor<<4 | Residual, S = sign(Q8), I = S>0 ? Q8 : -Q8-1.
// Anchor-only: a = signed Anchor, S = sign(a), V = S>0 ? a : -a-1, I = 16V+7.
//
// Lookup tables live in shared memory, replicated so that every lane reads
// its own bank: full mode a 256-entry signed table per lane (32 KB); anchor
// mode a 256-entry table over the anchor BYTE (two channels) per half-warp
// lane (32 KB), giving both values of the byte with one 8-byte load.
#include "common.cuh"
#include "internal.h"

namespace lynx {

constexpr int kDecThreads = 256;

template <bool FULL, bool BF16OUT>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(const uint32_t* __restrict__ anchor, const uint32_t* __restrict__ residual,
              const float* __restrict__ meta, const int64_t nblk, const int64_t NB,
              const int H, const int64_t L, const int P, const int C,
              void* __restrict__ out, const __grid_constant__ ExpandTable tab) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid & 15, slot = tid >> 4;

  // ---- tables
  if constexpr (FULL) {
    float* lut = reinterpret_cast<float*>(smem);          // [256][32]
    for (int i = tid; i < 256 * 32; i += kDecThreads) {
      const int code = i >> 5;
      lut[i] = code < 128 ? tab.x[code] : -tab.x[255 - code];
    }
  } else {
    float2* lut = reinterpret_cast<float2*>(smem);        // [256][16]
    for (int i = tid; i < 256 * 16; i += kDecThreads) {
      const int byte = i >> 4;
      const int a0 = byte & 15, a1 = byte >> 4;
      const float v0 = a0 < 8 ? tab.x[16 * a0 + 7] : -tab.x[16 * (15 - a0) + 7];
      const float v1 = a1 < 8 ? tab.x[16 * a1 + 7] : -tab.x[16 * (15 - a1) + 7];
      lut[i] = make_float2(v0, v1);
    }
  }
  __syncthreads();

  const int run = P >> 4;                 // tokens per thread per block (4, 8 or 16)
  const int NC = P / C;
  const int meta_rows = 2 + 2 * NC;
  const int t0 = slot * run;
  const int chunk = t0 / C;

  // Software pipeline over the CTA's blocks: the codes and metadata of the
  // next block are loaded before the current block is decoded, so every
  // thread keeps 8 code words (+ 8 residual words) and 8 metadata vectors in
  // flight while it computes.
  struct Loads {
    uint32_t a[8], r[8];
    float4 m[8];
  };
  auto load = [&](int64_t blk, int r0, Loads& ld) {
    const uint32_t* arow = anchor + (blk * P + t0 + r0) * 16 + g;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      ld.a[r] = ldg_stream32(arow + r * 16);
      if constexpr (FULL) ld.r[r] = ldg_stream32(residual + (blk * P + t0 + r0 + r) * 16 + g);
    }
    const float* mrow = meta + blk * (int64_t)meta_rows * kD + 8 * g;
    const float4* q0 = reinterpret_cast<const float4*>(mrow);
    const float4* q1 = reinterpret_cast<const float4*>(mrow + kD);
    const float4* q2 = reinterpret_cast<const float4*>(mrow + (2 + chunk) * kD);
    const float4* q3 = reinterpret_cast<const float4*>(mrow + (2 + NC + chunk) * kD);
    ld.m[0] = __ldg(q0); ld.m[1] = __ldg(q0 + 1);
    ld.m[2] = __ldg(q1); ld.m[3] = __ldg(q1 + 1);
    ld.m[4] = __ldg(q2); ld.m[5] = __ldg(q2 + 1);
    ld.m[6] = __ldg(q3); ld.m[7] = __ldg(q3 + 1);
  };

  auto decode8 = [&](int64_t blk, int r0, const Loads& ld) {
    const int64_t h = blk % H, rest = blk / H;
    const int64_t p = rest % NB, b = rest / NB;
    float gm[8], gsc[8], mu[8], sgc[8];
    const float* mv = reinterpret_cast<const float*>(ld.m);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      gm[i] = mv[i];
      gsc[i] = __fadd_rn(mv[8 + i], kEps);
      mu[i] = mv[16 + i];
      sgc[i] = __fadd_rn(mv[24 + i], kEps);
    }
    const int64_t orow0 = ((b * L + p * P + t0 + r0) * H + h) * kD + 8 * g;
    const int64_t ostride = (int64_t)H * kD;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v[8];  // channel order 0..7 of the group
      if constexpr (FULL) {
        const float* lut = reinterpret_cast<const float*>(smem);
        const uint32_t E = ((ld.a[r] << 4) & 0xf0f0f0f0u) | (ld.r[r] & 0x0f0f0f0fu);  // ch 0-3
        const uint32_t O = (ld.a[r] & 0xf0f0f0f0u) | ((ld.r[r] >> 4) & 0x0f0f0f0fu);  // ch 4-7
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[k] = lut[((E >> (8 * k)) & 0xffu) * 32 + lane];
          v[k + 4] = lut[((O >> (8 * k)) & 0xffu) * 32 + lane];
        }
      } else {
        const float2* lut = reinterpret_cast<const float2*>(smem);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 pv = lut[((ld.a[r] >> (8 * k)) & 0xffu) * 16 + (lane & 15)];
          v[k] = pv.x;
          v[k + 4] = pv.y;
        }
      }
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = fmaf(fmaf(v[i], sgc[i], mu[i]), gsc[i], gm[i]);
      char* o = reinterpret_cast<char*>(out);
      const int64_t off = orow0 + (int64_t)r * ostride;
      if constexpr (BF16OUT) {
        uint4 pkd;
        pkd.x = f2_to_bf2(x[0], x[1]);
        pkd.y = f2_to_bf2(x[2], x[3]);
        pkd.z = f2_to_bf2(x[4], x[5]);
        pkd.w = f2_to_bf2(x[6], x[7]);
        stg_stream(o + off * 2, pkd);
      } else {
        stg_stream(o + off * 4, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                           __float_as_uint(x[2]), __float_as_uint(x[3])));
        stg_stream(o + off * 4 + 16, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                                                __float_as_uint(x[6]), __float_as_uint(x[7])));
      }
    }
  };

  // Work items: (block, 8-token part of the thread's run).  run/8 parts per
  // block when run >= 8; for run == 4 (page 64) two threads' worth of rows
  // are not needed, so half-runs are handled by the tail path below.
  if (run >= 8) {
    const int parts = run / 8;
    const int64_t items = ((nblk - blockIdx.x + gridDim.x - 1) / gridDim.x) * parts;
    Loads cur, nxt;
    if (items > 0) load(blockIdx.x, 0, cur);
    for (int64_t it = 0; it < items; ++it) {
      const int64_t blk = blockIdx.x + (it / parts) * gridDim.x;
      const int r0 = (int)(it % parts) * 8;
      if (it + 1 < items)
        load(blockIdx.x + ((it + 1) / parts) * gridDim.x, (int)((it + 1) % parts) * 8, nxt);
      decode8(blk, r0, cur);
      cur = nxt;
    }
  } else {
    // page 64: 4 tokens per thread; loads of rows 4..7 would leave the run,
    // so this simple path loads and decodes 4 rows per block.
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
      const int64_t h = blk % H, rest = blk / H;
      const int64_t p = rest % NB, b = rest / NB;
      const float* mrow = meta + blk * (int64_t)meta_rows * kD + 8 * g;
      float gm[8], gsc[8], mu[8], sgc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gm[i] = __ldg(mrow + i);
        gsc[i] = __fadd_rn(__ldg(mrow + kD + i), kEps);
        mu[i] = __ldg(mrow + (2 + chunk) * kD + i);
        sgc[i] = __fadd_rn(__ldg(mrow + (2 + NC + chunk) * kD + i), kEps);
      }
      const uint32_t* arow = anchor + (blk * P + t0) * 16 + g;
      const uint32_t* rrow = FULL ? residual + (blk * P + t0) * 16 + g : nullptr;
      uint32_t aw[4], rw[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        aw[r] = ldg_stream32(arow + r * 16);
        if constexpr (FULL) rw[r] = ldg_stream32(rrow + r * 16);
      }
      const int64_t orow0 = ((b * L + p * P + t0) * H + h) * kD + 8 * g;
      const int64_t ostride = (int64_t)H * kD;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float v[8];
        if constexpr (FULL) {
          const float* lut = reinterpret_cast<const float*>(smem);
          const uint32_t E = ((aw[r] << 4) & 0xf0f0f0f0u) | (rw[r] & 0x0f0f0f0fu);
          const uint32_t O = (aw[r] & 0xf0f0f0f0u) | ((rw[r] >> 4) & 0x0f0f0f0fu);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[k] = lut[((E >> (8 * k)) & 0xffu) * 32 + lane];
            v[k + 4] = lut[((O >> (8 * k)) & 0xffu) * 32 + lane];
          }
        } else {
          const float2* lut = reinterpret_cast<const float2*>(smem);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 pv = lut[((aw[r] >> (8 * k)) & 0xffu) * 16 + (lane & 15)];
            v[k] = pv.x;
            v[k + 4] = pv.y;
          }
        }
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = fmaf(fmaf(v[i], sgc[i], mu[i]), gsc[i], gm[i]);
        char* o = reinterpret_cast<char*>(out);
        const int64_t off = orow0 + (int64_t)r * ostride;
        if constexpr (BF16OUT) {
          uint4 pkd;
          pkd.x = f2_to_bf2(x[0], x[1]);
          pkd.y = f2_to_bf2(x[2], x[3]);
          pkd.z = f2_to_bf2(x[4], x[5]);
          pkd.w = f2_to_bf2(x[6], x[7]);
          stg_stream(o + off * 2, pkd);
        } else {
          stg_stream(o + off * 4, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                             __float_as_uint(x[2]), __float_as_uint(x[3])));
          stg_stream(o + off * 4 + 16, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                                                  __float_as_uint(x[6]), __float_as_uint(x[7])));
        }
      }
    }
  }
}

template <bool FULL, bool BF16OUT>
static cudaError_t run_decode(const void* anchor, const void* residual, const float* meta,
                              const Shape& s, const ExpandTable& tab, void* out,
                              cudaStream_t stream) {
  auto fn = decode_kernel<FULL, BF16OUT>;
  constexpr size_t smem = 32768;
  static thread_local int configured_dev = -1;
  static thread_local int per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
    configured_dev = dev;
  }
  const int64_t nblk = s.blocks();
  int64_t grid = (int64_t)sm_count() * per_sm;
  if (grid > nblk) grid = nblk;
  fn<<<(unsigned)grid, kDecThreads, smem, stream>>>(
      static_cast<const uint32_t*>(anchor), static_cast<const uint32_t*>(residual), meta, nblk,
      s.NB(), s.H, s.L, s.page, s.C, out, tab);
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* anchor, const void* residual, const float* meta,
                          const Shape& s, const ExpandTable& tab, void* out, bool bf16_out,
                          cudaStream_t stream) {
  if (s.blocks() == 0) return cudaSuccess;
  const bool full = residual != nullptr;
  if (full)
    return bf16_out ? run_decode<true, true>(anchor, residual, meta, s, tab, out, stream)
                    : run_decode<true, false>(anchor, residual, meta, s, tab, out, stream);
  return bf16_out ? run_decode<false, true>(anchor, nullptr, meta, s, tab, out, stream)
                  : run_decode<false, false>(anchor, nullptr, meta, s, tab, out, stream);
}

}  // namespace lynx
