// decode.cu -- the two decoders of "Lynx: Progressive Speculative KV Cache
// Transfer for Disaggregated LLM Inference" (technical review, Mechanism 2:
// Anchor Phase "Q_approx = dequant(Q_anc, gamma, mu, sigma)" and Residual
// Phase "Q_full = dequant(Q_anc + Q_res)"; Worked Example Eq. 14-15).
//
// One persistent kernel per (mode, output type).  A CTA walks units of up to
// 256 tokens: a whole page block, or one half of a 512-token page.  The
// unit's anchor codes, residual codes and metadata rows (contiguous in HBM;
// for a half page, the gamma rows and the mu and sigma rows of its chunks)
// arrive in shared memory by bulk asynchronous copies, one stage ahead of
// the unit being decoded.  Thread (slot, g) of 256 decodes a run of unit/16
// consecutive tokens (always inside one chunk) for channels 8g..8g+7, so it
// reads its chunk's constants once per unit.
//
// Reconstruction of one element (identical in both modes once v is known):
//   v = S * X(I), X(I) = ((1+alpha)^(I/127) - 1)/alpha rounded to float32,
//   n = fma(v, sigma + eps, mu),  x = fma(n, gamma_scale + eps, gamma_min).
// Full: Q8 = Anchor<<4 | Residual, S = sign(Q8), I = S>0 ? Q8 : -Q8-1.
// Anchor-only: a = signed Anchor, S = sign(a), V = S>0 ? a : -a-1, I = 16V+7.
//
// Lookup tables live in shared memory, one row per byte value, replicated so
// that every lane reads its own bank: full mode 256 rows of 256 bytes (32
// lanes x float per 8-bit code), anchor mode 256 rows of 128 bytes (16 lane
// slots x float2 per anchor byte, both channels of the byte in one load).  A lookup
// address is one byte permute, (byte << 8) | lane offset (halved in anchor
// mode), and the load adds the fixed shared-window base as its immediate
// offset.
#include "common.cuh"
#include "internal.h"

namespace lynx {

constexpr int kDecThreads = 256;
constexpr int kDecUnit = 256;   // most tokens of a decode unit
constexpr int kDecStages = 2;
constexpr int kDecLut = 65536;   // full mode: 256 rows of 256 bytes
constexpr int kDecLutAnchor = 32768;   // anchor mode: 256 rows of 128 bytes
template <bool FULL> constexpr int dec_lut_bytes() { return FULL ? kDecLut : kDecLutAnchor; }
// Shared-window address of the first byte of dynamic shared memory for a
// kernel without static shared memory (the block's reserved shared memory
// comes first); checked by the host before launch and by the kernel.
constexpr uint32_t kDecSmemBase = 1024;

// Set by a decoder whose bounded wait on a stage gave up (the kernel then
// returns early).  Read through read_decode_wait_timeout(); never reset.
__device__ unsigned int g_dec_wait_timeout = 0;

cudaError_t read_decode_wait_timeout(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_dec_wait_timeout, sizeof(unsigned int));
}

__device__ __forceinline__ uint32_t dec_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Table offset of byte POS of w: [lane_off, w.b_POS, 0, 0].
template <int POS>
__device__ __forceinline__ uint32_t dec_lut_off(uint32_t w, uint32_t lane_off) {
  return dec_prmt(w, lane_off, 0x7604u | ((uint32_t)POS << 4));
}
// Table reads; the table is written once before the first barrier.
__device__ __forceinline__ float dec_lut_f1(uint32_t off) {
  float v;
  asm("ld.shared.f32 %0, [%1+1024];" : "=f"(v) : "r"(off));
  return v;
}
__device__ __forceinline__ float2 dec_lut_f2(uint32_t off) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2+1024];" : "=f"(v.x), "=f"(v.y) : "r"(off));
  return v;
}
static_assert(kDecSmemBase == 1024, "immediate offset of the table loads");

template <bool BF16OUT>
__device__ __forceinline__ void store8(void* out, int64_t off, const float (&x)[8]) {
  char* o = reinterpret_cast<char*>(out);
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

template <bool FULL, bool BF16OUT>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(const uint8_t* __restrict__ anchor, const uint8_t* __restrict__ residual,
              const float* __restrict__ meta, const int64_t nblk, const int64_t NB,
              const int H, const int64_t L, const int P, const int C,
              void* __restrict__ out, const int32_t* __restrict__ bt, const int64_t nphys,
              const __grid_constant__ ExpandTable tab) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid & 15, slot = tid >> 4;
  const int U = P < kDecUnit ? P : kDecUnit;   // tokens of a unit
  const int parts = P / U;                     // units of a page block
  const int64_t nunit = nblk * parts;
  const int NC = U / C;                        // chunks of a unit
  const int blk_meta_rows = 2 + 2 * (P / C);
  const uint32_t code_bytes = (uint32_t)U * (kD / 2);          // one stream of a unit
  const uint32_t meta_bytes = (uint32_t)(2 + 2 * NC) * kD * 4;
  const uint32_t stage_bytes = code_bytes * (FULL ? 2 : 1) + meta_bytes;
  uint8_t* stages = smem + dec_lut_bytes<FULL>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + kDecStages * stage_bytes);
  const int run = U >> 4;                 // tokens per thread per unit (4, 8 or 16)
  const int t0 = slot * run;
  const int chunk = t0 / C;
  const int64_t ostride = (int64_t)H * kD;

  if (smem_u32(smem) != kDecSmemBase) {   // table loads would read the wrong bytes
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __int_as_float(0x7fc00000);
    for (int64_t un = blockIdx.x; un < nunit; un += gridDim.x) {
      const int64_t blk = un / parts, part = un % parts;
      const int64_t h = blk % H, rest = blk / H;
      const int64_t p = rest % NB, b = rest / NB;
      for (int r = 0; r < run; ++r)
        store8<BF16OUT>(out, ((b * L + p * P + part * U + t0 + r) * H + h) * kD + 8 * g, x);
    }
    return;
  }

  // ---- tables
  for (int i = tid; i < 256 * 32; i += kDecThreads) {
    const int row = i >> 5, l = i & 31;
    if constexpr (FULL) {
      reinterpret_cast<float*>(smem + row * 256)[l] = row < 128 ? tab.x[row] : -tab.x[255 - row];
    } else if (l < 16) {
      const int a0 = row & 15, a1 = row >> 4;
      reinterpret_cast<float2*>(smem + row * 128)[l] =
          make_float2(a0 < 8 ? tab.x[16 * a0 + 7] : -tab.x[16 * (15 - a0) + 7],
                      a1 < 8 ? tab.x[16 * a1 + 7] : -tab.x[16 * (15 - a1) + 7]);
    }
  }
  if (tid == 0) {
    for (int i = 0; i < kDecStages; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // anchor mode: the permute gives (byte << 8) | 16 slot, halved at the load
  const uint32_t lane_off = FULL ? (uint32_t)lane * 4u : (uint32_t)(lane & 15) * 16u;

  auto issue = [&](int64_t un, int stage) {
    const int64_t part = un % parts;
    const int64_t blk = checked_index(phys_block(bt, nphys, un / parts, H, &g_dec_wait_timeout),
                                      bt ? nphys * H : nblk, &g_dec_wait_timeout);
    uint8_t* st = stages + stage * stage_bytes;
    const int64_t code_off = (blk * parts + part) * code_bytes;
    mbar_expect_tx(&bars[stage], stage_bytes);
    bulk_load(st, anchor + code_off, code_bytes, &bars[stage]);
    if constexpr (FULL) bulk_load(st + code_bytes, residual + code_off, code_bytes, &bars[stage]);
    uint8_t* sm = st + code_bytes * (FULL ? 2 : 1);
    const float* mb = meta + blk * (int64_t)blk_meta_rows * kD;
    if (parts == 1) {
      bulk_load(sm, mb, meta_bytes, &bars[stage]);
    } else {  // gamma rows, then the unit's mu rows and sigma rows
      const uint32_t rows = (uint32_t)NC * kD * 4;
      bulk_load(sm, mb, 2 * kD * 4, &bars[stage]);
      bulk_load(sm + 2 * kD * 4, mb + (2 + part * NC) * kD, rows, &bars[stage]);
      bulk_load(sm + 2 * kD * 4 + rows, mb + (2 + P / C + part * NC) * kD, rows, &bars[stage]);
    }
  };
  if (tid == 0)
    for (int i = 0; i < kDecStages; ++i) {
      const int64_t un = blockIdx.x + (int64_t)i * gridDim.x;
      if (un < nunit) issue(un, i);
    }

  int it = 0;
  for (int64_t un = blockIdx.x; un < nunit; un += gridDim.x, ++it) {
    const int stage = it % kDecStages;
    const uint32_t phase = (uint32_t)(it / kDecStages) & 1u;
    const bool ok = mbar_wait(&bars[stage], phase);
    const uint8_t* st = stages + stage * stage_bytes;
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(st) + t0 * 16 + g;
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(st + code_bytes) + t0 * 16 + g;
    const float* mrow = reinterpret_cast<const float*>(st + code_bytes * (FULL ? 2 : 1)) + 8 * g;
    const float4 gm_a = *reinterpret_cast<const float4*>(mrow);
    const float4 gm_b = *reinterpret_cast<const float4*>(mrow + 4);
    const float4 gs_a = *reinterpret_cast<const float4*>(mrow + kD);
    const float4 gs_b = *reinterpret_cast<const float4*>(mrow + kD + 4);
    const float4 mu_a = *reinterpret_cast<const float4*>(mrow + (2 + chunk) * kD);
    const float4 mu_b = *reinterpret_cast<const float4*>(mrow + (2 + chunk) * kD + 4);
    const float4 sg_a = *reinterpret_cast<const float4*>(mrow + (2 + NC + chunk) * kD);
    const float4 sg_b = *reinterpret_cast<const float4*>(mrow + (2 + NC + chunk) * kD + 4);
    const int64_t blk = un / parts, part = un % parts;
    const int64_t h = blk % H, rest = blk / H;
    const int64_t p = rest % NB, b = rest / NB;
    const int64_t row0 = checked_index(b * L + p * P + part * U + t0, nblk / H * P - run + 1,
                                       &g_dec_wait_timeout);
    const int64_t orow0 = (row0 * H + h) * kD + 8 * g;

    if constexpr (FULL) {
      // pairs (k, k+1) in channel order
      const f2 e2 = make_float2(kEps, kEps);
      const f2 gm[4] = {make_float2(gm_a.x, gm_a.y), make_float2(gm_a.z, gm_a.w),
                        make_float2(gm_b.x, gm_b.y), make_float2(gm_b.z, gm_b.w)};
      const f2 gs[4] = {add2(make_float2(gs_a.x, gs_a.y), e2), add2(make_float2(gs_a.z, gs_a.w), e2),
                        add2(make_float2(gs_b.x, gs_b.y), e2), add2(make_float2(gs_b.z, gs_b.w), e2)};
      const f2 mu[4] = {make_float2(mu_a.x, mu_a.y), make_float2(mu_a.z, mu_a.w),
                        make_float2(mu_b.x, mu_b.y), make_float2(mu_b.z, mu_b.w)};
      const f2 sg[4] = {add2(make_float2(sg_a.x, sg_a.y), e2), add2(make_float2(sg_a.z, sg_a.w), e2),
                        add2(make_float2(sg_b.x, sg_b.y), e2), add2(make_float2(sg_b.z, sg_b.w), e2)};
#pragma unroll 4
      for (int r = 0; r < run; ++r) {
        const uint32_t a = aw[r * 16], rr = rw[r * 16];
        const uint32_t E = ((a << 4) & 0xf0f0f0f0u) | (rr & 0x0f0f0f0fu);  // codes of ch 0-3
        const uint32_t O = (a & 0xf0f0f0f0u) | ((rr >> 4) & 0x0f0f0f0fu);  // codes of ch 4-7
        f2 v[4];
        v[0] = make_float2(dec_lut_f1(dec_lut_off<0>(E, lane_off)), dec_lut_f1(dec_lut_off<1>(E, lane_off)));
        v[1] = make_float2(dec_lut_f1(dec_lut_off<2>(E, lane_off)), dec_lut_f1(dec_lut_off<3>(E, lane_off)));
        v[2] = make_float2(dec_lut_f1(dec_lut_off<0>(O, lane_off)), dec_lut_f1(dec_lut_off<1>(O, lane_off)));
        v[3] = make_float2(dec_lut_f1(dec_lut_off<2>(O, lane_off)), dec_lut_f1(dec_lut_off<3>(O, lane_off)));
        float x[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const f2 y = fma2(fma2(v[k], sg[k], mu[k]), gs[k], gm[k]);
          x[2 * k] = y.x;
          x[2 * k + 1] = y.y;
        }
        store8<BF16OUT>(out, orow0 + (int64_t)r * ostride, x);
      }
    } else {
      const float gm[8] = {gm_a.x, gm_a.y, gm_a.z, gm_a.w, gm_b.x, gm_b.y, gm_b.z, gm_b.w};
      const float gsr[8] = {gs_a.x, gs_a.y, gs_a.z, gs_a.w, gs_b.x, gs_b.y, gs_b.z, gs_b.w};
      const float mu[8] = {mu_a.x, mu_a.y, mu_a.z, mu_a.w, mu_b.x, mu_b.y, mu_b.z, mu_b.w};
      const float sgr[8] = {sg_a.x, sg_a.y, sg_a.z, sg_a.w, sg_b.x, sg_b.y, sg_b.z, sg_b.w};
      float gs[8], sg[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gs[i] = __fadd_rn(gsr[i], kEps);
        sg[i] = __fadd_rn(sgr[i], kEps);
      }
#pragma unroll 4
      for (int r = 0; r < run; ++r) {
        const uint32_t a = aw[r * 16];
        float v[8];  // channel order 0..7 of the group
        {
          const float2 p0 = dec_lut_f2(dec_lut_off<0>(a, lane_off) >> 1);
          const float2 p1 = dec_lut_f2(dec_lut_off<1>(a, lane_off) >> 1);
          const float2 p2 = dec_lut_f2(dec_lut_off<2>(a, lane_off) >> 1);
          const float2 p3 = dec_lut_f2(dec_lut_off<3>(a, lane_off) >> 1);
          v[0] = p0.x; v[4] = p0.y; v[1] = p1.x; v[5] = p1.y;
          v[2] = p2.x; v[6] = p2.y; v[3] = p3.x; v[7] = p3.y;
        }
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = fmaf(fmaf(v[i], sg[i], mu[i]), gs[i], gm[i]);
        store8<BF16OUT>(out, orow0 + (int64_t)r * ostride, x);
      }
    }

    if (!__syncthreads_and(ok)) {
      // A stage never arrived: record it and stop this CTA (bounded waits
      // only, so the context stays usable).
      if (tid == 0) {
        atomicOr(&g_dec_wait_timeout, kFlagWaitTimeout);
        for (int i = 0; i < kDecStages; ++i) (void)mbar_wait(&bars[i], phase);
      }
      return;
    }
    // every thread is done with this stage: refill it kDecStages units ahead
    if (tid == 0) {
      const int64_t nxt = un + (int64_t)kDecStages * gridDim.x;
      if (nxt < nunit) {
        fence_proxy_async();
        issue(nxt, stage);
      }
    }
  }
}

template <bool FULL, bool BF16OUT>
static cudaError_t run_decode(const void* anchor, const void* residual, const float* meta,
                              const Shape& s, const ExpandTable& tab, void* out,
                              cudaStream_t stream, const Paging& pg) {
  auto fn = decode_kernel<FULL, BF16OUT>;
  const int U = s.page < kDecUnit ? s.page : kDecUnit;
  const size_t stage = (size_t)U * (kD / 2) * (FULL ? 2 : 1) + (size_t)(2 + 2 * (U / s.C)) * kD * 4;
  const size_t smem = dec_lut_bytes<FULL>() + kDecStages * stage + kDecStages * 8;
  constexpr size_t kMaxSmem = kDecLut + kDecStages * (256 * 64 * 2 + 34 * kD * 4) + 64;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    int reserved = -1;
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    if (reserved != (int)kDecSmemBase) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  static thread_local size_t last_smem = 0;
  static thread_local int per_sm = 1;
  if (smem != last_smem) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
    last_smem = smem;
  }
  const int64_t nblk = s.blocks();
  int64_t grid = (int64_t)sm_count() * per_sm;
  if (grid > nblk * (s.page / U)) grid = nblk * (s.page / U);
  fn<<<(unsigned)grid, kDecThreads, smem, stream>>>(
      static_cast<const uint8_t*>(anchor), static_cast<const uint8_t*>(residual), meta, nblk,
      s.NB(), s.H, s.L, s.page, s.C, out, pg.table, pg.nphys, tab);
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* anchor, const void* residual, const float* meta,
                          const Shape& s, const ExpandTable& tab, void* out, bool bf16_out,
                          cudaStream_t stream, const Paging& pg) {
  if (s.blocks() == 0) return cudaSuccess;
  const bool full = residual != nullptr;
  if (full)
    return bf16_out ? run_decode<true, true>(anchor, residual, meta, s, tab, out, stream, pg)
                    : run_decode<true, false>(anchor, residual, meta, s, tab, out, stream, pg);
  return bf16_out ? run_decode<false, true>(anchor, nullptr, meta, s, tab, out, stream, pg)
                  : run_decode<false, false>(anchor, nullptr, meta, s, tab, out, stream, pg);
}

}  // namespace lynx
