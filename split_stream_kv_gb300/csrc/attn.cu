// attn.cu -- decode attention O = softmax(q K^T / sqrt(d)) V ("Lynx:
// Progressive Speculative KV Cache Transfer for Disaggregated LLM Inference",
// Prerequisites Eq. 1) read straight from the packed Lynx streams: the draft
// step over Anchor codes (Mechanism 2, Anchor Phase) and the T-token
// verification pass over Anchor + Residual (Mechanism 3).
//
// K and V are reconstructed in registers exactly as the decoders do with BF16
// output (same lookup values, same two fused multiply-adds, round to nearest
// even), then fed to mma.sync m16n8k16 (bf16 x bf16 -> f32):
//   scores  S^T[token][row] = K^[token][:] . q[row][:]     (A = K^, B = Q^T)
//   output  O^T[ch][row]   += V^[:][ch]^T . P^T[:][row]    (A = V^T, B = P^T)
// A query "row" is one (query token, query head of the group): up to 8 rows
// per pass; more rows run as further row groups (grid z).
// The contraction index (channel) of the scores is permuted so that a lane's
// fragment bytes are contiguous in a packed row: lane c (= lane % 4) owns the
// 16 bytes 16c..16c+15 (channels 32c..32c+31) for K; for V, lane g (= lane/4)
// owns the 8 bytes 8g..8g+7 (channels 16g..16g+15) and m-tile mt takes byte
// 8g+mt, whose two channels are the rows g and g+8 of that m-tile.
// P is split into bf16 hi + lo parts (two MMAs) so the softmax weights keep
// about 16 mantissa bits; movmatrix turns the S^T accumulator layout into the
// P^T operand layout.
//
// Work split (flash-decoding): grid = (splits, H_kv, batch * row groups).
// Each warp walks its own 32-token chunks of the CTA's token range with its
// own running max / sum / output; the CTA merges its 4 warps and writes one
// partial (m, l, o) per split; attn_combine merges the splits.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "lynx.h"

namespace lynx {

constexpr int kAttnWarps = 4;
constexpr int kRows = 8;                 // query rows per pass (one n-tile)
constexpr int kPartFloats = 2 * kRows + kRows * kD;
constexpr int kScratchFloats = 2 * 6 * kD;  // per warp: K and V constant rows

struct AttnParams {
  const uint16_t* q;
  const uint8_t *ka, *kr, *va, *vr;
  const float *km, *vm;
  float* part;
  float* out;
  int batch, T, Hq, Hkv, G, R, nrg, S;
  int64_t L, NB, NCH;
  int P, C, NC;
  float scale_log2;
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint4 ldg128(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg64(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Values of the two channels of one packed byte position (anchor byte a and,
// in full mode, residual byte r): (low-nibble channel, high-nibble channel).
template <bool FULL>
__device__ __forceinline__ float2 lookup_pair(const uint8_t* lut, uint32_t a, uint32_t r,
                                              int lane) {
  if constexpr (FULL) {
    const float* t = reinterpret_cast<const float*>(lut);
    const uint32_t c_lo = ((a & 0x0fu) << 4) | (r & 0x0fu);
    const uint32_t c_hi = (a & 0xf0u) | (r >> 4);
    return make_float2(t[c_lo * 32 + lane], t[c_hi * 32 + lane]);
  } else {
    const float2* t = reinterpret_cast<const float2*>(lut);
    return t[a * 16 + (lane & 15)];
  }
}

// One packed byte position -> bf16x2 (low-nibble channel in the low half).
template <bool FULL>
__device__ __forceinline__ uint32_t dequant_pair(const uint8_t* lut, uint32_t a, uint32_t r,
                                                 int lane, float gm0, float gm1, float gs0,
                                                 float gs1, float mu0, float mu1, float sg0,
                                                 float sg1) {
  const float2 v = lookup_pair<FULL>(lut, a, r, lane);
  const float x0 = fmaf(fmaf(v.x, sg0, mu0), gs0, gm0);
  const float x1 = fmaf(fmaf(v.y, sg1, mu1), gs1, gm1);
  return f2_to_bf2(x0, x1);
}

template <bool FULL>
__global__ void __launch_bounds__(kAttnWarps * 32, 3)
attn_kernel(const __grid_constant__ AttnParams a, const __grid_constant__ ExpandTable tab) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* lut = smem;                                   // 32 KB
  float* scratch_all = reinterpret_cast<float*>(smem + 32768);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;

  if constexpr (FULL) {
    float* t = reinterpret_cast<float*>(lut);
    for (int i = tid; i < 256 * 32; i += kAttnWarps * 32) {
      const int code = i >> 5;
      t[i] = code < 128 ? tab.x[code] : -tab.x[255 - code];
    }
  } else {
    float2* t = reinterpret_cast<float2*>(lut);
    for (int i = tid; i < 256 * 16; i += kAttnWarps * 32) {
      const int byte = i >> 4, a0 = byte & 15, a1 = byte >> 4;
      t[i] = make_float2(a0 < 8 ? tab.x[16 * a0 + 7] : -tab.x[16 * (15 - a0) + 7],
                         a1 < 8 ? tab.x[16 * a1 + 7] : -tab.x[16 * (15 - a1) + 7]);
    }
  }
  __syncthreads();

  const int split = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / a.nrg, rg = blockIdx.z % a.nrg;
  const int row0 = rg * kRows;

  // ---- Q^T fragments (B operand), channel order matching the K bytes
  uint32_t qf[8][2];
  {
    const int r = row0 + g;
    const bool valid = r < a.R;
    const int tq = valid ? r / a.G : 0, gq = valid ? r % a.G : 0;
    const uint16_t* qrow = a.q + ((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD;
#pragma unroll
    for (int kt = 0; kt < 8; ++kt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int beta = 16 * c + 2 * kt + hh;
        const int lo = 8 * (beta >> 2) + (beta & 3);
        qf[kt][hh] = valid ? ((uint32_t)qrow[lo] | ((uint32_t)qrow[lo + 4] << 16)) : 0u;
      }
  }

  float* scr = scratch_all + w * kScratchFloats;   // [tensor][6][128]
  const int64_t cb = a.NCH * split / a.S, ce = a.NCH * (split + 1) / a.S;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const int meta_rows = 2 + 2 * a.NC;

  for (int64_t qc = cb + w; qc < ce; qc += kAttnWarps) {
    const int64_t t0 = qc * 32;
    const int64_t p = t0 / a.P;
    const int tp = (int)(t0 - p * a.P);
    const int64_t blk = ((int64_t)b * a.NB + p) * a.Hkv + h;
    const int64_t code_off = (blk * a.P + tp) * (kD / 2);

    // ---- packed codes of this chunk
    uint4 kA[4], kR[4];
    uint2 vA[8], vR[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int row = 16 * (jj >> 1) + g + 8 * (jj & 1);
      kA[jj] = ldg128(a.ka + code_off + row * 64 + 16 * c);
      if constexpr (FULL) kR[jj] = ldg128(a.kr + code_off + row * 64 + 16 * c);
    }
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int kk = ii & 3;
      const int row = 16 * (ii >> 2) + 2 * c + (kk & 1) + 8 * (kk >> 1);
      vA[ii] = ldg64(a.va + code_off + row * 64 + 8 * g);
      if constexpr (FULL) vR[ii] = ldg64(a.vr + code_off + row * 64 + 8 * g);
    }
    // ---- constants: gamma_min, gamma_scale+eps, mu (2 sub-tiles), sigma+eps
    {
      const int cc0 = tp / a.C, cc1 = (tp + 16) / a.C;
      const int src_row[6] = {0, 1, 2 + cc0, 2 + cc1, 2 + a.NC + cc0, 2 + a.NC + cc1};
#pragma unroll
      for (int tsr = 0; tsr < 2; ++tsr) {
        const float* mb = (tsr == 0 ? a.km : a.vm) + blk * (int64_t)meta_rows * kD;
#pragma unroll
        for (int rr = 0; rr < 6; ++rr) {
          float4 v = __ldg(reinterpret_cast<const float4*>(mb + src_row[rr] * kD) + lane);
          if (rr == 1 || rr >= 4) {
            v.x = __fadd_rn(v.x, kEps); v.y = __fadd_rn(v.y, kEps);
            v.z = __fadd_rn(v.z, kEps); v.w = __fadd_rn(v.w, kEps);
          }
          reinterpret_cast<float4*>(scr + (tsr * 6 + rr) * kD)[lane] = v;
        }
      }
    }
    __syncwarp();

    // ---- scores: S^T for m-tiles j = 0, 1 (tokens 16j .. 16j+15)
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      const int grp = 4 * c + G4;  // channels 8grp .. 8grp+7
      float gm[8], gs[8], mu[2][8], sg[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float4 x0 = reinterpret_cast<const float4*>(scr + 0 * kD + 8 * grp)[i];
        const float4 x1 = reinterpret_cast<const float4*>(scr + 1 * kD + 8 * grp)[i];
        gm[4 * i] = x0.x; gm[4 * i + 1] = x0.y; gm[4 * i + 2] = x0.z; gm[4 * i + 3] = x0.w;
        gs[4 * i] = x1.x; gs[4 * i + 1] = x1.y; gs[4 * i + 2] = x1.z; gs[4 * i + 3] = x1.w;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float4 y0 = reinterpret_cast<const float4*>(scr + (2 + j) * kD + 8 * grp)[i];
          const float4 y1 = reinterpret_cast<const float4*>(scr + (4 + j) * kD + 8 * grp)[i];
          mu[j][4 * i] = y0.x; mu[j][4 * i + 1] = y0.y; mu[j][4 * i + 2] = y0.z; mu[j][4 * i + 3] = y0.w;
          sg[j][4 * i] = y1.x; sg[j][4 * i + 1] = y1.y; sg[j][4 * i + 2] = y1.z; sg[j][4 * i + 3] = y1.w;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int kt = 2 * G4 + kk;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t af[4];
#pragma unroll
          for (int i = 0; i < 2; ++i) {       // row g (i=0) / g+8 (i=1)
            const uint32_t wa = word_of(kA[2 * j + i], G4);
            const uint32_t wr = FULL ? word_of(kR[2 * j + i], G4) : 0u;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // k 2c..2c+1 (hh=0) / 2c+8.. (hh=1)
              const int jb = 2 * kk + hh;     // byte within the word = channel 8grp+jb
              const uint32_t ab = (wa >> (8 * jb)) & 0xffu;
              const uint32_t rb = (wr >> (8 * jb)) & 0xffu;
              af[i + 2 * hh] = dequant_pair<FULL>(lut, ab, rb, lane, gm[jb], gm[jb + 4], gs[jb],
                                                  gs[jb + 4], mu[j][jb], mu[j][jb + 4],
                                                  sg[j][jb], sg[j][jb + 4]);
            }
          }
          mma_bf16(s[j], af, qf[kt][0], qf[kt][1]);
        }
      }
    }

    // ---- online softmax (log2 domain); rows 2c, 2c+1
    float cmax0 = fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2]));
    float cmax1 = fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]));
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      cmax0 = fmaxf(cmax0, __shfl_xor_sync(kFull, cmax0, x));
      cmax1 = fmaxf(cmax1, __shfl_xor_sync(kFull, cmax1, x));
    }
    const float mn0 = fmaxf(m_run[0], cmax0 * a.scale_log2);
    const float mn1 = fmaxf(m_run[1], cmax1 * a.scale_log2);
    const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    l_run[0] *= al0;
    l_run[1] *= al1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
    }
    uint32_t pb_hi[2][2], pb_lo[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float p0 = exp2f(fmaf(s[j][0], a.scale_log2, -mn0));
      const float p1 = exp2f(fmaf(s[j][1], a.scale_log2, -mn1));
      const float p2 = exp2f(fmaf(s[j][2], a.scale_log2, -mn0));
      const float p3 = exp2f(fmaf(s[j][3], a.scale_log2, -mn1));
      l_run[0] += p0 + p2;
      l_run[1] += p1 + p3;
      const uint32_t top = f2_to_bf2(p0, p1), bot = f2_to_bf2(p2, p3);
      const f2 th = bf2_to_f2(top), bh = bf2_to_f2(bot);
      const uint32_t topl = f2_to_bf2(p0 - th.x, p1 - th.y);
      const uint32_t botl = f2_to_bf2(p2 - bh.x, p3 - bh.y);
      pb_hi[j][0] = movtrans(top);
      pb_hi[j][1] = movtrans(bot);
      pb_lo[j][0] = movtrans(topl);
      pb_lo[j][1] = movtrans(botl);
    }

    // ---- output: O^T += V^T P^T over V m-tiles mt (byte 8g + mt)
#pragma unroll
    for (int G2 = 0; G2 < 2; ++G2) {
      const int grp = 2 * g + G2;
      const float* vs = scr + 6 * kD;
      float gm[8], gs[8], mu[2][8], sg[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float4 x0 = reinterpret_cast<const float4*>(vs + 0 * kD + 8 * grp)[i];
        const float4 x1 = reinterpret_cast<const float4*>(vs + 1 * kD + 8 * grp)[i];
        gm[4 * i] = x0.x; gm[4 * i + 1] = x0.y; gm[4 * i + 2] = x0.z; gm[4 * i + 3] = x0.w;
        gs[4 * i] = x1.x; gs[4 * i + 1] = x1.y; gs[4 * i + 2] = x1.z; gs[4 * i + 3] = x1.w;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float4 y0 = reinterpret_cast<const float4*>(vs + (2 + j) * kD + 8 * grp)[i];
          const float4 y1 = reinterpret_cast<const float4*>(vs + (4 + j) * kD + 8 * grp)[i];
          mu[j][4 * i] = y0.x; mu[j][4 * i + 1] = y0.y; mu[j][4 * i + 2] = y0.z; mu[j][4 * i + 3] = y0.w;
          sg[j][4 * i] = y1.x; sg[j][4 * i + 1] = y1.y; sg[j][4 * i + 2] = y1.z; sg[j][4 * i + 3] = y1.w;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int mt = 4 * G2 + kk;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t W[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {   // tokens 2c, 2c+1, 2c+8, 2c+9
            const uint2 va = vA[4 * j + q4];
            const uint32_t wa = G2 == 0 ? va.x : va.y;
            uint32_t wr = 0;
            if constexpr (FULL) wr = G2 == 0 ? vR[4 * j + q4].x : vR[4 * j + q4].y;
            const uint32_t ab = (wa >> (8 * kk)) & 0xffu;
            const uint32_t rb = (wr >> (8 * kk)) & 0xffu;
            W[q4] = dequant_pair<FULL>(lut, ab, rb, lane, gm[kk], gm[kk + 4], gs[kk], gs[kk + 4],
                                       mu[j][kk], mu[j][kk + 4], sg[j][kk], sg[j][kk + 4]);
          }
          uint32_t af[4];
          af[0] = prmt(W[0], W[1], 0x5410u);  // row g   (low channel), tokens 2c, 2c+1
          af[1] = prmt(W[0], W[1], 0x7632u);  // row g+8 (high channel)
          af[2] = prmt(W[2], W[3], 0x5410u);  // row g,   tokens 2c+8, 2c+9
          af[3] = prmt(W[2], W[3], 0x7632u);
          mma_bf16(o[mt], af, pb_hi[j][0], pb_hi[j][1]);
          mma_bf16(o[mt], af, pb_lo[j][0], pb_lo[j][1]);
        }
      }
    }
    __syncwarp();
  }

  // ---- merge the 4 warps of the CTA, write this split's partial
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], x);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], x);
  }
  __syncthreads();  // everyone is done with the lookup table; reuse it
  float* sm_m = reinterpret_cast<float*>(smem);                 // [4][8]
  float* sm_l = sm_m + kAttnWarps * kRows;                       // [4][8]
  float* sm_o = sm_l + kAttnWarps * kRows;                       // [4][8][128]
  if (g == 0) {
    sm_m[w * kRows + 2 * c] = m_run[0];
    sm_m[w * kRows + 2 * c + 1] = m_run[1];
    sm_l[w * kRows + 2 * c] = l_run[0];
    sm_l[w * kRows + 2 * c + 1] = l_run[1];
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int beta = 8 * g + mt;
    const int ch_lo = 8 * (beta >> 2) + (beta & 3), ch_hi = ch_lo + 4;
    float* ow = sm_o + w * kRows * kD;
    ow[(2 * c) * kD + ch_lo] = o[mt][0];
    ow[(2 * c + 1) * kD + ch_lo] = o[mt][1];
    ow[(2 * c) * kD + ch_hi] = o[mt][2];
    ow[(2 * c + 1) * kD + ch_hi] = o[mt][3];
  }
  __syncthreads();
  float* part = a.part + ((((int64_t)b * a.Hkv + h) * a.nrg + rg) * a.S + split) * kPartFloats;
  for (int i = tid; i < kRows * kD; i += kAttnWarps * 32) {
    const int r = i / kD, d = i % kD;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kAttnWarps; ++ww) M = fmaxf(M, sm_m[ww * kRows + r]);
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int ww = 0; ww < kAttnWarps; ++ww) {
      const float mw = sm_m[ww * kRows + r];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      acc += f * sm_o[(ww * kRows + r) * kD + d];
      den += f * sm_l[ww * kRows + r];
    }
    part[2 * kRows + r * kD + d] = acc;
    if (d == 0) {
      part[r] = M;
      part[kRows + r] = den;
    }
  }
}

// Merge the splits of one (sequence, KV head, row group): out = sum e^(m_s-M)
// o_s / sum e^(m_s-M) l_s, written to out[b][t][hq][:].
__global__ void __launch_bounds__(kD) attn_combine(const __grid_constant__ AttnParams a) {
  const int z = blockIdx.x;  // (b * Hkv + h) * nrg + rg
  const int rg = z % a.nrg, bh = z / a.nrg, h = bh % a.Hkv, b = bh / a.Hkv;
  const int d = threadIdx.x;
  const float* part = a.part + (int64_t)z * a.S * kPartFloats;
  for (int r = 0; r < kRows; ++r) {
    const int row = rg * kRows + r;
    if (row >= a.R) break;
    float M = -INFINITY;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, part[s * kPartFloats + r]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < a.S; ++s) {
      const float* ps = part + s * kPartFloats;
      const float f = ps[r] == -INFINITY ? 0.f : exp2f(ps[r] - M);
      num += f * ps[2 * kRows + r * kD + d];
      den += f * ps[kRows + r];
    }
    const int tq = row / a.G, gq = row % a.G;
    a.out[((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD + d] = num / den;
  }
}

// ------------------------------------------------------------------ host

static int row_groups(int G, int T) { return (G * T + kRows - 1) / kRows; }

// Splits per (sequence, KV head, row group): about 512 CTAs in all, each
// with at least 4 chunks of 32 tokens (one per warp).  Device independent,
// so the workspace size is a pure function of the shapes.
static int splits_for(int batch, int Hkv, int nrg, int64_t NCH) {
  const int64_t units = (int64_t)batch * Hkv * nrg;
  int64_t s = (512 + units - 1) / units;
  const int64_t cap = NCH / kAttnWarps > 0 ? NCH / kAttnWarps : 1;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return (int)s;
}

size_t attn_workspace_bytes(int batch, int T, int H_q, int H_kv, int64_t L) {
  const int G = H_q / H_kv, nrg = row_groups(G, T);
  const int S = splits_for(batch, H_kv, nrg, L / 32);
  return (size_t)batch * H_kv * nrg * S * kPartFloats * sizeof(float);
}

template <bool FULL>
static cudaError_t run_attn(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  auto fn = attn_kernel<FULL>;
  constexpr size_t smem = 32768 + (size_t)kAttnWarps * kScratchFloats * sizeof(float);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  dim3 grid((unsigned)prm.S, (unsigned)prm.Hkv, (unsigned)(prm.batch * prm.nrg));
  fn<<<grid, kAttnWarps * 32, smem, stream>>>(prm, tab);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine<<<(unsigned)(prm.batch * prm.Hkv * prm.nrg), kD, 0, stream>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_attn(const AttnArgs& x, const ExpandTable& tab, cudaStream_t stream) {
  AttnParams prm;
  prm.q = static_cast<const uint16_t*>(x.q);
  prm.ka = static_cast<const uint8_t*>(x.k_anchor);
  prm.kr = static_cast<const uint8_t*>(x.k_residual);
  prm.va = static_cast<const uint8_t*>(x.v_anchor);
  prm.vr = static_cast<const uint8_t*>(x.v_residual);
  prm.km = x.k_meta;
  prm.vm = x.v_meta;
  prm.part = static_cast<float*>(x.workspace);
  prm.out = x.out;
  prm.batch = x.batch;
  prm.T = x.T;
  prm.Hq = x.H_q;
  prm.Hkv = x.s.H;
  prm.G = x.H_q / x.s.H;
  prm.R = prm.G * x.T;
  prm.nrg = row_groups(prm.G, x.T);
  prm.L = x.s.L;
  prm.NB = x.s.NB();
  prm.NCH = x.s.L / 32;
  prm.S = splits_for(x.batch, prm.Hkv, prm.nrg, prm.NCH);
  prm.P = x.s.page;
  prm.C = x.s.C;
  prm.NC = x.s.NC();
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  return x.full ? run_attn<true>(prm, tab, stream) : run_attn<false>(prm, tab, stream);
}

}  // namespace lynx

// ------------------------------------------------- allocation-free variant
//
// Some callers cannot call cudaMalloc at all: code running while a CUDA graph
// is being captured on a stream, real-time or signal-safe paths that must not
// enter the allocator, and hosts whose memory manager forbids driver
// allocations after start-up.  For them lynx_attn_decode_noalloc uses a fixed
// scratch array that lives in this library's device image, so the caller only
// passes inputs and outputs.

namespace lynx {

// Split-K partials of one call.  Every GPU that loads the library holds it
// until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch for the current device, looked up once
// per device (cudaGetSymbolAddress with that device current) and cached.
static cudaError_t noalloc_scratch(void** ptr) {
  constexpr int kMaxDev = 64;
  static void* addr[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace lynx

extern "C" int lynx_attn_decode_noalloc(const void* q, int batch, int T, int H_q,
                                        const void* k_anchor, const void* k_residual,
                                        const float* k_meta, const void* v_anchor,
                                        const void* v_residual, const float* v_meta, int64_t L,
                                        int H_kv, int D, int page, int C, float alpha, int mode,
                                        float* out, void* stream) {
  size_t need = 0;
  int rc = lynx_attn_workspace_bytes(batch, T, H_q, L, H_kv, D, page, &need);
  if (rc != LYNX_OK) return rc;
  if (need > lynx::kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "lynx_attn_decode_noalloc: these sizes need %zu bytes of scratch, more than the "
             "built-in %zu; use lynx_attn_decode with a workspace",
             need, lynx::kNoAllocScratchBytes);
    return lynx::report_error(LYNX_EWORKSPACE, msg);
  }
  void* scratch = nullptr;
  cudaError_t e = lynx::noalloc_scratch(&scratch);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof msg, "lynx_attn_decode_noalloc: scratch address: %s",
             cudaGetErrorString(e));
    return lynx::report_error(LYNX_ECUDA, msg);
  }
  return lynx_attn_decode(q, batch, T, H_q, k_anchor, k_residual, k_meta, v_anchor, v_residual,
                          v_meta, L, H_kv, D, page, C, alpha, mode, out, scratch,
                          lynx::kNoAllocScratchBytes, stream);
}
