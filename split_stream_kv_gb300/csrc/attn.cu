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
// A query "row" is one (query token, query head of the group).
//
// Two shapes of one kernel template:
//  * single (up to 8 rows per KV head, e.g. the draft step): every warp owns
//    its own 32-token chunks and all 128 channels of K and V.
//  * pair (up to 32 rows, e.g. the T = 8 verification): two warps share each
//    32-token chunk.  Each dequantises half of the channels of K (its partial
//    scores are summed with the partner's through shared memory) and half of
//    the channels of V (it accumulates that half of O^T), so every packed
//    element is decoded once.
// The contraction index (channel) of the scores is permuted so that a lane's
// fragment bytes are contiguous in a packed row: lane c (= lane % 4) owns KB
// consecutive bytes of K rows, lane g (= lane / 4) owns VB consecutive bytes
// of V rows, and V m-tile mt takes byte VB*g + mt, whose two channels are the
// rows g and g+8 of that m-tile.
// P is split into bf16 hi + lo parts (two MMAs) so the softmax weights keep
// about 16 mantissa bits; movmatrix turns the S^T accumulator layout into the
// P^T operand layout.
//
// Work split (flash-decoding): grid = (splits, H_kv, batch * row groups).
// Each unit (warp, or warp pair) walks its own 32-token chunks of the CTA's
// token range with its own running max / sum / output; the CTA merges its
// units and writes one partial (m, l, o) per split; attn_combine merges the
// splits.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "lynx.h"

namespace lynx {

constexpr int kAttnWarps = 4;
// The lookup table has 256 rows of 256 bytes, one per byte value (anchor
// mode: one anchor byte = two channels; full mode: one 8-bit code).  The
// first 128 bytes of a row are the lane-replicated entries (anchor: 16
// lane slots x float2, full: 32 lanes x float), so a lookup address is
// (byte << 8) | lane_offset: a single byte permute.  The second 128 bytes of
// every row hold the per-warp constant scratch.
constexpr int kLutBytes = 65536;
// Per-warp constant rows (gamma_min, gamma_scale+eps, mu, sigma+eps; mu and
// sigma once more for the second 16-token half when C = 16) of K and V.  A
// row holds 128 channels in groups of 8, stored as the pairs (k, k+4) of the
// nibble pairing so that one 16-byte load gives two float2 operands, with 16
// bytes of padding after every 4 groups so that lanes reading different
// groups hit different banks.  Float f of the scratch lives at byte
// (f / 32) * 256 + 128 + (f % 32) * 4 of the table.
constexpr int kRowFloats = 144;
template <bool ONE>
struct Scratch {
  static constexpr int kRows = ONE ? 4 : 6;                 // per tensor
  static constexpr int kFloats = 2 * kRows * kRowFloats;    // K and V
};
static_assert(kAttnWarps * Scratch<false>::kFloats <= 256 * 32, "scratch fits the table rows");

__device__ __forceinline__ uint32_t scr_byte(int f) {
  return ((uint32_t)(f >> 5) << 8) | 128u | ((uint32_t)(f & 31) << 2);
}

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
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}
template <int N>
struct Bytes;  // N packed bytes loaded from one row
template <>
struct Bytes<16> {
  uint32_t w[4];
  __device__ __forceinline__ void load(const uint8_t* p) {
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p));
  }
};
template <>
struct Bytes<8> {
  uint32_t w[2];
  __device__ __forceinline__ void load(const uint8_t* p) {
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
  }
};
template <>
struct Bytes<4> {
  uint32_t w[1];
  __device__ __forceinline__ void load(const uint8_t* p) {
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(w[0]) : "l"(p));
  }
};

// Float offset of the first of channel group grp's 8 values in a row.
__device__ __forceinline__ int grp_off(int grp) { return grp * 8 + (grp >> 2) * 4; }

struct Consts {  // pairs (k, k+4) of one channel group, k = 0..3
  f2 gm[4], gs[4], mu[4], sg[4];
};
__device__ __forceinline__ float4 ld_scr(const uint8_t* smem, int f) {
  return *reinterpret_cast<const float4*>(smem + scr_byte(f));
}
// rows: first float of this tensor's rows in the warp's scratch.
__device__ __forceinline__ void load_consts(Consts& k, const uint8_t* smem, int rows, int grp,
                                            int jrow) {
  const int base = rows + grp_off(grp);
  const float4 g0 = ld_scr(smem, base), g1 = ld_scr(smem, base + 4);
  const float4 s0 = ld_scr(smem, base + kRowFloats), s1 = ld_scr(smem, base + kRowFloats + 4);
  const int mr = base + (2 + 2 * jrow) * kRowFloats, ar = base + (3 + 2 * jrow) * kRowFloats;
  const float4 m0 = ld_scr(smem, mr), m1 = ld_scr(smem, mr + 4);
  const float4 a0 = ld_scr(smem, ar), a1 = ld_scr(smem, ar + 4);
  k.gm[0] = {g0.x, g0.y}; k.gm[1] = {g0.z, g0.w}; k.gm[2] = {g1.x, g1.y}; k.gm[3] = {g1.z, g1.w};
  k.gs[0] = {s0.x, s0.y}; k.gs[1] = {s0.z, s0.w}; k.gs[2] = {s1.x, s1.y}; k.gs[3] = {s1.z, s1.w};
  k.mu[0] = {m0.x, m0.y}; k.mu[1] = {m0.z, m0.w}; k.mu[2] = {m1.x, m1.y}; k.mu[3] = {m1.z, m1.w};
  k.sg[0] = {a0.x, a0.y}; k.sg[1] = {a0.z, a0.w}; k.sg[2] = {a1.x, a1.y}; k.sg[3] = {a1.z, a1.w};
}

// Table byte address of byte `pos` (0..3) of word w, row-major with lane_off.
template <int POS>
__device__ __forceinline__ uint32_t lut_addr(uint32_t w, uint32_t lane_off) {
  // result bytes: [lane_off.b0, w.b_POS, 0, 0] (lane_off < 256)
  return prmt(w, lane_off, 0x6504u | ((uint32_t)POS << 4));
}

// Values of the two channels of byte POS of an anchor word a (and, in full
// mode, of residual word r): (low-nibble channel, high-nibble channel).
template <bool FULL, int POS>
__device__ __forceinline__ f2 lookup_pair(const uint8_t* lut, uint32_t a, uint32_t r,
                                          uint32_t lane_off) {
  if constexpr (FULL) {
    const uint32_t E = ((a << 4) & 0xf0f0f0f0u) | (r & 0x0f0f0f0fu);  // low-nibble codes
    const uint32_t O = (a & 0xf0f0f0f0u) | ((r >> 4) & 0x0f0f0f0fu);  // high-nibble codes
    f2 v;
    v.x = *reinterpret_cast<const float*>(lut + lut_addr<POS>(E, lane_off));
    v.y = *reinterpret_cast<const float*>(lut + lut_addr<POS>(O, lane_off));
    return v;
  } else {
    const float2 p = *reinterpret_cast<const float2*>(lut + lut_addr<POS>(a, lane_off));
    return f2{p.x, p.y};
  }
}

// One packed byte position -> bf16x2 of the exact decoder output
// (low-nibble channel in the low half).
template <bool FULL, int POS>
__device__ __forceinline__ uint32_t dequant_pair(const uint8_t* lut, uint32_t a, uint32_t r,
                                                 uint32_t lane_off, const Consts& k) {
  const f2 v = lookup_pair<FULL, POS>(lut, a, r, lane_off);
  const f2 x = fma2(fma2(v, k.sg[POS], k.mu[POS]), k.gs[POS], k.gm[POS]);
  return f2_to_bf2(x.x, x.y);
}

template <bool FULL, int NT, bool PAIR, bool ONE>
__global__ void __launch_bounds__(kAttnWarps * 32, PAIR ? 2 : 3)
attn_kernel(const __grid_constant__ AttnParams a, const __grid_constant__ ExpandTable tab) {
  constexpr int KCH = PAIR ? 64 : 128;  // channels of K and of V per warp
  constexpr int NKT = KCH / 16;         // score k-tiles = output m-tiles per warp
  constexpr int KB = KCH / 8;           // K bytes per token row per lane (c)
  constexpr int VB = KCH / 16;          // V bytes per token row per lane (g)
  constexpr int NU = PAIR ? kAttnWarps / 2 : kAttnWarps;  // work units per CTA
  constexpr int RP = 8 * NT;            // query rows per pass
  using SC = Scratch<ONE>;

  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* lut = smem;
  float* xchg_all = reinterpret_cast<float*>(smem + kLutBytes);  // pair: partial scores
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int unit = PAIR ? (w >> 1) : w;
  const int half = PAIR ? (w & 1) : 0;
  const int hb = half * 32;             // first byte of this warp's channel half

  for (int i = tid; i < 256 * 32; i += kAttnWarps * 32) {
    const int row = i >> 5, l = i & 31;
    if constexpr (FULL) {
      reinterpret_cast<float*>(lut + row * 256)[l] =
          row < 128 ? tab.x[row] : -tab.x[255 - row];
    } else if (l < 16) {
      const int a0 = row & 15, a1 = row >> 4;
      reinterpret_cast<float2*>(lut + row * 256)[l] =
          make_float2(a0 < 8 ? tab.x[16 * a0 + 7] : -tab.x[16 * (15 - a0) + 7],
                      a1 < 8 ? tab.x[16 * a1 + 7] : -tab.x[16 * (15 - a1) + 7]);
    }
  }
  __syncthreads();
  const uint32_t lane_off = FULL ? (uint32_t)lane * 4u : (uint32_t)(lane & 15) * 8u;

  const int split = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / a.nrg, rg = blockIdx.z % a.nrg;
  const int row0 = rg * RP;

  // ---- Q^T fragments (B operand), channel order matching the K bytes
  uint32_t qf[NKT][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = row0 + nt * 8 + g;
    const bool valid = r < a.R;
    const int tq = valid ? r / a.G : 0, gq = valid ? r % a.G : 0;
    const uint16_t* qrow = a.q + ((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD;
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int beta = hb + KB * c + 2 * kt + hh;
        const int lo = 8 * (beta >> 2) + (beta & 3);
        qf[kt][nt][hh] = valid ? ((uint32_t)qrow[lo] | ((uint32_t)qrow[lo + 4] << 16)) : 0u;
      }
  }

  const int scr = w * SC::kFloats;     // this warp's scratch (K rows, then V rows)
  const int scrV = scr + SC::kRows * kRowFloats;
  const int64_t cb = a.NCH * split / a.S, ce = a.NCH * (split + 1) / a.S;
  float m_run[NT][2], l_run[NT][2];
  float o[NKT][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int i = 0; i < NKT; ++i) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
  }
  const int meta_rows = 2 + 2 * a.NC;
  int it = 0;

  for (int64_t qc = cb + unit; qc < ce; qc += NU, ++it) {
    const int64_t t0 = qc * 32;
    const int64_t p = t0 / a.P;
    const int tp = (int)(t0 - p * a.P);
    const int64_t blk = ((int64_t)b * a.NB + p) * a.Hkv + h;
    const int64_t code_off = (blk * a.P + tp) * (kD / 2);

    // ---- packed codes of this chunk (K: 4 rows per lane, V: 8 rows)
    Bytes<KB> kA[4], kR[4];
    Bytes<VB> vA[8], vR[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int row = 16 * (jj >> 1) + g + 8 * (jj & 1);
      kA[jj].load(a.ka + code_off + row * 64 + hb + KB * c);
      if constexpr (FULL) kR[jj].load(a.kr + code_off + row * 64 + hb + KB * c);
    }
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int kk = ii & 3;
      const int row = 16 * (ii >> 2) + 2 * c + (kk & 1) + 8 * (kk >> 1);
      vA[ii].load(a.va + code_off + row * 64 + hb + VB * g);
      if constexpr (FULL) vR[ii].load(a.vr + code_off + row * 64 + hb + VB * g);
    }
    // ---- warm L2 with the next chunk of this unit (2 KB per stream)
    if (qc + NU < ce) {
      const int64_t t1 = (qc + NU) * 32;
      const int64_t p1 = t1 / a.P;
      const int64_t blk1 = ((int64_t)b * a.NB + p1) * a.Hkv + h;
      const int64_t off1 = (blk1 * a.P + (t1 - p1 * a.P)) * (kD / 2) + lane * 64;
      prefetch_l2(a.ka + off1);
      prefetch_l2(a.va + off1);
      if constexpr (FULL) {
        prefetch_l2(a.kr + off1);
        prefetch_l2(a.vr + off1);
      }
    }
    // ---- constant rows -> scratch (pairs (k, k+4) interleaved, +eps folded)
    {
      const int cc0 = tp / a.C, cc1 = (tp + 16) / a.C;
      const int grp = lane >> 1, hf = lane & 1;
#pragma unroll
      for (int tsr = 0; tsr < 2; ++tsr) {
        const float* mb = (tsr == 0 ? a.km : a.vm) + blk * (int64_t)meta_rows * kD + 8 * grp + 2 * hf;
        const int rows = tsr == 0 ? scr : scrV;
#pragma unroll
        for (int rr = 0; rr < SC::kRows; ++rr) {
          const int src = rr == 0 ? 0 : rr == 1 ? 1 : rr == 2 ? 2 + cc0 : rr == 3 ? 2 + a.NC + cc0
                        : rr == 4 ? 2 + cc1 : 2 + a.NC + cc1;
          const float2 lo = __ldg(reinterpret_cast<const float2*>(mb + src * kD));
          const float2 hi = __ldg(reinterpret_cast<const float2*>(mb + src * kD + 4));
          float4 v = make_float4(lo.x, hi.x, lo.y, hi.y);
          if (rr == 1 || rr == 3 || rr == 5) {
            v.x = __fadd_rn(v.x, kEps); v.y = __fadd_rn(v.y, kEps);
            v.z = __fadd_rn(v.z, kEps); v.w = __fadd_rn(v.w, kEps);
          }
          *reinterpret_cast<float4*>(smem + scr_byte(rows + rr * kRowFloats + grp_off(grp) + 4 * hf)) = v;
        }
      }
    }
    __syncwarp();

    // ---- scores: S^T for m-tiles j = 0, 1 (tokens 16j .. 16j+15)
    float s[2][NT][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[j][nt][0] = s[j][nt][1] = s[j][nt][2] = s[j][nt][3] = 0.f;
    // one 16-token m-tile j of the scores with this group's constants
    auto qk = [&](const Consts& kc, int j, int gi) {
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int kt = 2 * gi + kk;
        uint32_t af[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {       // row g (i=0) / g+8 (i=1)
          const uint32_t wa = kA[2 * j + i].w[gi];
          const uint32_t wr = FULL ? kR[2 * j + i].w[gi] : 0u;
          if (kk == 0) {                    // k 2c..2c+1 / 2c+8..2c+9 = bytes 0 / 1
            af[i] = dequant_pair<FULL, 0>(lut, wa, wr, lane_off, kc);
            af[i + 2] = dequant_pair<FULL, 1>(lut, wa, wr, lane_off, kc);
          } else {                          // bytes 2 / 3
            af[i] = dequant_pair<FULL, 2>(lut, wa, wr, lane_off, kc);
            af[i + 2] = dequant_pair<FULL, 3>(lut, wa, wr, lane_off, kc);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(s[j][nt], af, qf[kt][nt][0], qf[kt][nt][1]);
      }
    };
#pragma unroll
    for (int gi = 0; gi < KB / 4; ++gi) {      // channel groups of this lane (K)
      const int grp = (hb + KB * c) / 4 + gi;
      if constexpr (ONE) {
        Consts kc;
        load_consts(kc, smem, scr, grp, 0);
        qk(kc, 0, gi);
        qk(kc, 1, gi);
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          Consts kc;
          load_consts(kc, smem, scr, grp, j);
          qk(kc, j, gi);
        }
      }
    }

    if constexpr (PAIR) {
      // partial scores over this warp's channel half + the partner's half
      float* mine = xchg_all + ((unit * 2 + half) * 2 + (it & 1)) * (32 * 8 * NT);
      const float* other = xchg_all + ((unit * 2 + (half ^ 1)) * 2 + (it & 1)) * (32 * 8 * NT);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<float4*>(mine + ((j * NT + nt) * 32 + lane) * 4) =
              make_float4(s[j][nt][0], s[j][nt][1], s[j][nt][2], s[j][nt][3]);
      asm volatile("bar.sync %0, 64;" :: "r"(1 + unit) : "memory");
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float4 v = *reinterpret_cast<const float4*>(other + ((j * NT + nt) * 32 + lane) * 4);
          s[j][nt][0] += v.x; s[j][nt][1] += v.y; s[j][nt][2] += v.z; s[j][nt][3] += v.w;
        }
    }

    // ---- online softmax (log2 domain); rows nt*8 + 2c, nt*8 + 2c + 1
    uint32_t pb_hi[2][NT][2], pb_lo[2][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float cmax0 = fmaxf(fmaxf(s[0][nt][0], s[0][nt][2]), fmaxf(s[1][nt][0], s[1][nt][2]));
      float cmax1 = fmaxf(fmaxf(s[0][nt][1], s[0][nt][3]), fmaxf(s[1][nt][1], s[1][nt][3]));
#pragma unroll
      for (int x = 4; x <= 16; x <<= 1) {
        cmax0 = fmaxf(cmax0, __shfl_xor_sync(kFull, cmax0, x));
        cmax1 = fmaxf(cmax1, __shfl_xor_sync(kFull, cmax1, x));
      }
      const float mn0 = fmaxf(m_run[nt][0], cmax0 * a.scale_log2);
      const float mn1 = fmaxf(m_run[nt][1], cmax1 * a.scale_log2);
      if (mn0 != m_run[nt][0] || mn1 != m_run[nt][1]) {
        const float al0 = ex2(m_run[nt][0] - mn0), al1 = ex2(m_run[nt][1] - mn1);
        l_run[nt][0] *= al0;
        l_run[nt][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < NKT; ++mt) {
          o[mt][nt][0] *= al0; o[mt][nt][1] *= al1; o[mt][nt][2] *= al0; o[mt][nt][3] *= al1;
        }
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float p0 = ex2(fmaf(s[j][nt][0], a.scale_log2, -mn0));
        const float p1 = ex2(fmaf(s[j][nt][1], a.scale_log2, -mn1));
        const float p2 = ex2(fmaf(s[j][nt][2], a.scale_log2, -mn0));
        const float p3 = ex2(fmaf(s[j][nt][3], a.scale_log2, -mn1));
        l_run[nt][0] += p0 + p2;
        l_run[nt][1] += p1 + p3;
        const uint32_t top = f2_to_bf2(p0, p1), bot = f2_to_bf2(p2, p3);
        const f2 th = bf2_to_f2(top), bh = bf2_to_f2(bot);
        pb_hi[j][nt][0] = movtrans(top);
        pb_hi[j][nt][1] = movtrans(bot);
        pb_lo[j][nt][0] = movtrans(f2_to_bf2(p0 - th.x, p1 - th.y));
        pb_lo[j][nt][1] = movtrans(f2_to_bf2(p2 - bh.x, p3 - bh.y));
      }
    }

    // ---- output: O^T += V^T P^T over this warp's V m-tiles (byte VB*g + mt)
    auto pv = [&](const Consts& kc, int jt, int gi) {
#pragma unroll
      for (int kk = 0; kk < (VB < 4 ? VB : 4); ++kk) {
        const int mt = 4 * gi + kk;
        uint32_t W[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {   // tokens 2c, 2c+1, 2c+8, 2c+9
          const uint32_t wa = vA[4 * jt + q4].w[gi];
          const uint32_t wr = FULL ? vR[4 * jt + q4].w[gi] : 0u;
          W[q4] = kk == 0 ? dequant_pair<FULL, 0>(lut, wa, wr, lane_off, kc)
                : kk == 1 ? dequant_pair<FULL, 1>(lut, wa, wr, lane_off, kc)
                : kk == 2 ? dequant_pair<FULL, 2>(lut, wa, wr, lane_off, kc)
                          : dequant_pair<FULL, 3>(lut, wa, wr, lane_off, kc);
        }
        uint32_t af[4];
        af[0] = prmt(W[0], W[1], 0x5410u);  // row g   (low channel), tokens 2c, 2c+1
        af[1] = prmt(W[0], W[1], 0x7632u);  // row g+8 (high channel)
        af[2] = prmt(W[2], W[3], 0x5410u);  // row g,   tokens 2c+8, 2c+9
        af[3] = prmt(W[2], W[3], 0x7632u);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16(o[mt][nt], af, pb_hi[jt][nt][0], pb_hi[jt][nt][1]);
          mma_bf16(o[mt][nt], af, pb_lo[jt][nt][0], pb_lo[jt][nt][1]);
        }
      }
    };
#pragma unroll
    for (int gi = 0; gi < (VB + 3) / 4; ++gi) {
      const int grp = (hb + VB * g) / 4 + gi;
      if constexpr (ONE) {
        Consts kc;
        load_consts(kc, smem, scrV, grp, 0);
        pv(kc, 0, gi);
        pv(kc, 1, gi);
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          Consts kc;
          load_consts(kc, smem, scrV, grp, j);
          pv(kc, j, gi);
        }
      }
    }
    __syncwarp();
  }

  // ---- merge the units of the CTA, write this split's partial
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      l_run[nt][0] += __shfl_xor_sync(kFull, l_run[nt][0], x);
      l_run[nt][1] += __shfl_xor_sync(kFull, l_run[nt][1], x);
    }
  __syncthreads();  // every warp is done with the tables and scratch; reuse them
  float* sm_m = reinterpret_cast<float*>(smem);       // [NU][RP]
  float* sm_l = sm_m + NU * RP;                        // [NU][RP]
  float* sm_o = sm_l + NU * RP;                        // [NU][RP][128]
  if (g == 0 && half == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sm_m[unit * RP + nt * 8 + 2 * c] = m_run[nt][0];
      sm_m[unit * RP + nt * 8 + 2 * c + 1] = m_run[nt][1];
      sm_l[unit * RP + nt * 8 + 2 * c] = l_run[nt][0];
      sm_l[unit * RP + nt * 8 + 2 * c + 1] = l_run[nt][1];
    }
  }
#pragma unroll
  for (int mt = 0; mt < NKT; ++mt) {
    const int beta = hb + VB * g + mt;
    const int ch_lo = 8 * (beta >> 2) + (beta & 3), ch_hi = ch_lo + 4;
    float* ow = sm_o + unit * RP * kD;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      ow[(nt * 8 + 2 * c) * kD + ch_lo] = o[mt][nt][0];
      ow[(nt * 8 + 2 * c + 1) * kD + ch_lo] = o[mt][nt][1];
      ow[(nt * 8 + 2 * c) * kD + ch_hi] = o[mt][nt][2];
      ow[(nt * 8 + 2 * c + 1) * kD + ch_hi] = o[mt][nt][3];
    }
  }
  __syncthreads();
  const int part_floats = 2 * RP + RP * kD;
  float* part = a.part + ((((int64_t)b * a.Hkv + h) * a.nrg + rg) * a.S + split) * part_floats;
  for (int i = tid; i < RP * kD; i += kAttnWarps * 32) {
    const int r = i / kD, d = i % kD;
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < NU; ++u) M = fmaxf(M, sm_m[u * RP + r]);
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const float mu_ = sm_m[u * RP + r];
      const float f = mu_ == -INFINITY ? 0.f : exp2f(mu_ - M);
      acc += f * sm_o[(u * RP + r) * kD + d];
      den += f * sm_l[u * RP + r];
    }
    part[2 * RP + r * kD + d] = acc;
    if (d == 0) {
      part[r] = M;
      part[RP + r] = den;
    }
  }
}

// Merge the splits of one (sequence, KV head, row group): out = sum e^(m_s-M)
// o_s / sum e^(m_s-M) l_s, written to out[b][t][hq][:].
__global__ void __launch_bounds__(kD) attn_combine(const __grid_constant__ AttnParams a, int RP) {
  const int z = blockIdx.x;  // (b * Hkv + h) * nrg + rg
  const int rg = z % a.nrg, bh = z / a.nrg, h = bh % a.Hkv, b = bh / a.Hkv;
  const int d = threadIdx.x;
  const int part_floats = 2 * RP + RP * kD;
  const float* part = a.part + (int64_t)z * a.S * part_floats;
  for (int r = 0; r < RP; ++r) {
    const int row = rg * RP + r;
    if (row >= a.R) break;
    float M = -INFINITY;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, part[s * part_floats + r]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < a.S; ++s) {
      const float* ps = part + s * part_floats;
      const float f = ps[r] == -INFINITY ? 0.f : exp2f(ps[r] - M);
      num += f * ps[2 * RP + r * kD + d];
      den += f * ps[RP + r];
    }
    const int tq = row / a.G, gq = row % a.G;
    a.out[((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD + d] = num / den;
  }
}

// ------------------------------------------------------------------ host

// Query rows per pass: one n-tile (8 rows) for small groups, else a warp
// pair over four n-tiles (32 rows).
static int rows_per_pass(int R) { return R <= 8 ? 8 : 32; }
static int row_groups(int R) { const int rp = rows_per_pass(R); return (R + rp - 1) / rp; }

// Splits per (sequence, KV head, row group): as many as fit one wave of
// CTAs on the 152 SMs of a GB300 (3 resident CTAs per SM for the single-warp
// shape, 2 for the warp-pair shape), so that no partial second wave leaves
// SMs idle; at least one 32-token chunk per work unit.  Device independent,
// so the workspace size is a pure function of the shapes.
constexpr int kGB300SMs = 152;
static int splits_for(int batch, int Hkv, int nrg, int64_t NCH, int R) {
  const int64_t units = (int64_t)batch * Hkv * nrg;
  const int64_t slots = (int64_t)kGB300SMs * (R <= 8 ? 3 : 2);
  int64_t s = slots / units;
  const int64_t nu = R <= 8 ? kAttnWarps : kAttnWarps / 2;
  const int64_t cap = NCH / nu > 0 ? NCH / nu : 1;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return (int)s;
}

size_t attn_workspace_bytes(int batch, int T, int H_q, int H_kv, int64_t L) {
  const int R = (H_q / H_kv) * T;
  const int RP = rows_per_pass(R), nrg = row_groups(R);
  const int S = splits_for(batch, H_kv, nrg, L / 32, R);
  return (size_t)batch * H_kv * nrg * S * (2 * RP + RP * kD) * sizeof(float);
}

template <bool FULL, int NT, bool PAIR, bool ONE>
static cudaError_t run_attn(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  auto fn = attn_kernel<FULL, NT, PAIR, ONE>;
  constexpr size_t xchg = PAIR ? (size_t)kAttnWarps * 2 * 32 * 8 * NT * sizeof(float) : 0;
  constexpr size_t smem = kLutBytes + xchg;
  static_assert((size_t)(kAttnWarps / (PAIR ? 2 : 1)) * (2 + 128) * 8 * NT * sizeof(float) <= smem,
                "merge buffers fit in the reused tables");
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  dim3 grid((unsigned)prm.S, (unsigned)prm.Hkv, (unsigned)(prm.batch * prm.nrg));
  fn<<<grid, kAttnWarps * 32, smem, stream>>>(prm, tab);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine<<<(unsigned)(prm.batch * prm.Hkv * prm.nrg), kD, 0, stream>>>(prm, 8 * NT);
  return cudaGetLastError();
}

template <bool FULL, int NT, bool PAIR>
static cudaError_t run_attn_c(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  return prm.C >= 32 ? run_attn<FULL, NT, PAIR, true>(prm, tab, stream)
                     : run_attn<FULL, NT, PAIR, false>(prm, tab, stream);
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
  prm.nrg = row_groups(prm.R);
  prm.L = x.s.L;
  prm.NB = x.s.NB();
  prm.NCH = x.s.L / 32;
  prm.S = splits_for(x.batch, prm.Hkv, prm.nrg, prm.NCH, prm.R);
  prm.P = x.s.page;
  prm.C = x.s.C;
  prm.NC = x.s.NC();
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  const bool small = prm.R <= 8;
  if (x.full)
    return small ? run_attn_c<true, 1, false>(prm, tab, stream)
                 : run_attn_c<true, 4, true>(prm, tab, stream);
  return small ? run_attn_c<false, 1, false>(prm, tab, stream)
               : run_attn_c<false, 4, true>(prm, tab, stream);
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
