// attn.cu -- decode attention O = softmax(q K^T / sqrt(d)) V ("Lynx:
// Progressive Speculative KV Cache Transfer for Disaggregated LLM Inference",
// Prerequisites Eq. 1) read straight from the packed Lynx streams: the draft
// step over Anchor codes (Mechanism 2, Anchor Phase) and the T-token
// verification pass over Anchor + Residual (Mechanism 3).
//
// K and V are reconstructed in registers from the decoders' lookup values
// with one fused multiply-add, x = fma(v, A, B), A = (sigma + eps)(gamma_scale
// + eps) and B = fma(mu, gamma_scale + eps, gamma_min) built once per chunk and
// channel, then rounded to nearest even BF16, and fed to mma.sync m16n8k16
// (bf16 x bf16 -> f32).  The decoders apply the same affine map as two fused
// multiply-adds; the two float32 results differ by at most 2^-22 of the
// channel's gamma_scale + eps, so their BF16 roundings differ on about 2e-4 of
// the values: by one BF16 ulp, or, for a value that nearly cancels to zero in
// its channel, by that 2^-22 of the range.
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
#include <utility>

#include "common.cuh"
#include "attn_params.h"
#include "internal.h"
#include "lynx.h"

namespace lynx {

// Shared memory of one CTA (offsets from the start of the dynamic window):
//  [0, 64 KiB)  lookup table, 256 rows of 256 bytes, one row per byte value
//               (anchor mode: one anchor byte = two channels; full mode: one
//               8-bit code).  The first 128 bytes of a row are the
//               lane-replicated entries (anchor: 16 lane slots x float2, full:
//               32 lanes x float); the second 128 bytes ("tails") hold the
//               per-warp constant rows.  A lookup address is
//               (byte << 8) | lane_offset, one byte permute, plus the
//               constant shared-window base as the load's immediate offset.
//  [64 KiB, ..) Q fragments, the partner-score exchange of the warp-pair
//               shape, and at the end the merge buffers.
constexpr int kLutBytes = 65536;

template <bool FULL, bool PAIR, bool ONE>
struct Cfg {
  // 8 warps where everything fits 128 registers (anchor codes, up to 8 rows,
  // C >= 32: two CTAs = 16 warps per SM), else 4 warps at up to 255.
  static constexpr int kWarps = (!FULL && !PAIR && ONE) ? 8 : 4;
  static constexpr int kNU = PAIR ? kWarps / 2 : kWarps;  // work units
  // Constant rows per tensor in the table tails: the one-FMA decode constants
  // (A, B) of the chunk of each 16-token half (one pair when C >= 32), in the
  // (k, k+4) channel pairs of the nibble layout.
  static constexpr int kRows = ONE ? 2 : 4;
  static constexpr int kTails = 2 * kRows * 4;  // per warp: K then V, 4 tails a row
  // Raw metadata rows per tensor, in channel order: gamma_min, gamma_scale,
  // then (mu, sigma) of each 16-token half.  A warp pair stages them in the
  // free tails (a row of its 64 channels is 2 tails), a single warp (128
  // channels, 512-byte rows) in the extra region.
  static constexpr int kRawRows = ONE ? 4 : 6;
  static constexpr int kRawTails = PAIR ? 2 * kRawRows * 2 : 0;
  static_assert(kWarps * (kTails + kRawTails) <= 256, "constant rows fit the table tails");
};

// Bytes after the table: during the chunk loop the staged Q fragments (one
// set per segment), the pair exchange and the packed-block bases of the two
// segments; at the end the merge buffers.
template <bool FULL, bool PAIR, bool ONE, int NT>
struct ExtraLayout {
  using CF = Cfg<FULL, PAIR, ONE>;
  static constexpr int NKT = PAIR ? 4 : 8;
  static constexpr int kHalves = PAIR ? 2 : 1;
  static constexpr size_t kQ = (size_t)2 * kHalves * NKT * NT * 32 * 8;  // [seg][half][kt][nt][lane]
  static constexpr size_t kXchg = PAIR ? (size_t)CF::kWarps * 2 * 32 * 8 * NT * 4 : 0;
  static constexpr size_t kInfo = kQ + kXchg;  // int64 page-row base and head of segments 0, 1
  static constexpr size_t kRaw = kInfo + 32;   // single warps: raw rows, [warp][K, V][row][512 B]
  static constexpr size_t kRawBytes = PAIR ? 0 : (size_t)CF::kWarps * 2 * CF::kRawRows * 512;
  static_assert(kLutBytes + kRaw + kRawBytes <= 113 * 1024, "two CTAs per SM");
  static constexpr size_t kLoop = kRaw + kRawBytes;
  static constexpr size_t kMerge = (size_t)CF::kNU * 8 * NT * (2 + kD) * 4 + (size_t)CF::kNU * 8;
  static constexpr size_t kBytes = kLoop > kMerge ? kLoop : kMerge;
};
template <bool FULL, bool PAIR, bool ONE, int NT>
constexpr size_t attn_smem_bytes() {
  return kLutBytes + ExtraLayout<FULL, PAIR, ONE, NT>::kBytes;
}

// Byte offset (from the table start) of float4 unit h (0, 1) of channel
// group grp (8 channels) in constant row r of a tensor whose rows start at
// tail tb.  A row is 4 tails of 128 bytes; tail (grp >> 2) of the row holds
// groups 4(grp>>2) .. +3 at 32-byte slots XOR-swizzled by the tail index, so
// that lanes reading the same group slot of different tails hit different
// banks.  Unit h of a group holds the pairs (k, k+4) and (k+1, k+5) for
// k = 2h: the channels of nibble positions 2h and 2h+1 of the group's bytes.
__device__ __forceinline__ uint32_t unit_off(int tb, int r, int grp, int h) {
  return (uint32_t)((tb + r * 4 + (grp >> 2)) * 256 + 128 + (((grp & 3) ^ ((grp >> 2) & 3)) << 5) +
                    h * 16);
}
constexpr int kRowStride = 4 * 256;  // bytes between constant rows

// Set when a block-table entry was out of range (bit kFlagBadBlock); read
// through read_attn_flags(), never reset.
__device__ unsigned int g_attn_flags = 0;

cudaError_t read_attn_flags(unsigned int* flag) {
  unsigned int mine = 0, tc = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&mine, g_attn_flags, sizeof(unsigned int));
  if (e == cudaSuccess) e = read_attn_tc_flags(&tc);
  *flag = mine | tc;
  return e;
}


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
// Table reads.  The table is written once before the first barrier and never
// again, so these loads carry no ordering against other memory operations.
__device__ __forceinline__ float2 lut_f2(uint32_t off) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2+1024];" : "=f"(v.x), "=f"(v.y) : "r"(off));
  return v;
}
__device__ __forceinline__ float lut_f1(uint32_t off) {
  float v;
  asm("ld.shared.f32 %0, [%1+1024];" : "=f"(v) : "r"(off));
  return v;
}
static_assert(kSmemBase == 1024, "immediate offset of the table loads");
// 16-byte asynchronous copy global -> shared, cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
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

// One-FMA decode constants of two nibble positions (2hh, 2hh+1) of one
// channel group: the pairs (k, k+4) for k = 2hh, 2hh+1 of
// A = (sigma + eps)(gamma_scale + eps) and B = fma(mu, gamma_scale + eps, gamma_min).
struct Half {
  f2 A[2], B[2];
};
// gb: byte offset of unit 0 of the group in row 0 (unit_off(tb, 0, grp, 0)).
// Rows 2 jrow and 2 jrow + 1 hold A and B of the chunk of token half jrow.
__device__ __forceinline__ void load_half(Half& k, const uint8_t* smem, uint32_t gb, int jrow,
                                          int hh) {
  const uint8_t* p = smem + gb + hh * 16;
  const float4 a = *reinterpret_cast<const float4*>(p + (2 * jrow) * kRowStride);
  const float4 b = *reinterpret_cast<const float4*>(p + (2 * jrow + 1) * kRowStride);
  k.A[0] = make_float2(a.x, a.y);
  k.A[1] = make_float2(a.z, a.w);
  k.B[0] = make_float2(b.x, b.y);
  k.B[1] = make_float2(b.z, b.w);
}

// Table offset of byte `pos` (0..3) of word w: [lane_off, w.b_pos, 0, 0].
template <int POS>
__device__ __forceinline__ uint32_t lut_off(uint32_t w, uint32_t lane_off) {
  return prmt(w, lane_off, 0x7604u | ((uint32_t)POS << 4));
}

// Values of the two channels of byte POS of an anchor word a (and, in full
// mode, of residual word r): (low-nibble channel, high-nibble channel).
template <bool FULL, int POS>
__device__ __forceinline__ f2 lookup_pair(uint32_t a, uint32_t r, uint32_t lane_off) {
  if constexpr (FULL) {
    const uint32_t E = ((a << 4) & 0xf0f0f0f0u) | (r & 0x0f0f0f0fu);  // low-nibble codes
    const uint32_t O = (a & 0xf0f0f0f0u) | ((r >> 4) & 0x0f0f0f0fu);  // high-nibble codes
    return make_float2(lut_f1(lut_off<POS>(E, lane_off)), lut_f1(lut_off<POS>(O, lane_off)));
  } else {
    return lut_f2(lut_off<POS>(a, lane_off));
  }
}

// Byte POS (0..3) of the packed words -> bf16x2 of the exact decoder output
// (low-nibble channel in the low half); k holds the constants of positions
// POS & ~1 and POS | 1.
template <bool FULL, int POS>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t a, uint32_t r, uint32_t lane_off,
                                                 const Half& k) {
  constexpr int i = POS & 1;
  const f2 v = lookup_pair<FULL, POS>(a, r, lane_off);
  const f2 x = fma2(v, k.A[i], k.B[i]);
  return f2_to_bf2(x.x, x.y);
}

// DIRECT: every work unit lies in one CTA's share and there is no draft-token
// tail, so the CTA writes the unit's output rows itself (no split combine).
template <bool FULL, int NT, bool PAIR, bool ONE, bool PAGED, bool DIRECT>
__global__ void __launch_bounds__(Cfg<FULL, PAIR, ONE>::kWarps * 32, 2)
attn_kernel(const __grid_constant__ AttnParams a, const __grid_constant__ ExpandTable tab) {
  using CF = Cfg<FULL, PAIR, ONE>;
  constexpr int NW = CF::kWarps;
  constexpr int KCH = PAIR ? 64 : 128;  // channels of K and of V per warp
  constexpr int NKT = KCH / 16;         // score k-tiles = output m-tiles per warp
  constexpr int KB = KCH / 8;           // K bytes per token row per lane (c)
  constexpr int VB = KCH / 16;          // V bytes per token row per lane (g)
  constexpr int NU = CF::kNU;
  constexpr int RP = 8 * NT;            // query rows per pass

  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* extra = smem + kLutBytes;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int unit = PAIR ? (w >> 1) : w;
  const int half = PAIR ? (w & 1) : 0;
  const int hb = half * 32;             // first byte of this warp's channel half
  // The CTA's equal share of the flattened (unit, chunk) space, a unit being
  // one (sequence, KV head, row group); a share is at most NCH chunks long,
  // so it touches the units u0 and (perhaps) u0 + 1: segments 0 and 1.
  const int cta = blockIdx.x;
  const int64_t cta_b = a.n_chunks * cta / a.n_cta, cta_e = a.n_chunks * (cta + 1) / a.n_cta;
  const int64_t u0 = cta_b / a.NCH;
  const int part_floats = 2 * RP + RP * kD;
  float* part = a.part + (int64_t)(2 * cta) * part_floats;               // segments 0, 1
  float* flush = a.part + ((int64_t)2 * a.n_cta + cta) * part_floats;    // see below
  // (sequence, KV head, row group) of the two units, packed as
  // (sequence * Hkv + head) * nrg + row group = the unit index itself
  const int rg0 = (int)(u0 % a.nrg), rg1 = (int)((u0 + 1) % a.nrg);
  const int h0 = (int)((u0 / a.nrg) % a.Hkv), h1 = (int)(((u0 + 1) / a.nrg) % a.Hkv);
  const int b0 = (int)(u0 / a.nrg / a.Hkv), b1 = (int)((u0 + 1) / a.nrg / a.Hkv);

  if (smem_u32(smem) != kSmemBase) {  // table loads would read the wrong bytes
    for (int i = tid; i < 2 * part_floats; i += NW * 32) part[i] = __int_as_float(0x7fc00000);
    return;
  }

  for (int i = tid; i < 256 * 32; i += NW * 32) {
    const int row = i >> 5, l = i & 31;
    if constexpr (FULL) {
      reinterpret_cast<float*>(smem + row * 256)[l] = row < 128 ? tab.x[row] : -tab.x[255 - row];
    } else if (l < 16) {
      const int a0 = row & 15, a1 = row >> 4;
      reinterpret_cast<float2*>(smem + row * 256)[l] =
          make_float2(a0 < 8 ? tab.x[16 * a0 + 7] : -tab.x[16 * (15 - a0) + 7],
                      a1 < 8 ? tab.x[16 * a1 + 7] : -tab.x[16 * (15 - a1) + 7]);
    }
  }
  // ---- Q^T fragments (B operand), channel order matching the K bytes
  auto q_frag = [&](int sg, int hf, int kt, int nt, int gg, int cc) -> uint2 {
    const int r = (sg ? rg1 : rg0) * RP + nt * 8 + gg;
    if (r >= a.R || u0 + sg >= a.n_chunks / a.NCH) return make_uint2(0u, 0u);
    const int tq = r / a.G, gq = r % a.G;
    const uint16_t* qrow =
        a.q + ((int64_t)((sg ? b1 : b0) * a.T + tq) * a.Hq + (sg ? h1 : h0) * a.G + gq) * kD;
    uint32_t v[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int beta = hf * 32 + KB * cc + 2 * kt + hh;
      const int lo = 8 * (beta >> 2) + (beta & 3);
      v[hh] = (uint32_t)qrow[lo] | ((uint32_t)qrow[lo + 4] << 16);
    }
    return make_uint2(v[0], v[1]);
  };
  // Q^T fragments of both segments, staged once per CTA:
  // [seg][half][kt][nt][lane] uint2
  {
    constexpr int NH = PAIR ? 2 : 1;
    for (int i = tid; i < 2 * NH * NKT * NT * 32; i += NW * 32) {
      const int ln = i & 31, nt = (i >> 5) % NT, kt = (i >> 5) / NT % NKT;
      const int hf = (i >> 5) / (NT * NKT) % NH, sg = (i >> 5) / (NT * NKT * NH);
      reinterpret_cast<uint2*>(extra)[i] = q_frag(sg, hf, kt, nt, ln >> 2, ln & 3);
    }
  }
  if (tid < 2) {
    // dense: [0..1] block index of page 0 of each segment, (b*NB)*Hkv + h;
    // paged: [0..1] first table row b*NB of each segment, [2..3] its KV head
    int64_t* info = reinterpret_cast<int64_t*>(extra + ExtraLayout<FULL, PAIR, ONE, NT>::kInfo);
    const int64_t row = (int64_t)(tid ? b1 : b0) * a.NB, hh = tid ? h1 : h0;
    if constexpr (PAGED) {
      info[tid] = row;
      info[2 + tid] = hh;
    } else {
      info[tid] = row * a.Hkv + hh;
    }
  }
  __syncthreads();
  const uint32_t lane_off = FULL ? (uint32_t)lane * 4u : (uint32_t)(lane & 15) * 8u;
  const uint32_t sbase = smem_u32(smem);

  // ---- this work unit's contiguous run [ub, ue) of the CTA's share
  const int64_t ub = cta_b + (cta_e - cta_b) * unit / NU;
  const int64_t ue = cta_b + (cta_e - cta_b) * (unit + 1) / NU;
  const int meta_rows = 2 + 2 * a.NC;
  const int tbK = w * CF::kTails, tbV = tbK + CF::kRows * 4;
  // raw rows: piece q (16 bytes, channels 4q..4q+3 of the warp's range) of row
  // r of tensor t; pieces are xor-swizzled by bit 3 so that the build's reads
  // of groups g and g + 4 land in different banks
  auto raw_off = [&](int t, int r, int q) -> uint32_t {
    const int qs = q ^ ((q >> 3) & 1);
    if constexpr (PAIR) {
      const int tail = NW * CF::kTails + (w * 2 + t) * CF::kRawRows * 2 + r * 2 + (qs >> 3);
      return (uint32_t)(tail * 256 + 128 + (qs & 7) * 16);
    } else {
      return (uint32_t)(kLutBytes + ExtraLayout<FULL, PAIR, ONE, NT>::kRaw +
                        ((w * 2 + t) * CF::kRawRows + r) * 512 + qs * 16);
    }
  };
  // Packed block (sequence, page, KV head) of chunk qc of segment sg.
  const int64_t* seg_blk =
      reinterpret_cast<const int64_t*>(extra + ExtraLayout<FULL, PAIR, ONE, NT>::kInfo);
  // Paged streams: a two-entry cache of (table row -> page) per lane.  Chunks
  // walk pages in order, so a table entry is read once per page.  (Prefetching
  // the codes two chunks ahead into L2 was measured and dropped: verification
  // ran 4 % faster dense and 8 % faster paged without it, the draft the same.)
  int64_t c_row0 = -1, c_pg0 = 0, c_row1 = -1, c_pg1 = 0;
  auto page_of = [&](int64_t row) -> int64_t {
    if (row == c_row1) return c_pg1;
    if (row == c_row0) return c_pg0;
    int64_t pg = __ldg(a.bt + row);
    if (pg < 0 || pg >= a.nphys) {
      atomicOr(&g_attn_flags, kFlagBadBlock);
      pg = 0;
    }
    c_row0 = c_row1;
    c_pg0 = c_pg1;
    c_row1 = row;
    c_pg1 = pg;
    return pg;
  };
  auto chunk_blk = [&](int sg, int qc, int& tp) -> int64_t {
    const int t0 = qc * 32;
    const int p = t0 >> a.lgP;
    tp = t0 & (a.P - 1);
    if constexpr (PAGED) {  // the table names the physical page
      return checked_index(page_of(seg_blk[sg] + p) * a.Hkv + seg_blk[2 + sg], a.nphys * a.Hkv,
                           &g_attn_flags);
    } else {
      return checked_index(seg_blk[sg] + p * a.Hkv, (int64_t)a.batch * a.NB * a.Hkv,
                           &g_attn_flags);
    }
  };
  // Asynchronous 16-byte copies of the raw metadata rows of chunk qc of one
  // tensor (t: 0 = K, 1 = V) into the warp's staging rows (the gamma rows
  // only with_gamma): a single warp copies one 512-byte row per instruction,
  // a warp pair's warp two 256-byte rows.
  auto copy_raw = [&](const float* meta, int t, int sg, int qc, bool with_gamma) {
    int tp;
    const int64_t blk = chunk_blk(sg, qc, tp);
    const int cc0 = tp >> a.lgC, cc1 = (tp + 16) >> a.lgC;
    const float* mb = meta + blk * (int64_t)meta_rows * kD + hb * 2;
    constexpr int kPieces = KCH / 4;               // 16-byte pieces of a row
    constexpr int kPerInst = 32 / kPieces;         // rows per copy instruction
    const int q = lane % kPieces;
#pragma unroll
    for (int r0 = 0; r0 < CF::kRawRows; r0 += kPerInst) {
      const int rr = r0 + lane / kPieces;
      if (rr < 2 && !with_gamma) continue;
      const int src = rr == 0 ? 0 : rr == 1 ? 1 : rr == 2 ? 2 + cc0 : rr == 3 ? 2 + a.NC + cc0
                    : rr == 4 ? 2 + cc1 : 2 + a.NC + cc1;
      cp_async16(sbase + raw_off(t, rr, q), mb + src * kD + 4 * q);
    }
  };
  // The (A, B) rows of one tensor from its raw rows (after they have landed):
  // lane (group g, unit h) computes the channel pairs (2h, 2h+4) and
  // (2h+1, 2h+5) of g, for each token half of the chunk.
  auto build_ab = [&](int t, int tb) {
    constexpr int kUnits = (KCH / 8) * 2;          // 32 (single warp) or 16 (pair)
    constexpr int kJ = ONE ? 1 : 2;
    const int u = lane % kUnits, jl = lane / kUnits;
    const int gl = u >> 1, h = u & 1;
    const int grp = hb / 4 + gl;
#pragma unroll
    for (int j0 = 0; j0 < kJ; j0 += 32 / kUnits) {
      const int j = j0 + jl;
      if (j >= kJ) continue;
      auto rd = [&](int r, int q) -> f2 {
        return *reinterpret_cast<const float2*>(smem + raw_off(t, r, q) + 8 * h);
      };
      const f2 e = make_float2(kEps, kEps);
      const f2 gm_lo = rd(0, 2 * gl), gm_hi = rd(0, 2 * gl + 1);
      const f2 gs_lo = add2(rd(1, 2 * gl), e), gs_hi = add2(rd(1, 2 * gl + 1), e);
      const f2 mu_lo = rd(2 + 2 * j, 2 * gl), mu_hi = rd(2 + 2 * j, 2 * gl + 1);
      const f2 sg_lo = add2(rd(3 + 2 * j, 2 * gl), e), sg_hi = add2(rd(3 + 2 * j, 2 * gl + 1), e);
      const f2 A_lo = mul2(sg_lo, gs_lo), A_hi = mul2(sg_hi, gs_hi);
      const f2 B_lo = fma2(mu_lo, gs_lo, gm_lo), B_hi = fma2(mu_hi, gs_hi, gm_hi);
      const uint32_t ub = unit_off(tb, 2 * j, grp, h);
      *reinterpret_cast<float4*>(smem + ub) = make_float4(A_lo.x, A_hi.x, A_lo.y, A_hi.y);
      *reinterpret_cast<float4*>(smem + ub + kRowStride) =
          make_float4(B_lo.x, B_hi.x, B_lo.y, B_hi.y);
    }
  };

  float m_run[NT][2], l_run[NT][2];
  float o[NKT][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int i = 0; i < NKT; ++i) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
  }

  Bytes<KB> kA[4], kR[4];
  auto load_k = [&](int sg, int qc) {
    int tp;
    const int64_t blk = chunk_blk(sg, qc, tp);
    const int64_t off = (blk * a.P + tp) * (kD / 2) + hb + KB * c;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int row = 16 * (jj >> 1) + g + 8 * (jj & 1);
      kA[jj].load(a.ka + off + row * 64);
      if constexpr (FULL) kR[jj].load(a.kr + off + row * 64);
    }
  };
  // segment and chunk (within its unit) of the run's current chunk
  const int sg_start = (int)(ub / a.NCH - u0);
  int sg = sg_start;
  int qc = (int)(ub - (u0 + sg) * a.NCH);
  if (ub < ue) {
    copy_raw(a.km, 0, sg, qc, true);
    cp_commit();
    copy_raw(a.vm, 1, sg, qc, true);
    cp_commit();
    load_k(sg, qc);
  }

  for (int left = (int)(ue - ub); left > 0; --left) {
    int tp;
    const int64_t blk = chunk_blk(sg, qc, tp);
    const int64_t code_off = (blk * a.P + tp) * (kD / 2);
    const bool has_next = left > 1;
    // the next chunk (recomputed where used, to keep registers free)
    auto cross = [&] { return qc + 1 == a.NCH; };  // it starts the next unit
    auto sg_n = [&] { return cross() ? sg + 1 : sg; };
    auto qc_n = [&] { return cross() ? 0 : qc + 1; };
    auto next_gamma = [&] { return cross() || ((qc + 1) * 32 >> a.lgP) != (qc * 32 >> a.lgP); };

    // ---- V codes of this chunk (used after the scores)
    Bytes<VB> vA[8], vR[8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int kk = ii & 3;
      const int row = 16 * (ii >> 2) + 2 * c + (kk & 1) + 8 * (kk >> 1);
      vA[ii].load(a.va + code_off + row * 64 + hb + VB * g);
      if constexpr (FULL) vR[ii].load(a.vr + code_off + row * 64 + hb + VB * g);
    }
    // ---- scores: S^T for m-tiles j = 0, 1 (tokens 16j .. 16j+15)
    cp_wait<1>();  // raw rows of K for this chunk have landed
    __syncwarp();
    build_ab(0, tbK);
    __syncwarp();  // (A, B) of K ready; its raw rows are free for the next chunk
    if (has_next) copy_raw(a.km, 0, sg_n(), qc_n(), next_gamma());
    cp_commit();
    float s[2][NT][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[j][nt][0] = s[j][nt][1] = s[j][nt][2] = s[j][nt][3] = 0.f;
#pragma unroll
    for (int gi = 0; gi < KB / 4; ++gi) {      // channel groups of this lane (K)
      const int grp = (hb + KB * c) / 4 + gi;
      const uint32_t gb = unit_off(tbK, 0, grp, 0);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {         // k-tile 2gi+kk: byte positions 2kk, 2kk+1
        const int kt = 2 * gi + kk;
        uint32_t qb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 v = reinterpret_cast<const uint2*>(
              extra)[((((sg * (PAIR ? 2 : 1) + half) * NKT + kt) * NT + nt) * 32 + lane)];
          qb[nt][0] = v.x;
          qb[nt][1] = v.y;
        }
        Half kc;
        if constexpr (ONE) load_half(kc, smem, gb, 0, kk);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if constexpr (!ONE) load_half(kc, smem, gb, j, kk);
          uint32_t af[4];
#pragma unroll
          for (int i = 0; i < 2; ++i) {        // row g (i=0) / g+8 (i=1)
            const uint32_t wa = kA[2 * j + i].w[gi];
            const uint32_t wr = FULL ? kR[2 * j + i].w[gi] : 0u;
            if (kk == 0) {
              af[i] = dequant_pair<FULL, 0>(wa, wr, lane_off, kc);
              af[i + 2] = dequant_pair<FULL, 1>(wa, wr, lane_off, kc);
            } else {
              af[i] = dequant_pair<FULL, 2>(wa, wr, lane_off, kc);
              af[i + 2] = dequant_pair<FULL, 3>(wa, wr, lane_off, kc);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16(s[j][nt], af, qb[nt][0], qb[nt][1]);
        }
      }
    }
    __syncwarp();  // every lane is done with this chunk's K constants and codes
    if (has_next) load_k(sg_n(), qc_n());

    // ---- the warp's own n-tiles: all NT of them for a single warp; for a
    // warp pair, half of them each (tiles half*OWN .. +OWN-1), so that the
    // two warps split the softmax.  Their full scores: the pair swaps the
    // partial scores of the partner's tiles (a reduce-scatter).
    constexpr int OWN = PAIR ? NT / 2 : NT;
    float sc[2][OWN][4];
    if constexpr (PAIR) {
      float* xs = reinterpret_cast<float*>(extra + ExtraLayout<FULL, PAIR, ONE, NT>::kQ);
      float* mine = xs + (unit * 2 + half) * (2 * OWN * 32 * 4);
      const float* other = xs + (unit * 2 + (half ^ 1)) * (2 * OWN * 32 * 4);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q) {            // the partner's tile (1-half)*OWN + q
          float4 v;
          v.x = half ? s[j][q][0] : s[j][OWN + q][0];
          v.y = half ? s[j][q][1] : s[j][OWN + q][1];
          v.z = half ? s[j][q][2] : s[j][OWN + q][2];
          v.w = half ? s[j][q][3] : s[j][OWN + q][3];
          *reinterpret_cast<float4*>(mine + ((j * OWN + q) * 32 + lane) * 4) = v;
        }
      asm volatile("bar.sync %0, 64;" :: "r"(1 + unit) : "memory");
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(other + ((j * OWN + q) * 32 + lane) * 4);
          sc[j][q][0] = (half ? s[j][OWN + q][0] : s[j][q][0]) + v.x;
          sc[j][q][1] = (half ? s[j][OWN + q][1] : s[j][q][1]) + v.y;
          sc[j][q][2] = (half ? s[j][OWN + q][2] : s[j][q][2]) + v.z;
          sc[j][q][3] = (half ? s[j][OWN + q][3] : s[j][q][3]) + v.w;
        }
    } else {
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[j][q][e] = s[j][q][e];
    }

    // ---- online softmax (log2 domain) of the own tiles; rows tile*8 + 2c,
    // tile*8 + 2c + 1.  m_run / l_run hold the own tiles' rows.  al: the
    // factor that rescales the output of each own row (1 if its max holds).
    uint32_t ph[2][OWN][2], pl[2][OWN][2];
    float al[OWN][2];
    bool rescale = false;
#pragma unroll
    for (int q = 0; q < OWN; ++q) {
      float cmax0 = fmaxf(fmaxf(sc[0][q][0], sc[0][q][2]), fmaxf(sc[1][q][0], sc[1][q][2]));
      float cmax1 = fmaxf(fmaxf(sc[0][q][1], sc[0][q][3]), fmaxf(sc[1][q][1], sc[1][q][3]));
#pragma unroll
      for (int x = 4; x <= 16; x <<= 1) {
        cmax0 = fmaxf(cmax0, __shfl_xor_sync(kFull, cmax0, x));
        cmax1 = fmaxf(cmax1, __shfl_xor_sync(kFull, cmax1, x));
      }
      const float mn0 = fmaxf(m_run[q][0], cmax0 * a.scale_log2);
      const float mn1 = fmaxf(m_run[q][1], cmax1 * a.scale_log2);
      al[q][0] = al[q][1] = 1.0f;
      if (mn0 != m_run[q][0] || mn1 != m_run[q][1]) {
        al[q][0] = ex2(m_run[q][0] - mn0);
        al[q][1] = ex2(m_run[q][1] - mn1);
        l_run[q][0] *= al[q][0];
        l_run[q][1] *= al[q][1];
        m_run[q][0] = mn0;
        m_run[q][1] = mn1;
        rescale = true;
        if constexpr (!PAIR) {                 // own tiles are all tiles: rescale here
#pragma unroll
          for (int mt = 0; mt < NKT; ++mt) {
            o[mt][q][0] *= al[q][0]; o[mt][q][1] *= al[q][1];
            o[mt][q][2] *= al[q][0]; o[mt][q][3] *= al[q][1];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float p0 = ex2(fmaf(sc[j][q][0], a.scale_log2, -mn0));
        const float p1 = ex2(fmaf(sc[j][q][1], a.scale_log2, -mn1));
        const float p2 = ex2(fmaf(sc[j][q][2], a.scale_log2, -mn0));
        const float p3 = ex2(fmaf(sc[j][q][3], a.scale_log2, -mn1));
        l_run[q][0] += p0 + p2;
        l_run[q][1] += p1 + p3;
        const uint32_t top = f2_to_bf2(p0, p1), bot = f2_to_bf2(p2, p3);
        const f2 th = bf2_to_f2(top), bh = bf2_to_f2(bot);
        ph[j][q][0] = movtrans(top);
        ph[j][q][1] = movtrans(bot);
        pl[j][q][0] = movtrans(f2_to_bf2(p0 - th.x, p1 - th.y));
        pl[j][q][1] = movtrans(f2_to_bf2(p2 - bh.x, p3 - bh.y));
      }
    }

    // ---- P^T operands (hi, lo) and row factors of all NT tiles
    uint32_t pb_hi[2][NT][2], pb_lo[2][NT][2];
    float alf[NT][2];
    if constexpr (PAIR) {
      // swap the own tiles' P operands and factors with the partner
      uint32_t* pxs = reinterpret_cast<uint32_t*>(
          extra + ExtraLayout<FULL, PAIR, ONE, NT>::kQ + (size_t)NU * 2 * (2 * OWN * 32 * 16));
      constexpr int PW = 2 * 2 * OWN * 2 + 2 * OWN;  // words per lane: P hi, lo; factors
      uint32_t* mine = pxs + (unit * 2 + half) * (PW * 32);
      const uint32_t* other = pxs + (unit * 2 + (half ^ 1)) * (PW * 32);
      rescale = __any_sync(kFull, rescale);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            mine[(((j * OWN + q) * 2 + e) * 2 + 0) * 32 + lane] = ph[j][q][e];
            mine[(((j * OWN + q) * 2 + e) * 2 + 1) * 32 + lane] = pl[j][q][e];
          }
#pragma unroll
      for (int q = 0; q < OWN; ++q)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          mine[(2 * 2 * OWN * 2 + q * 2 + e) * 32 + lane] = __float_as_uint(al[q][e]);
      // the partner's vote travels with its factors: a rescale anywhere
      // in the pair shows as a factor other than 1
      asm volatile("bar.sync %0, 64;" :: "r"(1 + unit) : "memory");
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t oh = other[(((j * OWN + q) * 2 + e) * 2 + 0) * 32 + lane];
            const uint32_t ol = other[(((j * OWN + q) * 2 + e) * 2 + 1) * 32 + lane];
            pb_hi[j][q][e] = half ? oh : ph[j][q][e];
            pb_lo[j][q][e] = half ? ol : pl[j][q][e];
            pb_hi[j][OWN + q][e] = half ? ph[j][q][e] : oh;
            pb_lo[j][OWN + q][e] = half ? pl[j][q][e] : ol;
          }
      bool other_rescale = false;
#pragma unroll
      for (int q = 0; q < OWN; ++q)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float of = __uint_as_float(other[(2 * 2 * OWN * 2 + q * 2 + e) * 32 + lane]);
          other_rescale |= of != 1.0f;
          alf[q][e] = half ? of : al[q][e];
          alf[OWN + q][e] = half ? al[q][e] : of;
        }
      rescale = rescale || __any_sync(kFull, other_rescale);
    } else {
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < OWN; ++q)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pb_hi[j][q][e] = ph[j][q][e];
            pb_lo[j][q][e] = pl[j][q][e];
          }
    }
    if (PAIR && rescale) {
#pragma unroll
      for (int mt = 0; mt < NKT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[mt][nt][0] *= alf[nt][0]; o[mt][nt][1] *= alf[nt][1];
          o[mt][nt][2] *= alf[nt][0]; o[mt][nt][3] *= alf[nt][1];
        }
    }

    // ---- output: O^T += V^T P^T over this warp's V m-tiles (byte VB*g + mt)
    cp_wait<1>();  // raw rows of V for this chunk have landed
    __syncwarp();
    build_ab(1, tbV);
    __syncwarp();  // (A, B) of V ready; its raw rows are free for the next chunk
    if (has_next) copy_raw(a.vm, 1, sg_n(), qc_n(), next_gamma());
    cp_commit();
#pragma unroll
    for (int gi = 0; gi < VB / 4; ++gi) {
      const int grp = (hb + VB * g) / 4 + gi;
      const uint32_t gb = unit_off(tbV, 0, grp, 0);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {         // byte positions 2hh, 2hh+1
        Half vc;
        if constexpr (ONE) load_half(vc, smem, gb, 0, hh);
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
          if constexpr (!ONE) load_half(vc, smem, gb, jt, hh);
#pragma unroll
          for (int kq = 0; kq < 2; ++kq) {
            const int kk = 2 * hh + kq, mt = 4 * gi + kk;
            uint32_t W[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {   // tokens 2c, 2c+1, 2c+8, 2c+9
              const uint32_t wa = vA[4 * jt + q4].w[gi];
              const uint32_t wr = FULL ? vR[4 * jt + q4].w[gi] : 0u;
              W[q4] = kk == 0 ? dequant_pair<FULL, 0>(wa, wr, lane_off, vc)
                    : kk == 1 ? dequant_pair<FULL, 1>(wa, wr, lane_off, vc)
                    : kk == 2 ? dequant_pair<FULL, 2>(wa, wr, lane_off, vc)
                              : dequant_pair<FULL, 3>(wa, wr, lane_off, vc);
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
        }
      }
    }
    __syncwarp();  // every lane is done with this chunk's V constants

    if (cross() && has_next) {
      // The run leaves unit u0 (only one work unit of a CTA can): park its
      // state for unit u0 in the CTA's flush record, start afresh on u0 + 1.
      float lr[OWN][2];
#pragma unroll
      for (int q = 0; q < OWN; ++q)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = l_run[q][e];
#pragma unroll
          for (int x = 4; x <= 16; x <<= 1) v += __shfl_xor_sync(kFull, v, x);
          lr[q][e] = v;
        }
      if (g == 0) {                            // the own tiles' rows
#pragma unroll
        for (int q = 0; q < OWN; ++q)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = (half * OWN + q) * 8 + 2 * c + e;
            flush[row] = m_run[q][e];
            flush[RP + row] = lr[q][e];
          }
      }
#pragma unroll
      for (int mt = 0; mt < NKT; ++mt) {
        const int beta = hb + VB * g + mt;
        const int ch_lo = 8 * (beta >> 2) + (beta & 3), ch_hi = ch_lo + 4;
        float* fo = flush + 2 * RP;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          fo[(nt * 8 + 2 * c) * kD + ch_lo] = o[mt][nt][0];
          fo[(nt * 8 + 2 * c + 1) * kD + ch_lo] = o[mt][nt][1];
          fo[(nt * 8 + 2 * c) * kD + ch_hi] = o[mt][nt][2];
          fo[(nt * 8 + 2 * c + 1) * kD + ch_hi] = o[mt][nt][3];
          o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < OWN; ++q) {
        m_run[q][0] = m_run[q][1] = -INFINITY;
        l_run[q][0] = l_run[q][1] = 0.f;
      }
    }
    if (has_next) {
      const int sgn = sg_n(), qcn = qc_n();
      sg = sgn;
      qc = qcn;
    }
  }
  cp_wait<0>();

  // ---- merge the work units of the CTA per segment, write its partials
  constexpr int OWNF = PAIR ? NT / 2 : NT;   // own tiles of a warp (see the loop)
#pragma unroll
  for (int q = 0; q < OWNF; ++q)
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      l_run[q][0] += __shfl_xor_sync(kFull, l_run[q][0], x);
      l_run[q][1] += __shfl_xor_sync(kFull, l_run[q][1], x);
    }
  __syncthreads();  // every warp is done with Q, the exchange and the scratch
  float* sm_m = reinterpret_cast<float*>(extra);      // [NU][RP]
  float* sm_l = sm_m + NU * RP;                        // [NU][RP]
  float* sm_o = sm_l + NU * RP;                        // [NU][RP][128]
  int* sm_tag = reinterpret_cast<int*>(sm_o + NU * RP * kD);  // [NU] segment of the state
  int* sm_fl = sm_tag + NU;                                    // [NU] parked a state
  if (g == 0) {
#pragma unroll
    for (int q = 0; q < OWNF; ++q) {
      const int row = (half * OWNF + q) * 8 + 2 * c;
      sm_m[unit * RP + row] = m_run[q][0];
      sm_m[unit * RP + row + 1] = m_run[q][1];
      sm_l[unit * RP + row] = l_run[q][0];
      sm_l[unit * RP + row + 1] = l_run[q][1];
    }
    if (c == 0 && half == 0) {
      sm_tag[unit] = sg;
      sm_fl[unit] = (ub < ue && sg != sg_start) ? 1 : 0;  // crossed, so parked a state
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
  __syncthreads();  // (also orders the flush record's global writes before its reads)
  bool parked = false;
#pragma unroll
  for (int u = 0; u < NU; ++u) parked |= sm_fl[u] != 0;
  const int nseg = (int)((cta_e - 1) / a.NCH - u0) + 1;
  for (int i = tid; i < nseg * RP * kD; i += NW * 32) {
    const int sgm = i / (RP * kD), r = (i / kD) % RP, d = i % kD;
    const bool use_flush = sgm == 0 && parked;
    float M = use_flush ? flush[r] : -INFINITY;
#pragma unroll
    for (int u = 0; u < NU; ++u)
      if (sm_tag[u] == sgm) M = fmaxf(M, sm_m[u * RP + r]);
    float acc = 0.f, den = 0.f;
    if (use_flush && flush[r] != -INFINITY) {
      const float f = exp2f(flush[r] - M);
      acc = f * flush[2 * RP + r * kD + d];
      den = f * flush[RP + r];
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const float mu_ = sm_m[u * RP + r];
      if (sm_tag[u] != sgm || mu_ == -INFINITY) continue;
      const float f = exp2f(mu_ - M);
      acc += f * sm_o[(u * RP + r) * kD + d];
      den += f * sm_l[u * RP + r];
    }
    if constexpr (DIRECT) {
      // the unit's whole softmax: out = o / l (what the combine computes
      // from a single partial).  One unit per CTA: it is u0, segment 0.
      const int row = rg0 * RP + r;
      if (row < a.R) {
        const int tq = row / a.G, gq = row % a.G;
        a.out[((int64_t)(b0 * a.T + tq) * a.Hq + h0 * a.G + gq) * kD + d] = acc / den;
      }
    } else {
      float* ps = part + sgm * part_floats;
      ps[2 * RP + r * kD + d] = acc;
      if (d == 0) {
        ps[r] = M;
        ps[RP + r] = den;
      }
    }
  }
  // the split combine may launch now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Merge the partials of one query row of one unit (sequence, KV head, row
// group): the CTAs whose shares touch the unit, each through the partial of
// the matching segment.  One warp per (unit, row), four channels a lane; the
// splits merge online (running max, rescaled sums), kCombineBatch of them per
// round of independent loads:
// out = sum e^(m_s-M) o_s / sum e^(m_s-M) l_s, written to out[b][t][hq][:].
// With the draft tokens' own keys and values, query token t also attends to
// draft tokens 0..t ("Lynx", Mechanism 3, single parallel verification
// pass): their scores join the same softmax.
__device__ __forceinline__ float bf16_to_f32(uint16_t x) {
  return __uint_as_float((uint32_t)x << 16);
}
constexpr int kCombineWarps = 4;
constexpr int kCombineBatch = 8;
__global__ void __launch_bounds__(32 * kCombineWarps)
attn_combine(const __grid_constant__ AttnParams a, int RP) {
  // launched as a programmatic dependent of the attention kernel: wait until
  // that grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t z = blockIdx.x;  // (b * Hkv + h) * nrg + rg
  const int r = blockIdx.y * kCombineWarps + (threadIdx.x >> 5);
  if (r >= RP) return;
  const int rg = (int)(z % a.nrg), bh = (int)(z / a.nrg), h = bh % a.Hkv, b = bh / a.Hkv;
  const int row = rg * RP + r;
  if (row >= a.R) return;
  const int tq = row / a.G, gq = row % a.G;
  const int part_floats = 2 * RP + RP * kD;
  // CTA holding flattened chunk x: floor(((x + 1) n_cta - 1) / n_chunks)
  const int64_t first = z * a.NCH, last = first + a.NCH - 1;
  const int k0 = (int)(((first + 1) * a.n_cta - 1) / a.n_chunks);
  const int k1 = (int)(((last + 1) * a.n_cta - 1) / a.n_chunks);
  float M = -INFINITY, Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  auto merge = [&](float m, float l, float4 o) {
    if (m == -INFINITY) return;                 // a share with no chunk of this unit
    const float Mn = fmaxf(M, m);
    const float fo = exp2f(M - Mn), fn = exp2f(m - Mn);  // exp2(-inf) = 0 on the first
    O.x = O.x * fo + fn * o.x; O.y = O.y * fo + fn * o.y;
    O.z = O.z * fo + fn * o.z; O.w = O.w * fo + fn * o.w;
    Lsum = Lsum * fo + fn * l;
    M = Mn;
  };
  for (int kb = k0; kb <= k1; kb += kCombineBatch) {
    float mv[kCombineBatch], lv[kCombineBatch];
    float4 ov[kCombineBatch];
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const int k = kb + i;
      if (k <= k1) {
        const int64_t seg = z - (a.n_chunks * k / a.n_cta) / a.NCH;
        const float* ps = a.part + checked_index(2 * k + seg, 2 * (int64_t)a.n_cta,
                                                 &g_attn_flags) * part_floats;
        mv[i] = ps[r];
        lv[i] = ps[RP + r];
        ov[i] = *reinterpret_cast<const float4*>(ps + 2 * RP + r * kD + 4 * lane);
      } else {
        mv[i] = -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) merge(mv[i], lv[i], ov[i]);
  }
  if (a.kt) {
    const uint2 qw = *reinterpret_cast<const uint2*>(
        a.q + ((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD + 4 * lane);
    const float q0 = bf16_to_f32((uint16_t)qw.x), q1 = bf16_to_f32((uint16_t)(qw.x >> 16));
    const float q2 = bf16_to_f32((uint16_t)qw.y), q3 = bf16_to_f32((uint16_t)(qw.y >> 16));
    for (int j = 0; j <= tq; ++j) {
      const int64_t off = ((int64_t)(b * a.T + j) * a.Hkv + h) * kD + 4 * lane;
      const uint2 kw = *reinterpret_cast<const uint2*>(a.kt + off);
      float prod = q0 * bf16_to_f32((uint16_t)kw.x) + q1 * bf16_to_f32((uint16_t)(kw.x >> 16)) +
                   q2 * bf16_to_f32((uint16_t)kw.y) + q3 * bf16_to_f32((uint16_t)(kw.y >> 16));
#pragma unroll
      for (int o = 16; o; o >>= 1) prod += __shfl_xor_sync(kFull, prod, o);
      const uint2 vw = *reinterpret_cast<const uint2*>(a.vt + off);
      merge(prod * a.scale_log2, 1.0f,
            make_float4(bf16_to_f32((uint16_t)vw.x), bf16_to_f32((uint16_t)(vw.x >> 16)),
                        bf16_to_f32((uint16_t)vw.y), bf16_to_f32((uint16_t)(vw.y >> 16))));
    }
  }
  *reinterpret_cast<float4*>(a.out + ((int64_t)(b * a.T + tq) * a.Hq + h * a.G + gq) * kD +
                             4 * lane) =
      make_float4(O.x / Lsum, O.y / Lsum, O.z / Lsum, O.w / Lsum);
}

// ------------------------------------------------------------------ host

// Query rows per pass: one n-tile (8 rows) for small groups, else a warp
// pair over four n-tiles (32 rows).
static int rows_per_pass(int R) { return R <= 8 ? 8 : 32; }
static int row_groups(int R) { const int rp = rows_per_pass(R); return (R + rp - 1) / rp; }

// CTAs of the attention grid.  Every shape runs two CTAs per SM, so `sms`
// SMs hold 2 sms at once: one wave of equal shares of the flattened
// (unit, chunk) space, with at least 2 chunks per work unit (8 of them per
// CTA up to 8 query rows, 2 warp pairs above), and at least one CTA per unit
// so that a share never exceeds one unit's chunks (several waves when there
// are more units than that).  The launch takes the device's SM count, capped
// at kMaxWaveSMs; the workspace is sized for that cap, so its size is a pure
// function of the shapes and holds the partials on any device.
constexpr int kMaxWaveSMs = 256;
static int ctas_for(int batch, int Hkv, int nrg, int64_t NCH, int R, int sms) {
  const int64_t units = (int64_t)batch * Hkv * nrg;
  const int64_t n_chunks = units * NCH;
  const int64_t nu = R <= 8 ? 8 : 2;
  int64_t n = (int64_t)(sms < kMaxWaveSMs ? sms : kMaxWaveSMs) * 2;
  if (n > n_chunks / (2 * nu)) n = n_chunks / (2 * nu);
  if (n < units) n = units;
  return (int)n;
}

// Workspace: two partials per CTA (its segments) and one parked state per
// CTA (a work unit's state for the first unit when its run crosses into the
// second), for the largest grid any device can launch.
size_t attn_workspace_bytes(int batch, int T, int H_q, int H_kv, int64_t L) {
  const int R = (H_q / H_kv) * T;
  const int RP = rows_per_pass(R), nrg = row_groups(R);
  const int n = ctas_for(batch, H_kv, nrg, L / 32, R, kMaxWaveSMs);
  return (size_t)3 * n * (2 * RP + RP * kD) * sizeof(float);
}

template <bool FULL, int NT, bool PAIR, bool ONE, bool PAGED, bool DIRECT>
static cudaError_t run_attn(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  auto fn = attn_kernel<FULL, NT, PAIR, ONE, PAGED, DIRECT>;
  constexpr size_t smem = attn_smem_bytes<FULL, PAIR, ONE, NT>();
  constexpr int threads = Cfg<FULL, PAIR, ONE>::kWarps * 32;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    // The table loads assume dynamic shared memory starts right after the
    // block's reserved shared memory at kSmemBase.
    int reserved = -1;
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    if (reserved != (int)kSmemBase) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  fn<<<(unsigned)prm.n_cta, threads, smem, stream>>>(prm, tab);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (DIRECT) return cudaSuccess;   // the kernel wrote the output rows
  return launch_attn_combine(prm, 8 * NT, stream);
}

cudaError_t launch_attn_combine(const AttnParams& prm, int RP, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(prm.batch * prm.Hkv * prm.nrg),
                     (unsigned)((RP + kCombineWarps - 1) / kCombineWarps));
  cfg.blockDim = dim3(32 * kCombineWarps);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_combine, prm, RP);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FULL, int NT, bool PAIR, bool DIRECT>
static cudaError_t run_attn_d(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  if (prm.bt)
    return prm.C >= 32 ? run_attn<FULL, NT, PAIR, true, true, DIRECT>(prm, tab, stream)
                       : run_attn<FULL, NT, PAIR, false, true, DIRECT>(prm, tab, stream);
  return prm.C >= 32 ? run_attn<FULL, NT, PAIR, true, false, DIRECT>(prm, tab, stream)
                     : run_attn<FULL, NT, PAIR, false, false, DIRECT>(prm, tab, stream);
}

// One CTA per work unit (short sequences) and no draft-token tail: the single
// shape writes its output rows itself and no combine is launched.
template <bool FULL, int NT, bool PAIR>
static cudaError_t run_attn_c(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  if constexpr (!PAIR) {
    if (prm.n_cta * prm.NCH == prm.n_chunks && prm.kt == nullptr)
      return run_attn_d<FULL, NT, PAIR, true>(prm, tab, stream);
  }
  return run_attn_d<FULL, NT, PAIR, false>(prm, tab, stream);
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
  prm.bt = x.paging.table;
  prm.nphys = x.paging.nphys;
  prm.kt = static_cast<const uint16_t*>(x.k_tail);
  prm.vt = static_cast<const uint16_t*>(x.v_tail);
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
  prm.n_chunks = (int64_t)x.batch * prm.Hkv * prm.nrg * prm.NCH;
  prm.n_cta = ctas_for(x.batch, prm.Hkv, prm.nrg, prm.NCH, prm.R, sm_count());
  prm.P = x.s.page;
  prm.C = x.s.C;
  prm.NC = x.s.NC();
  prm.lgP = __builtin_ctz((unsigned)x.s.page);
  prm.lgC = __builtin_ctz((unsigned)x.s.C);
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  const bool small = prm.R <= 8;
  if (x.full && !small && x.s.L % 128 == 0) {
    // the verification pass: tensor-memory kernel over tiles of 128 tokens
    prm.NCH = x.s.L / 128;
    prm.n_chunks = (int64_t)x.batch * prm.Hkv * prm.nrg * prm.NCH;
    prm.n_cta = attn_tc_ctas(x.batch, prm.Hkv, prm.nrg, prm.NCH, sm_count());
    return launch_attn_tc(prm, tab, stream);
  }
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

// Unique id of the calling thread's current CUDA context (cuCtxGetId ids are
// never reused within a process), through the runtime's driver entry points
// (the library does not link the driver library); 0 if unavailable.
static unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static const auto fns = [] {
    void* cur = nullptr;
    void* id = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess || q1 != cudaDriverEntryPointSuccess)
      cur = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess || q2 != cudaDriverEntryPointSuccess)
      id = nullptr;
    return std::make_pair(reinterpret_cast<GetCurrentFn>(cur), reinterpret_cast<GetIdFn>(id));
  }();
  if (!fns.first || !fns.second) return 0;
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx || fns.second(ctx, &v) != CUDA_SUCCESS) return 0;
  return v;
}

// Device address of g_attn_scratch for the current device: looked up with
// cudaGetSymbolAddress (that device current) on the first call and again
// whenever the device's context has changed since (after cudaDeviceReset the
// old address belongs to a destroyed context), else taken from the cache.
static cudaError_t noalloc_scratch(void** ptr) {
  constexpr int kMaxDev = 64;
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  static Entry cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].addr || ctx == 0 || cache[dev].ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    // the lookup initialises the context if it was not yet: record its id
    cache[dev] = Entry{ctx != 0 ? ctx : current_context_id(), p};
  }
  *ptr = cache[dev].addr;
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
