// encode.cu -- Algorithm 1 of "Lynx: Progressive Speculative KV Cache Transfer
// for Disaggregated LLM Inference" (technical review, Mechanism 1, Stages 1-4)
// as one persistent sm_103a kernel.
//
// Work unit: W channels of one page block (`page` tokens of one KV head; the
// statistics are per channel, so a block splits into 128/W independent units).
// A 2D TMA load stages the unit's BF16 tile (page x 2W bytes, rows strided by
// H*256 bytes in HBM) in shared memory; the next one or two tiles are in
// flight per CTA while the CTA computes on the current one.
//
// Thread layout: a warp owns a slice of a unit, one chunk of C tokens x
// 2048/C channels, so a chunk's statistics never leave the warp.  In a warp,
// lane = k * CG + cg with TL = C/8 token-lane slots k and CG = 256/C channel
// groups of 8 channels (16 bytes of a BF16 row, 4 bytes of each packed row);
// register m holds chunk token i = TL*m + tl(k).  The chunk mean's
// pairwise-halving sum (v[i] += v[i+h], h = C/2 .. 1) then reduces the
// register index first (the top bits of i), then the token lanes by shuffles
// with h = TL/2 .. 1: exactly the order the oracle uses.  The token-lane
// levels are a reduce-scatter: each level halves the channels a lane keeps,
// so every lane finishes the statistics of 8/TL channels (one when TL >= 8)
// and hands them to the other lanes through a small per-warp exchange in
// shared memory.  The per-chunk minima and maxima reduce the same way.  Only
// the page minimum and maximum cross warps (one block barrier per unit).
//
// Arithmetic, each step one IEEE binary32 rounding (no contraction):
//   gmin = min x (a zero minimum as -0), gmax = max x, gs = gmax - gmin,
//   rg = rn(1/(gs + eps)), n = (x - gmin) * rg,
//   mu = tree_sum(n) * (1/C), d = n - mu, sg = max|d|, rs = rn(1/(sg + eps)),
//   a = |d * rs|, S = sign(d) (+1 at zero).
// Stage 3 (Eq. 7) is decided against the float64 thresholds of the host:
// a fast MUFU log2 path gives the code unless its value lies within
// kAmbiguityK * 2^-16 of a rounding boundary; then the threshold decides.
// Stage 4 (Eq. 9 at 8 bits): code8 = S > 0 ? I : 255 - I; Anchor = code8 >> 4,
// Residual = code8 & 15, packed two channels (8G+k, 8G+k+4) per byte.
#include "common.cuh"
#include "internal.h"

namespace lynx {

// Set by a kernel whose bounded wait on a TMA stage gave up (the kernel then
// returns early).  Read through read_wait_timeout(); never reset.
__device__ unsigned int g_wait_timeout = 0;

cudaError_t read_wait_timeout(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_wait_timeout, sizeof(unsigned int));
}

// s = floor((Y' + 1/2) * 65536 + K) + 2^23 with Y' = lg * c16 / 65536.
// Byte 2 of the bits is the code (Y' + 1/2 < 128), the low 16 bits locate
// the value relative to the rounding boundary.
constexpr float kC0 = 8388608.0f + 32768.0f + (float)kAmbiguityK;

// Two values at once: per lane the same roundings as t = rn(alpha*a + 1),
// s = rm(lg2(t)*c16 + kC0), issued as packed pairs.
__device__ __forceinline__ void compand_fast2(f2 a, f2 alpha2, f2 c16_2, uint32_t& b0,
                                              uint32_t& b1) {
  const f2 t = __ffma2_rn(alpha2, a, make_float2(1.0f, 1.0f));
  const f2 l = make_float2(lg2_approx(t.x), lg2_approx(t.y));
  const f2 s = __ffma2_rd(l, c16_2, make_float2(kC0, kC0));
  b0 = __float_as_uint(s.x);
  b1 = __float_as_uint(s.y);
}
__device__ __forceinline__ bool compand_ambiguous(uint32_t bits) {
  return (bits & 0xffffu) < 2u * kAmbiguityK;
}
// Exact code from the thresholds, for a value flagged ambiguous.
__device__ __forceinline__ uint32_t compand_exact(uint32_t bits, float a, const float* thr) {
  int I = (int)((bits >> 16) & 0xffu);
  int b = I > 0 ? I - 1 : 0;
  return (uint32_t)(b + (a >= thr[b] ? 1 : 0));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Channel width of a work unit.  The statistics are per channel, so a page
// block splits into independent ranges of W channels.  A warp covers C
// tokens x 2048/C channels (TL = C/8 token lanes x 8 registers, CG = 256/C
// groups of 8 channels), so W >= 2048/C; below that bound W is chosen so that
// a tile (P x W BF16) is 32 KiB where possible: three stages of it and the
// statistics of two CTAs fit one SM.
template <int P, int C>
constexpr int enc_width() {
  constexpr int lo = 2048 / C;
  constexpr int want = P <= 128 ? 128 : 16384 / P;
  return lo > want ? (lo > 128 ? 128 : lo) : want;
}

template <int P, int C>
struct EncGeom {
  static constexpr int kW = enc_width<P, C>();
  static constexpr int kUnits = kD / kW;        // work units per page block
  static constexpr int kNC = P / C;
  static constexpr int kTL = C / 8;             // token lanes
  static constexpr int kCG = 256 / C;           // channel groups of 8 per warp
  static constexpr int kSlices = P * kW / 2048; // (chunk, channel range) slices of a unit
  static constexpr int kSlicesPerChunk = kW * C / 2048;
  static constexpr int kWarps = kSlices < 8 ? kSlices : 8;
  static constexpr int kSlicesPerWarp = kSlices / kWarps;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kRowBytes = kW * 2;
  static constexpr int kTileBytes = P * kRowBytes;
  static constexpr int kStages = kTileBytes <= 32768 ? 3 : kTileBytes <= 65536 ? 2 : 1;
  // 128-byte tile rows are loaded with the TMA's 128-byte swizzle (16-byte
  // chunk j of row r lands at chunk j ^ (r & 7)), so that the token lanes of
  // a quarter-warp, which read the same chunks of different rows, hit
  // different banks.
  static constexpr bool kSwizzle = kRowBytes == 128;
  static constexpr int kMetaRows = 2 + 2 * kNC;
  // per-chunk min/max partials (2 x kNC x kW), double-buffered by block parity
  // when the next tile is in flight (a warp may still read one block's
  // partials while a faster warp writes the next block's)
  static constexpr int kRedSets = kStages > 1 ? 2 : 1;
  static constexpr int kRedFloats = kRedSets * 2 * kNC * kW;
  // page-statistic channels each token lane computes (of its group's 8)
  static constexpr int kCPL = kTL >= 8 ? 1 : 8 / kTL;
  // reduce-scatter over the token lanes (the chunk sum's levels h = TL/2 .. 1):
  // with 16 token lanes the first level is an all-reduce; every later level
  // halves the channels a lane keeps (channel bit 2, then 1, then 0), so a
  // lane ends with the kCPL channels whose statistics it finishes
  static constexpr int kLevels = kTL == 2 ? 1 : kTL == 4 ? 2 : kTL == 8 ? 3 : 4;
  static constexpr int kSplits = kLevels < 3 ? kLevels : 3;
  static constexpr int kAllLevels = kLevels - kSplits;
  // per-warp exchange of the finished statistics: [value][half][group][4]
  static constexpr int kScrFloats = 32 * kCG;
  static constexpr size_t kSmem = (size_t)kStages * kTileBytes + (size_t)kRedFloats * 4 +
                                  (size_t)kWarps * kScrFloats * 4 + kStages * 8;
  static_assert(C >= 16 && C <= P, "chunk");
  static_assert(P >= 64 && P <= 512, "page");
  static_assert(kSlices % kWarps == 0 && kW * C % 2048 == 0, "slices");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Token lane of lane slot k (lane / CG).  With swizzled tiles the 8 lanes of
// a quarter-warp hold 8/CG token lanes whose rows must differ in the row bits
// that select the swizzle, not in the low ones: slot k = (8/CG) q + j takes
// token lane CG j + (q mod CG) + 8 (q div CG).  Otherwise the identity.
template <int TL, int CG, bool SW>
__device__ __forceinline__ constexpr int enc_tl(int k) {
  if constexpr (!SW || TL < 8) {
    return k;
  } else {
    constexpr int nq = 8 / CG;
    const int q = k / nq, j = k % nq;
    return CG * j + q % CG + 8 * (q / CG);
  }
}
// Lane-slot xor that moves token lane tl to tl ^ hh (hh a power of two).
// The permutation above only reorders the bits of k, so this is the slot
// that holds token lane hh.
template <int TL, int CG, bool SW>
__device__ __forceinline__ constexpr int enc_kxor(int hh) {
  int k = 0;
  for (int b = 0; b < TL; ++b)
    if (enc_tl<TL, CG, SW>(b) == hh) k = b;
  return k;
}

// Lane-slot xor of level l of the token-lane reduction (token lanes tl and
// tl ^ TL/2^(l+1)).
template <int TL, int CG, bool SW>
__device__ __forceinline__ constexpr int enc_level_xor(int l) {
  return enc_kxor<TL, CG, SW>(TL >> (l + 1));
}
// First of the channels (of a group's 8) that lane slot k keeps after the
// split levels: split s keeps the half whose channel bit 2 - s equals the
// slot's bit at that level's xor.
template <int TL, int CG, bool SW, int ALL, int SPLITS>
__device__ __forceinline__ constexpr int enc_chan(int k) {
  int base = 0;
  for (int s = 0; s < SPLITS; ++s)
    if (k & enc_level_xor<TL, CG, SW>(ALL + s)) base |= 4 >> s;
  return base;
}

template <int P, int C>
__global__ void __launch_bounds__(EncGeom<P, C>::kThreads, (EncGeom<P, C>::kThreads <= 256 ? 2 : 1))
encode_kernel(const __grid_constant__ CUtensorMap tmap, const int64_t nunit,
              const int64_t NB, const int H, const int64_t L,
              uint32_t* __restrict__ anchor, uint32_t* __restrict__ residual,
              float* __restrict__ meta, const int32_t* __restrict__ bt, const int64_t nphys,
              const __grid_constant__ CompanderTable tab) {
  using G = EncGeom<P, C>;
  constexpr int W = G::kW;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  float* red_mn = reinterpret_cast<float*>(smem + G::kStages * G::kTileBytes);
  float* scr_all = red_mn + G::kRedFloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(scr_all + G::kWarps * G::kScrFloats);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int cg = lane % G::kCG, kl = lane / G::kCG;     // lane slot of the token lanes
  const int tl = enc_tl<G::kTL, G::kCG, G::kSwizzle>(kl);  // token offset in the chunk
  constexpr int kAll = G::kAllLevels, kSp = G::kSplits, kCPL = G::kCPL;
  // the kCPL channels of each group whose statistics this lane finishes
  const int cbase = enc_chan<G::kTL, G::kCG, G::kSwizzle, kAll, kSp>(kl);
  // one writer per channel (with an all-reduce level two lanes hold each)
  const bool owner = kAll == 0 || (kl & enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(0)) == 0;
  // which half a lane keeps at each split level
  const bool kb0 = kSp >= 1 && (kl & enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll)) != 0;
  const bool kb1 = kSp >= 2 && (kl & enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 1)) != 0;
  const bool kb2 = kSp >= 3 && (kl & enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 2)) != 0;
  // last split of the min / max words: keep {min, max} of channel bit kb2
  const uint32_t sel_keep = kb2 ? 0x7632u : 0x5410u, sel_send = kb2 ? 0x5410u : 0x7632u;
  // this warp's statistics exchange, [value][half][group][4]
  float* scr = scr_all + w * G::kScrFloats;
  auto scr_at = [&](int v, int j) { return scr + ((v * 2 + (j >> 2)) * G::kCG + cg) * 4 + (j & 3); };
  // write this lane's kCPL values of statistic v, then (after a __syncwarp)
  // read all 8 channels of the group as packed pairs
  auto scr_put = [&](int v, const float* x) {
    float* p = scr_at(v, cbase);
    if constexpr (kCPL == 1) p[0] = x[0];
    else if constexpr (kCPL == 2) *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    else *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  };
  auto scr_get = [&](int v, f2* out) {
    const float4 a = *reinterpret_cast<const float4*>(scr_at(v, 0));
    const float4 b = *reinterpret_cast<const float4*>(scr_at(v, 4));
    out[0] = make_float2(a.x, a.y);
    out[1] = make_float2(a.z, a.w);
    out[2] = make_float2(b.x, b.y);
    out[3] = make_float2(b.z, b.w);
  };

  if (G::kSwizzle && (smem_u32(tiles) & 1023u) != 0u) {
    // the swizzled reads assume 1024-byte aligned tiles; the host checks the
    // reserved shared memory before launching, so this is never taken
    if (tid == 0) atomicOr(&g_wait_timeout, kFlagWaitTimeout);
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < G::kStages; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const int64_t rows_total = nunit / G::kUnits / H * P;   // B * L rows of the BF16 view
  auto issue = [&](int64_t u, int stage) {
    const int64_t blk = u / G::kUnits, half = u % G::kUnits;
    const int64_t h = blk % H, rest = blk / H;
    const int64_t p = rest % NB, b = rest / NB;
    const int64_t x = checked_index(h * kD + half * W, (int64_t)H * kD - W + 1, &g_wait_timeout);
    const int64_t y = checked_index(b * L + p * P, rows_total - P + 1, &g_wait_timeout);
    mbar_expect_tx(&bars[stage], G::kTileBytes);
#pragma unroll
    for (int r0 = 0; r0 < P; r0 += 256)   // a box is at most 256 rows
      tma_load_2d(tiles + stage * G::kTileBytes + r0 * G::kRowBytes, &tmap, (int32_t)x,
                  (int32_t)(y + r0), &bars[stage]);
  };
  if (tid == 0)
    for (int i = 0; i < G::kStages; ++i) {
      const int64_t u = blockIdx.x + (int64_t)i * gridDim.x;
      if (u < nunit) issue(u, i);
    }

  // 16-byte chunk g of tile row t
  auto tile_at = [&](const uint4* tile, int t, int g) -> uint4 {
    if constexpr (G::kSwizzle) return tile[t * 8 + (g ^ (t & 7))];
    else return tile[t * (W / 8) + g];
  };

  const f2 alpha2 = make_float2(tab.alpha, tab.alpha), c16_2 = make_float2(tab.c16, tab.c16);
  const float inv_C = 1.0f / (float)C;
  int it = 0;
  for (int64_t u = blockIdx.x; u < nunit; u += gridDim.x, ++it) {
    const int stage = it % G::kStages;
    const uint32_t phase = (uint32_t)(it / G::kStages) & 1u;
    const bool ok = mbar_wait(&bars[stage], phase);
    const uint4* tile = reinterpret_cast<const uint4*>(tiles + stage * G::kTileBytes);
    const int64_t blk = u / G::kUnits;
    const int wofs = (int)(u % G::kUnits) * (W / 8);   // first channel group of the unit

    // ---- Stage 1a: per-chunk min / max of each channel (exact, on bf16
    // pairs) for every slice of the warp, into the partials
    float* pmn = red_mn + (G::kRedSets > 1 ? (it & 1) : 0) * (2 * G::kNC * W);  // [kNC][W]
    float* pmx = pmn + G::kNC * W;                                              // [kNC][W]
#pragma unroll 1
    for (int sl = 0; sl < G::kSlicesPerWarp; ++sl) {
      const int slice = w + G::kWarps * sl;
      const int c = slice / G::kSlicesPerChunk;
      const int g = (slice % G::kSlicesPerChunk) * G::kCG + cg;   // group within the unit
      uint32_t mn[4], mx[4];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint4 v = tile_at(tile, c * C + G::kTL * m + tl, g);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          mn[k] = m == 0 ? vv[k] : bf2_min(mn[k], vv[k]);
          mx[k] = m == 0 ? vv[k] : bf2_max(mx[k], vv[k]);
        }
      }
      // across the token lanes: all-reduce levels, then split levels that
      // leave each lane the extremes of its own kCPL channels
#pragma unroll
      for (int l = 0; l < kAll; ++l) {
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(l) * G::kCG;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          mn[k] = bf2_min(mn[k], __shfl_xor_sync(kFull, mn[k], x));
          mx[k] = bf2_max(mx[k], __shfl_xor_sync(kFull, mx[k], x));
        }
      }
      if constexpr (kSp >= 1) {   // channel bit 2: words {0, 1} or {2, 3}
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll) * G::kCG;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t smn = kb0 ? mn[j] : mn[j + 2], kmn = kb0 ? mn[j + 2] : mn[j];
          const uint32_t smx = kb0 ? mx[j] : mx[j + 2], kmx = kb0 ? mx[j + 2] : mx[j];
          mn[j] = bf2_min(kmn, __shfl_xor_sync(kFull, smn, x));
          mx[j] = bf2_max(kmx, __shfl_xor_sync(kFull, smx, x));
        }
      }
      if constexpr (kSp >= 2) {   // channel bit 1: word 0 or 1
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 1) * G::kCG;
        const uint32_t smn = kb1 ? mn[0] : mn[1], kmn = kb1 ? mn[1] : mn[0];
        const uint32_t smx = kb1 ? mx[0] : mx[1], kmx = kb1 ? mx[1] : mx[0];
        mn[0] = bf2_min(kmn, __shfl_xor_sync(kFull, smn, x));
        mx[0] = bf2_max(kmx, __shfl_xor_sync(kFull, smx, x));
      }
      float plo[kCPL], phi[kCPL];
      if constexpr (kSp >= 3) {   // channel bit 0: one half of the min and max words
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 2) * G::kCG;
        const uint32_t keep = prmt(mn[0], mx[0], sel_keep);   // {min, max} halves
        const uint32_t r = __shfl_xor_sync(kFull, prmt(mn[0], mx[0], sel_send), x);
        const uint32_t mm = prmt(bf2_min(keep, r), bf2_max(keep, r), 0x7610u);
        plo[0] = __uint_as_float(mm << 16);
        phi[0] = __uint_as_float(mm & 0xffff0000u);
      } else {
#pragma unroll
        for (int j = 0; j < kCPL / 2; ++j) {
          const f2 a = bf2_to_f2(mn[j]), b = bf2_to_f2(mx[j]);
          plo[2 * j] = a.x;
          plo[2 * j + 1] = a.y;
          phi[2 * j] = b.x;
          phi[2 * j + 1] = b.y;
        }
      }
      if (owner) {
        float* pm = pmn + c * W + 8 * g + cbase;
        float* px = pmx + c * W + 8 * g + cbase;
        if constexpr (kCPL == 1) {
          pm[0] = plo[0];
          px[0] = phi[0];
        } else if constexpr (kCPL == 2) {
          *reinterpret_cast<float2*>(pm) = make_float2(plo[0], plo[1]);
          *reinterpret_cast<float2*>(px) = make_float2(phi[0], phi[1]);
        } else {
          *reinterpret_cast<float4*>(pm) = make_float4(plo[0], plo[1], plo[2], plo[3]);
          *reinterpret_cast<float4*>(px) = make_float4(phi[0], phi[1], phi[2], phi[3]);
        }
      }
    }
    if (!__syncthreads_and(ok)) {
      // A stage never arrived: record it and stop this CTA (bounded waits
      // only, so the context stays usable).
      if (tid == 0) {
        atomicOr(&g_wait_timeout, kFlagWaitTimeout);
        for (int i = 0; i < G::kStages; ++i) (void)mbar_wait(&bars[i], phase);
      }
      return;
    }
    // Every thread has finished the previous unit, so its stage can be
    // refilled with the unit kStages-1 iterations ahead of this one.  (With
    // one stage the refill waits for the end of this unit instead.)
    if (G::kStages > 1 && tid == 0 && it > 0) {
      const int64_t nxt = u + (int64_t)(G::kStages - 1) * gridDim.x;
      if (nxt < nunit) {
        fence_proxy_async();
        issue(nxt, (it - 1) % G::kStages);
      }
    }

    const int64_t pb = checked_index(phys_block(bt, nphys, blk, H, &g_wait_timeout),
                                     bt ? nphys * H : nunit / G::kUnits, &g_wait_timeout);
    float* mrow = meta + pb * (int64_t)(G::kMetaRows * kD) + 8 * wofs;
    uint32_t* arow = anchor + pb * (int64_t)(P * 16) + wofs;
    uint32_t* rrow = residual + pb * (int64_t)(P * 16) + wofs;
#pragma unroll 1
    for (int sl = 0; sl < G::kSlicesPerWarp; ++sl) {
      const int slice = w + G::kWarps * sl;
      const int c = slice / G::kSlicesPerChunk;
      const int g = (slice % G::kSlicesPerChunk) * G::kCG + cg;

      // ---- Stage 1b: gamma_min, gamma_scale, reciprocal.  The token lanes
      // that share a channel group split its 8 channels (kCPL each, the ones
      // the reduce-scatter leaves them; with 16 token lanes two lanes compute
      // each channel) and exchange them through the warp's exchange.
      float lo_q[G::kCPL], rg_q[G::kCPL];
#pragma unroll
      for (int q = 0; q < G::kCPL; ++q) {
        const int ch = 8 * g + cbase + q;
        float lo = pmn[ch], hi = pmx[ch];
#pragma unroll
        for (int cc = 1; cc < G::kNC; ++cc) {
          lo = fminf(lo, pmn[cc * W + ch]);
          hi = fmaxf(hi, pmx[cc * W + ch]);
        }
        // one sign for a zero extreme: -0 for the minimum (zero x then
        // centre to +0), +0 for the maximum
        if (lo == 0.0f) lo = -0.0f;
        if (hi == 0.0f) hi = 0.0f;
        const float gs = __fsub_rn(hi, lo);
        lo_q[q] = lo;
        rg_q[q] = __frcp_rn(__fadd_rn(gs, kEps));
        if (c == 0 && owner) {
          mrow[ch] = lo;
          mrow[kD + ch] = gs;
        }
      }
      // ---- Stage 1c: n = (x - gmin) * rg for the thread's 8 tokens x 8 ch,
      // with every channel's gmin and rg from the warp's exchange
      if (owner) {
        scr_put(0, lo_q);
        scr_put(1, rg_q);
      }
      __syncwarp();
      f2 gm2[4], rg2[4];
      scr_get(0, gm2);
      scr_get(1, rg2);
      f2 n[8][4];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint4 v = tile_at(tile, c * C + G::kTL * m + tl, g);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // scalar __fmul_rn, never contracted: a packed mul.rn.f32x2 here
          // was fused with the first add of the chunk sum below
          const f2 d = bf2_sub_f32(vv[k], gm2[k]);
          n[m][k].x = __fmul_rn(d.x, rg2[k].x);
          n[m][k].y = __fmul_rn(d.y, rg2[k].y);
        }
      }

      // ---- Stage 2a: chunk mean, pairwise-halving order: the register
      // index first, then the token lanes (all-reduce levels, then split
      // levels that leave each lane the sums of its own kCPL channels)
      f2 s[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f2 t0 = add2(n[0][k], n[4][k]), t1 = add2(n[1][k], n[5][k]);
        f2 t2 = add2(n[2][k], n[6][k]), t3 = add2(n[3][k], n[7][k]);
        t0 = add2(t0, t2);
        t1 = add2(t1, t3);
        s[k] = add2(t0, t1);
      }
      auto shfl2 = [&](f2 v, int x) {
        return make_float2(__shfl_xor_sync(kFull, v.x, x), __shfl_xor_sync(kFull, v.y, x));
      };
#pragma unroll
      for (int l = 0; l < kAll; ++l) {
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(l) * G::kCG;
#pragma unroll
        for (int k = 0; k < 4; ++k) s[k] = add2(s[k], shfl2(s[k], x));
      }
      if constexpr (kSp >= 1) {   // channel bit 2: pairs {0, 1} or {2, 3}
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll) * G::kCG;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const f2 snd = kb0 ? s[j] : s[j + 2], kp = kb0 ? s[j + 2] : s[j];
          s[j] = add2(kp, shfl2(snd, x));
        }
      }
      if constexpr (kSp >= 2) {   // channel bit 1: pair 0 or 1
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 1) * G::kCG;
        const f2 snd = kb1 ? s[0] : s[1], kp = kb1 ? s[1] : s[0];
        s[0] = add2(kp, shfl2(snd, x));
      }
      float mu_q[kCPL];
      if constexpr (kSp >= 3) {   // channel bit 0: one of the pair
        const int x = enc_level_xor<G::kTL, G::kCG, G::kSwizzle>(kAll + 2) * G::kCG;
        const float snd = kb2 ? s[0].x : s[0].y, kp = kb2 ? s[0].y : s[0].x;
        mu_q[0] = __fmul_rn(__fadd_rn(kp, __shfl_xor_sync(kFull, snd, x)), inv_C);
      } else {
#pragma unroll
        for (int j = 0; j < kCPL / 2; ++j) {
          mu_q[2 * j] = __fmul_rn(s[j].x, inv_C);
          mu_q[2 * j + 1] = __fmul_rn(s[j].y, inv_C);
        }
      }

      // ---- Stage 2b: d = n - mu; sigma = max |d| over the chunk.  Every
      // step x -> x - gmin -> * rg -> - mu rounds monotonically (rg > 0), so
      // the largest |d| is that of the chunk's largest or smallest x, which
      // stage 1a left in the partials.  Each lane finishes sigma and
      // rs = rn(1/(sigma + eps)) of its own channels; the warp's exchange
      // hands mu and rs of all 8 channels of the group to every lane.
      float rs_q[kCPL];
#pragma unroll
      for (int q = 0; q < kCPL; ++q) {
        const int ch = 8 * g + cbase + q;
        const float nlo = __fmul_rn(__fsub_rn(pmn[c * W + ch], lo_q[q]), rg_q[q]);
        const float nhi = __fmul_rn(__fsub_rn(pmx[c * W + ch], lo_q[q]), rg_q[q]);
        const float sg = fmaxf(fabsf(__fsub_rn(nlo, mu_q[q])), fabsf(__fsub_rn(nhi, mu_q[q])));
        rs_q[q] = __frcp_rn(__fadd_rn(sg, kEps));
        if (owner) {
          mrow[(2 + c) * kD + ch] = mu_q[q];
          mrow[(2 + G::kNC + c) * kD + ch] = sg;
        }
      }
      if (owner) {
        scr_put(2, mu_q);
        scr_put(3, rs_q);
      }
      __syncwarp();
      f2 mu2[4], rs2[4];
      scr_get(2, mu2);
      scr_get(3, rs2);
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) n[m][k] = sub2(n[m][k], mu2[k]);

      // ---- Stages 3-4: codes, sign map, nibble split, store one row per m
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int t = c * C + G::kTL * m + tl;
        float a[8];
        uint32_t bits[8], dbits[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const f2 xf = mul2(n[m][k], rs2[k]);
          a[2 * k] = fabsf(xf.x);
          a[2 * k + 1] = fabsf(xf.y);
          dbits[2 * k] = __float_as_uint(n[m][k].x);
          dbits[2 * k + 1] = __float_as_uint(n[m][k].y);
          compand_fast2(make_float2(a[2 * k], a[2 * k + 1]), alpha2, c16_2, bits[2 * k],
                        bits[2 * k + 1]);
        }
        // smallest distance to a rounding boundary (the low 16 bits) of the
        // 8 values: a 16-bit-lane minimum over the words (their high halves
        // are not looked at), then one test of the low half
        const uint32_t d01 = __vminu2(bits[0], bits[1]), d23 = __vminu2(bits[2], bits[3]);
        const uint32_t d45 = __vminu2(bits[4], bits[5]), d67 = __vminu2(bits[6], bits[7]);
        const uint32_t dmin = __vminu2(__vminu2(d01, d23), __vminu2(d45, d67));
        const bool amb = (dmin & 0xffffu) < 2u * kAmbiguityK;
        if (amb) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (compand_ambiguous(bits[i]))
              bits[i] = (bits[i] & 0xff00ffffu) | (compand_exact(bits[i], a[i], tab.thr) << 16);
        }
        // code bytes (byte 2 of bits) xor the replicated sign of d
        const uint32_t i01 = prmt(bits[0], bits[1], 0x0062u), i23 = prmt(bits[2], bits[3], 0x0062u);
        const uint32_t i45 = prmt(bits[4], bits[5], 0x0062u), i67 = prmt(bits[6], bits[7], 0x0062u);
        const uint32_t s01 = prmt(dbits[0], dbits[1], 0x00fbu), s23 = prmt(dbits[2], dbits[3], 0x00fbu);
        const uint32_t s45 = prmt(dbits[4], dbits[5], 0x00fbu), s67 = prmt(dbits[6], dbits[7], 0x00fbu);
        const uint32_t W0 = prmt(i01 ^ s01, i23 ^ s23, 0x5410u);
        const uint32_t W1 = prmt(i45 ^ s45, i67 ^ s67, 0x5410u);
        // byte k: Anchor = (ch k high nibble) | (ch k+4 high nibble) << 4, etc.
        const uint32_t Aw = ((W0 >> 4) & 0x0f0f0f0fu) | (W1 & 0xf0f0f0f0u);
        const uint32_t Rw = (W0 & 0x0f0f0f0fu) | ((W1 << 4) & 0xf0f0f0f0u);
        arow[t * 16 + g] = Aw;
        rrow[t * 16 + g] = Rw;
      }
    }
    if constexpr (G::kStages == 1) {
      // one stage: every warp has read the tile and the partials of this
      // unit; refill the stage with the next unit
      __syncthreads();
      if (tid == 0) {
        const int64_t nxt = u + gridDim.x;
        if (nxt < nunit) {
          fence_proxy_async();
          issue(nxt, 0);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ launch

template <int P, int C>
static cudaError_t run_encode(const CUtensorMap& map, const Shape& s, const CompanderTable& tab,
                              void* anchor, void* residual, float* meta, cudaStream_t stream,
                              const Paging& pg) {
  using G = EncGeom<P, C>;
  auto fn = encode_kernel<P, C>;
  static thread_local int configured_dev = -1;
  static thread_local int per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    if (G::kSwizzle) {
      // swizzled tiles start 1024-byte aligned only if dynamic shared memory
      // does (it follows the block's reserved shared memory)
      int reserved = -1;
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
      if (e != cudaSuccess) return e;
      if (reserved % 1024 != 0) return cudaErrorNotSupported;
    }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, G::kThreads, G::kSmem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
    configured_dev = dev;
  }
  const int64_t nunit = s.blocks() * G::kUnits;
  int64_t grid = (int64_t)sm_count() * per_sm;
  if (grid > nunit) grid = nunit;
  fn<<<(unsigned)grid, G::kThreads, G::kSmem, stream>>>(
      map, nunit, s.NB(), s.H, s.L, static_cast<uint32_t*>(anchor),
      static_cast<uint32_t*>(residual), meta, pg.table, pg.nphys, tab);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

template <int P, int C>
static cudaError_t encode_case(EncodeTiledFn enc, const void* kv, const Shape& s,
                               const CompanderTable& tab, void* anchor, void* residual,
                               float* meta, cudaStream_t stream, const Paging& pg) {
  using G = EncGeom<P, C>;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)s.H * kD, (cuuint64_t)(s.B * s.L)};
  const cuuint64_t strides[1] = {(cuuint64_t)s.H * kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)G::kW, (cuuint32_t)(P < 256 ? P : 256)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   G::kSwizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  return run_encode<P, C>(map, s, tab, anchor, residual, meta, stream, pg);
}

cudaError_t launch_encode(const void* kv, const Shape& s, const CompanderTable& tab,
                          void* anchor, void* residual, float* meta, cudaStream_t stream,
                          const Paging& pg) {
  if (s.blocks() == 0) return cudaSuccess;
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return cudaErrorNotSupported;
#define LYNX_ENC_CASE(PP, CC) \
  if (s.page == PP && s.C == CC)                                            \
    return encode_case<PP, CC>(enc, kv, s, tab, anchor, residual, meta, stream, pg);
  LYNX_ENC_CASE(64, 16) LYNX_ENC_CASE(64, 32) LYNX_ENC_CASE(64, 64)
  LYNX_ENC_CASE(128, 16) LYNX_ENC_CASE(128, 32) LYNX_ENC_CASE(128, 64) LYNX_ENC_CASE(128, 128)
  LYNX_ENC_CASE(256, 16) LYNX_ENC_CASE(256, 32) LYNX_ENC_CASE(256, 64) LYNX_ENC_CASE(256, 128)
  LYNX_ENC_CASE(512, 16) LYNX_ENC_CASE(512, 32) LYNX_ENC_CASE(512, 64) LYNX_ENC_CASE(512, 128)
#undef LYNX_ENC_CASE
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------ self-check

// For every float32 a in [0, 1]: fast path vs threshold count.
__global__ void compander_selfcheck_kernel(const __grid_constant__ CompanderTable tab,
                                           unsigned long long* counts) {
  __shared__ float thr[128];
  for (int i = threadIdx.x; i < 128; i += blockDim.x) thr[i] = tab.thr[i];
  __syncthreads();
  const uint32_t last = 0x3f800000u;  // bits of 1.0f
  unsigned long long n = 0, bad = 0, amb = 0, maxerr = 0;
  const double la = log1p((double)tab.alpha);
  for (uint64_t ub = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; ub <= last;
       ub += (uint64_t)gridDim.x * blockDim.x) {
    const float a = __uint_as_float((uint32_t)ub);
    uint32_t bits, unused;
    compand_fast2(make_float2(a, a), make_float2(tab.alpha, tab.alpha),
                  make_float2(tab.c16, tab.c16), bits, unused);
    int lo = 0, hi = 127;  // exact: number of thresholds <= a
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (a >= thr[mid]) lo = mid + 1; else hi = mid;
    }
    const uint32_t exact = (uint32_t)lo;
    ++n;
    if (compand_ambiguous(bits)) {
      ++amb;
      if (compand_exact(bits, a, thr) != exact) ++bad;
    } else if (((bits >> 16) & 0xffu) != exact) {
      ++bad;
    }
    // approximation error of Y' = lg * c16 / 65536 against float64 Y
    const double y = 127.0 * log1p((double)tab.alpha * (double)a) / la;
    const double yf = (double)lg2_approx(fmaf(tab.alpha, a, 1.0f)) * (double)tab.c16 / 65536.0;
    const double err = fabs(yf - y) * 4294967296.0;
    const unsigned long long e = (unsigned long long)(err < 1.8e19 ? err : 1.8e19);
    if (e > maxerr) maxerr = e;
  }
  // warp reduce then one atomic per warp
  for (int o = 16; o; o >>= 1) {
    n += __shfl_xor_sync(kFull, n, o);
    bad += __shfl_xor_sync(kFull, bad, o);
    amb += __shfl_xor_sync(kFull, amb, o);
    const unsigned long long m2 = __shfl_xor_sync(kFull, maxerr, o);
    maxerr = m2 > maxerr ? m2 : maxerr;
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&counts[0], n);
    atomicAdd(&counts[1], bad);
    atomicAdd(&counts[2], amb);
    atomicMax(&counts[3], maxerr);
  }
}

cudaError_t launch_compander_selfcheck(const CompanderTable& tab, uint64_t* counts,
                                       cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(counts, 0, 4 * sizeof(uint64_t), stream);
  if (e != cudaSuccess) return e;
  compander_selfcheck_kernel<<<sm_count() * 8, 256, 0, stream>>>(
      tab, reinterpret_cast<unsigned long long*>(counts));
  return cudaGetLastError();
}

}  // namespace lynx
