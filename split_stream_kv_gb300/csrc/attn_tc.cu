// attn_tc.cu -- the verification pass of decode attention (Prerequisites
// Eq. 1 over the Anchor + Residual codes: the T draft tokens verified in one
// pass of "Lynx: Progressive Speculative KV Cache Transfer for Disaggregated
// LLM Inference", Mechanism 3) on the tensor-memory path of sm_103a.
//
// One CTA per SM walks its share of the (unit, tile) space; a unit is one
// (sequence, KV head, group of up to 32 query rows), a tile 128 tokens.
// Warp roles:
//  * 8 producer warps rebuild the tile's keys and values from the packed
//    codes.  A code byte (Anchor nibble over Residual nibble) indexes a
//    lane-replicated table of the decoder's values v; x = fma(v, A, B) with
//    the chunk's one-FMA constants A = (sigma + eps)(gamma_scale + eps),
//    B = fma(mu, gamma_scale + eps, gamma_min), rounded to nearest even BF16,
//    goes to shared memory as 8 x 8 core matrices (two tile stages).
//  * the tcgen05 MMAs, issued by softmax thread 0: S^T = K^ Q^T (M = 128
//    tokens, N = 32 rows, K = 128 channels) into tensor memory once the K
//    producers have signalled the tile, and O^T += V^T [P_hi | P_lo]^T
//    (M = 128 channels, N = 64, K = 128 tokens) once the softmax warps have
//    written P and the V producers have signalled the tile, into an
//    accumulator that stays in tensor memory for the whole unit.
//  * 4 softmax warps, one thread per token (its tensor-memory lane), turn
//    the token's 32 scores into weights p = 2^(s log2(e)/sqrt(d) - m_r)
//    against each row's running maximum m_r.  m_r is raised only when some
//    weight of the tile would exceed 2^8 (a vote of the 4 warps per tile);
//    then the tile's row maxima are reduced across the threads and the
//    output accumulator and the row sums are rescaled.  A tile that raises
//    no maximum needs no cross-thread reduction.  P is split into bf16
//    hi + lo parts (about 16 mantissa bits) stored side by side as the 64
//    columns of the second MMA's B operand, so V^ is read once.
// At the end of a unit the softmax threads read O back (one thread per
// channel), add the hi and lo halves and write the CTA's partial (m, l, o)
// for the split combine (attn.cu), which also adds the draft tokens' own keys
// and values when the call has them.
//
// Every wait on an mbarrier is bounded.  A wait that runs out sets an abort
// word: from then on every wait of every role returns at once, the roles run
// their remaining iterations without waiting (so the named barriers stay
// matched), and the call's flag word records kFlagWaitTimeout.
#include <math.h>

#include "attn_params.h"
#include "common.cuh"
#include "internal.h"

namespace lynx {

__device__ unsigned int g_attn_tc_flags = 0;

cudaError_t read_attn_tc_flags(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_attn_tc_flags, sizeof(unsigned int));
}

namespace tc {

constexpr int kTile = 128;            // tokens per tile
constexpr int kRows = 32;             // query rows per pass
constexpr int kProdWarps = 8;
constexpr int kSoftWarps = 4;
// 12 warps: three per SM sub-partition, so up to 168 registers a thread
constexpr int kThreads = 32 * (kProdWarps + kSoftWarps);
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kSoftThreads = 32 * kSoftWarps;
// Shared memory, offsets from the start of the dynamic window (shared address
// kSmemBase; the host checks the block's reserved shared memory):
//  [0, 64K)    table: 256 rows of 256 bytes, one per code byte; bytes 0..127 the
//              32 lanes' copies of the value, bytes 128..255 the one-FMA
//              constants of each producer warp's chunks (see piece_off)
//  [64K,192K)  two stages of the K^ and V^ tiles (32 KiB each)
//  [192K,208K) Q of the CTA's two units (K-major core matrices, 8 KiB each)
//  [208K,224K) P^T: 64 columns (hi rows 0..31, lo rows 32..63) x 128 tokens;
//              also the row-sum scratch of the unit epilogue
//  then the mbarriers, the tensor-memory address, the abort word, the vote
//  words, and the softmax's row maxima (per-warp scratch, running, factors).
constexpr uint32_t kLut = 0;
constexpr uint32_t kStage = 0x10000;          // + stage * 64K: K^ then V^
constexpr uint32_t kTileBytes = 0x8000;
constexpr uint32_t kQ = kStage + 4 * kTileBytes;
constexpr uint32_t kQBytes = 0x2000;
constexpr uint32_t kP = kQ + 2 * kQBytes;
constexpr uint32_t kPBytes = 0x4000;
constexpr uint32_t kBar = kP + kPBytes;
// mbarrier indices
constexpr int kBKEmpty = 0, kBVEmpty = 2, kBKFull = 4, kBVFull = 6, kBSReady = 8, kBSFree = 10,
              kBODone = 12;
constexpr uint32_t kMisc = kBar + 8 * 16;     // [0] tmem address, [1] abort, [2..4] votes
constexpr uint32_t kRed = kMisc + 64;         // [4 warps][32 rows], [32], [32] floats
constexpr uint32_t kSmem = kRed + (kSoftWarps + 2) * kRows * 4;
static_assert(kSmem <= 227 * 1024, "one CTA per SM");
// Tensor memory columns: S^T of the two stages, then O^T (hi, lo).
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0, kColO = 64;

// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, the
// operand majors (1 = M/N-major) and the shape.
constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdS = idesc(128, kRows, 0, 0);
constexpr uint32_t kIdO = idesc(128, 2 * kRows, 1, 1);

// Shared-memory matrix descriptor without swizzle: start address, the byte
// stride between core matrices along K (lbo) and along M/N (sbo).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                     uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
// 32 columns of the calling warp's lane quarter, one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
         "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
         "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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
// Table value of byte POS of the code word w for this lane: the load address
// is [lane_off, w.byte POS] = byte << 8 | lane * 4, plus the window base.
template <int POS>
__device__ __forceinline__ float lut(uint32_t w, uint32_t lane_off) {
  const uint32_t off = prmt(w, lane_off, 0x7604u | ((uint32_t)POS << 4));
  float v;
  asm("ld.shared.f32 %0, [%1+1024];" : "=f"(v) : "r"(off));
  return v;
}
static_assert(kSmemBase == 1024, "immediate offset of the table loads");

// Byte offset of 16-byte constant piece k (0, 1: A of channels 8G..8G+3,
// 8G+4..8G+7; 2, 3: B) of channel group G, chunk ch (0, 1) of producer warp
// w's 32 tokens, in the table's row tails.  Pieces of groups G and G + 8 sit
// in consecutive rows, rotated by two slots, so that the four groups one load
// instruction reads (G = gi, gi + 4, gi + 8, gi + 12) hit distinct banks.
__device__ __forceinline__ uint32_t piece_off(int w, int ch, int k, int G) {
  const uint32_t pi = (uint32_t)((w * 2 + ch) * 64 + k * 16 + G);
  const uint32_t row = pi >> 3, slot = (pi + ((pi >> 3) & 1u) * 2u) & 7u;
  return row * 256u + 128u + slot * 16u;
}

// Bounded wait; false once the CTA has aborted (see the file comment).  A
// wait that runs out after limit_ns raises the CTA's abort word and records
// kFlagWaitTimeout in *flags.
__device__ __forceinline__ bool wait_bar_for(uint64_t* bar, uint32_t phase,
                                             volatile uint32_t* abort_w, uint64_t limit_ns,
                                             unsigned int* flags) {
  if (mbar_try_wait(bar, phase)) return true;
  if (*abort_w) return false;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, phase)) return true;
    if (*abort_w) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_w = 1u;
      atomicOr(flags, kFlagWaitTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t phase, volatile uint32_t* abort_w) {
  return wait_bar_for(bar, phase, abort_w, kWaitNs, &g_attn_tc_flags);
}

}  // namespace tc

// C16: chunks of 16 tokens (two per 32-token producer range), else >= 32.
template <bool PAGED, bool C16>
__global__ void __launch_bounds__(tc::kThreads, 1)
attn_tc_kernel(const __grid_constant__ AttnParams a, const __grid_constant__ ExpandTable tab) {
  using namespace tc;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int64_t cta_b = a.n_chunks * cta / a.n_cta, cta_e = a.n_chunks * (cta + 1) / a.n_cta;
  const int n = (int)(cta_e - cta_b);
  const int64_t u0 = cta_b / a.NCH;
  const int64_t units = a.n_chunks / a.NCH;
  constexpr int RP = kRows;
  const int part_floats = 2 * RP + RP * kD;

  if (smem_u32(smem) != kSmemBase) {  // table loads would read the wrong bytes
    for (int i = tid; i < 2 * part_floats; i += kThreads)
      a.part[(int64_t)2 * cta * part_floats + i] = __int_as_float(0x7fc00000);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kMisc);
  volatile uint32_t* abort_w = misc + 1;

  // (sequence, KV head, row group) of segment sg (unit u0 + sg)
  auto unit_b = [&](int sg) { return (int)((u0 + sg) / a.nrg / a.Hkv); };
  auto unit_h = [&](int sg) { return (int)(((u0 + sg) / a.nrg) % a.Hkv); };
  auto unit_rg = [&](int sg) { return (int)((u0 + sg) % a.nrg); };
  // A share spans at most two units (at least one CTA per unit), so tile i of
  // the share is tile ti0 + i of unit u0, or of unit u0 + 1 past its end: no
  // division per tile.
  const int64_t ti0 = cta_b - u0 * a.NCH;
  auto seg_of = [&](int i) { return ti0 + i >= a.NCH ? 1 : 0; };
  auto tile_tok = [&](int i) -> int64_t {   // first token of tile i in its sequence
    const int64_t t = ti0 + i;
    return (t >= a.NCH ? t - a.NCH : t) * kTile;
  };
  const int sb0 = unit_b(0), sb1 = unit_b(1), sh0 = unit_h(0), sh1 = unit_h(1);
  // Packed block holding token `tok` of segment sg's sequence.
  auto block_of = [&](int sg, int64_t tok) -> int64_t {
    const int64_t p = tok >> a.lgP;
    const int b = sg ? sb1 : sb0, h = sg ? sh1 : sh0;
    if constexpr (PAGED) {
      int64_t pg = __ldg(a.bt + (int64_t)b * a.NB + p);
      if (pg < 0 || pg >= a.nphys) {
        atomicOr(&g_attn_tc_flags, kFlagBadBlock);
        pg = 0;
      }
      return checked_index(pg * a.Hkv + h, a.nphys * a.Hkv, &g_attn_tc_flags);
    } else {
      return checked_index(((int64_t)b * a.NB + p) * a.Hkv + h, (int64_t)a.batch * a.NB * a.Hkv,
                           &g_attn_tc_flags);
    }
  };

  // ---- set-up: table, Q of both units, barriers, tensor memory
  for (int i = tid; i < 256 * 32; i += kThreads) {
    const int row = i >> 5, l = i & 31;
    reinterpret_cast<float*>(smem + kLut + row * 256)[l] =
        row < 128 ? tab.x[row] : -tab.x[255 - row];
  }
  for (int i = tid; i < 2 * RP * 16; i += kThreads) {
    const int sg = i / (RP * 16), r = (i / 16) % RP, G = i % 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const int rr = unit_rg(sg) * RP + r;
    if (u0 + sg < units && rr < a.R) {
      const int tq = rr / a.G, gq = rr % a.G;
      v = *reinterpret_cast<const uint4*>(
          a.q + ((int64_t)(unit_b(sg) * a.T + tq) * a.Hq + unit_h(sg) * a.G + gq) * kD + 8 * G);
    }
    *reinterpret_cast<uint4*>(smem + kQ + sg * kQBytes + (r >> 3) * 2048 + G * 128 +
                              (r & 7) * 16) = v;
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBKEmpty + i], 1);
      mbar_init(&bars[kBVEmpty + i], 1);
      mbar_init(&bars[kBKFull + i], kProdThreads / 2);
      mbar_init(&bars[kBVFull + i], kProdThreads / 2);
      mbar_init(&bars[kBSReady + i], 1);
      mbar_init(&bars[kBSFree + i], kSoftThreads);
    }
    mbar_init(&bars[kBODone], 1);
    for (int i = 1; i < 16; ++i) misc[i] = 0u;
    float* msm = reinterpret_cast<float*>(smem + kRed) + kSoftWarps * kRows;
    for (int r = 0; r < kRows; ++r) msm[r] = -INFINITY;
    fence_barrier_init();
  }
  if (w == kProdWarps) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(smem + kMisc)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();  // Q is read by the tensor core
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = misc[0];

  if (w < kProdWarps) {
    // ================= producers: K^ (warps 0-3) and V^ (warps 4-7).  No
    // barrier joins them: each warp computes the one-FMA constants of its own
    // chunk(s), and the tile's completion is signalled on an mbarrier per
    // tensor (K^: the softmax's thread 0 then issues the scores; V^: it
    // issues the output MMA).
    const int T = w >> 2, wr = w & 3;          // tensor, 32-token range of the tile
    const int gq = lane >> 3, t8 = lane & 7;   // channel groups 4gq..4gq+3, tokens t8 + 8j
    const uint8_t* an = T ? a.va : a.ka;
    const uint8_t* re = T ? a.vr : a.kr;
    const uint32_t lane_off = (uint32_t)lane * 4u;
    const int meta_rows = 2 + 2 * a.NC;
    constexpr int kChunks = C16 ? 2 : 1;       // chunks of the warp's 32 tokens
    // constant item of this lane: channels 8G + 4hh .. +3 of each chunk
    const int it_hh = lane & 1, it_G = lane >> 1;

    // codes of tile i for this lane: anchor / residual bytes 16gq..16gq+15
    // of tokens 32wr + t8 + 8j
    // (blk: the packed block of the warp's 32 tokens of tile i; a page holds at
    // least 64 tokens, so one block serves them)
    auto load_codes = [&](int i, int64_t blk, uint4 (&A)[4], uint4 (&R)[4]) {
      const int64_t tok = tile_tok(i) + 32 * wr;
      const int64_t row0 = blk * a.P + (tok & (a.P - 1));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t off = checked_index((row0 + t8 + 8 * j) * 64 + 16 * gq,
                                          (PAGED ? a.nphys * a.Hkv : (int64_t)a.batch * a.NB * a.Hkv) *
                                              a.P * 64, &g_attn_tc_flags);
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(A[j].x), "=r"(A[j].y), "=r"(A[j].z), "=r"(A[j].w) : "l"(an + off));
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(R[j].x), "=r"(R[j].y), "=r"(R[j].z), "=r"(R[j].w) : "l"(re + off));
      }
    };
    // raw metadata of the lane's constant items for tile i: gamma_min,
    // gamma_scale, mu, sigma of 4 channels per chunk
    float4 mr[kChunks][4];
    auto load_meta = [&](int i, int64_t blk) {
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int64_t tok = tile_tok(i) + 32 * wr + 16 * k;   // a token of chunk k
        const int cc = (int)((tok & (a.P - 1)) >> a.lgC);
        const float* mb = (T ? a.vm : a.km) + blk * (int64_t)meta_rows * kD + 8 * it_G + 4 * it_hh;
        mr[k][0] = __ldg(reinterpret_cast<const float4*>(mb));
        mr[k][1] = __ldg(reinterpret_cast<const float4*>(mb + kD));
        mr[k][2] = __ldg(reinterpret_cast<const float4*>(mb + (2 + cc) * kD));
        mr[k][3] = __ldg(reinterpret_cast<const float4*>(mb + (2 + a.NC + cc) * kD));
      }
    };
    auto warp_block = [&](int i) { return block_of(seg_of(i), tile_tok(i) + 32 * wr); };
    uint4 ca[4], cr[4];
    // paged: the block of tile i + 1, read from the block table a tile ahead
    // so that the code loads need not wait for it (dense: arithmetic)
    int64_t blk_next = 0;
    if (n > 0) {
      const int64_t blk0 = warp_block(0);
      load_codes(0, blk0, ca, cr);
      load_meta(0, blk0);
    }
    if (PAGED && n > 1) blk_next = warp_block(1);
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      // the one-FMA constants of this warp's chunk(s) of tile i (the warp's
      // last reads of the previous tile's constants precede this __syncwarp)
      __syncwarp();
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const f2 e = make_float2(kEps, kEps);
        const f2 gm0 = make_float2(mr[k][0].x, mr[k][0].y), gm1 = make_float2(mr[k][0].z, mr[k][0].w);
        const f2 gs0 = add2(make_float2(mr[k][1].x, mr[k][1].y), e);
        const f2 gs1 = add2(make_float2(mr[k][1].z, mr[k][1].w), e);
        const f2 mu0 = make_float2(mr[k][2].x, mr[k][2].y), mu1 = make_float2(mr[k][2].z, mr[k][2].w);
        const f2 sg0 = add2(make_float2(mr[k][3].x, mr[k][3].y), e);
        const f2 sg1 = add2(make_float2(mr[k][3].z, mr[k][3].w), e);
        const f2 A0 = mul2(sg0, gs0), A1 = mul2(sg1, gs1);
        const f2 B0 = fma2(mu0, gs0, gm0), B1 = fma2(mu1, gs1, gm1);
        *reinterpret_cast<float4*>(smem + piece_off(w, k, it_hh, it_G)) =
            make_float4(A0.x, A0.y, A1.x, A1.y);
        *reinterpret_cast<float4*>(smem + piece_off(w, k, 2 + it_hh, it_G)) =
            make_float4(B0.x, B0.y, B1.x, B1.y);
      }
      __syncwarp();
      uint4 na[4], nr[4];
      if (i + 1 < n) {
        const int64_t blk = PAGED ? blk_next : warp_block(i + 1);
        load_meta(i + 1, blk);
        load_codes(i + 1, blk, na, nr);
      }
      if (PAGED && i + 2 < n) blk_next = warp_block(i + 2);
      // this tensor's stage b is free once the scores (K^) or the output
      // (V^) of tile i-2 are done
      if (i >= 2)
        (void)wait_bar(&bars[(T ? kBVEmpty : kBKEmpty) + b], (uint32_t)((i - 2) >> 1) & 1u, abort_w);
      uint8_t* tile = smem + kStage + b * (2 * kTileBytes) + T * kTileBytes;
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const int G = 4 * gq + gi;
#pragma unroll
        for (int jc = 0; jc < 4; jc += (C16 ? 2 : 4)) {
          const int k = C16 ? (jc >> 1) : 0;
          const float4 A0 = *reinterpret_cast<const float4*>(smem + piece_off(w, k, 0, G));
          const float4 A1 = *reinterpret_cast<const float4*>(smem + piece_off(w, k, 1, G));
          const float4 B0 = *reinterpret_cast<const float4*>(smem + piece_off(w, k, 2, G));
          const float4 B1 = *reinterpret_cast<const float4*>(smem + piece_off(w, k, 3, G));
#pragma unroll
          for (int j = jc; j < jc + (C16 ? 2 : 4); ++j) {
            const uint32_t aw = gi == 0 ? ca[j].x : gi == 1 ? ca[j].y : gi == 2 ? ca[j].z : ca[j].w;
            const uint32_t rw = gi == 0 ? cr[j].x : gi == 1 ? cr[j].y : gi == 2 ? cr[j].z : cr[j].w;
            // byte k of E / O: the code of channel 8G + k / 8G + 4 + k
            const uint32_t E = ((aw << 4) & 0xf0f0f0f0u) | (rw & 0x0f0f0f0fu);
            const uint32_t O = (aw & 0xf0f0f0f0u) | ((rw >> 4) & 0x0f0f0f0fu);
            const f2 x01 = fma2(make_float2(lut<0>(E, lane_off), lut<1>(E, lane_off)),
                                make_float2(A0.x, A0.y), make_float2(B0.x, B0.y));
            const f2 x23 = fma2(make_float2(lut<2>(E, lane_off), lut<3>(E, lane_off)),
                                make_float2(A0.z, A0.w), make_float2(B0.z, B0.w));
            const f2 x45 = fma2(make_float2(lut<0>(O, lane_off), lut<1>(O, lane_off)),
                                make_float2(A1.x, A1.y), make_float2(B1.x, B1.y));
            const f2 x67 = fma2(make_float2(lut<2>(O, lane_off), lut<3>(O, lane_off)),
                                make_float2(A1.z, A1.w), make_float2(B1.z, B1.w));
            const int t = 32 * wr + t8 + 8 * j;
            *reinterpret_cast<uint4*>(tile + (t >> 3) * 2048 + G * 128 + (t & 7) * 16) =
                make_uint4(f2_to_bf2(x01.x, x01.y), f2_to_bf2(x23.x, x23.y),
                           f2_to_bf2(x45.x, x45.y), f2_to_bf2(x67.x, x67.y));
          }
        }
      }
      fence_proxy_async();  // the tile is read by the tensor core
      arrive(&bars[(T ? kBVFull : kBKFull) + b]);
      if (i + 1 < n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ca[j] = na[j];
          cr[j] = nr[j];
        }
      }
    }
  } else {
    // ================= softmax: thread = token 32q + lane of the tile
    const int q = w - kProdWarps;               // lane quarter of tensor memory
    const uint32_t tq = tm + ((uint32_t)(32 * q) << 16);
    const int t = 32 * q + lane;
    // shared by the four warps: red [4][32] row maxima of a tile per warp,
    // msm [32] the running row maxima, fsm [32] the factors of the last raise
    float* red = reinterpret_cast<float*>(smem + kRed);
    float* msm = red + kSoftWarps * RP;
    float* fsm = msm + RP;
    float ls[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) ls[r] = 0.f;
    bool o_waited = true;   // odone of the previous tile already waited for
    // S^T of tile i, issued by thread 0 once the tile's K^ is complete and
    // the tile two back has released its score buffer
    int s_next = 0;         // thread 0: the next tile whose scores are to be issued
    auto issue_s = [&](int i) {
      const int b = i & 1;
      (void)wait_bar(&bars[kBKFull + b], (uint32_t)(i >> 1) & 1u, abort_w);
      if (i >= 2) (void)wait_bar(&bars[kBSFree + b], (uint32_t)((i - 2) >> 1) & 1u, abort_w);
      fence_after();
      const uint32_t ka = smem_u32(smem + kStage + b * (2 * kTileBytes));  // K^ of stage b
      const uint32_t qa = smem_u32(smem + kQ + seg_of(i) * kQBytes);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k)
        umma(tm + kColS + 32 * b, sdesc(ka + 256 * k, 128, 2048), sdesc(qa + 256 * k, 128, 2048),
             kIdS, k > 0 ? 1u : 0u);
      umma_commit(&bars[kBSReady + b]);
      umma_commit(&bars[kBKEmpty + b]);
      s_next = i + 1;
    };
    auto try_issue_s = [&](int j) {   // thread 0: without waiting for K^
      if (s_next == j && j < n) {
        const int bk = j & 1;
        if (mbar_try_wait(&bars[kBKFull + bk], (uint32_t)(j >> 1) & 1u)) issue_s(j);
      }
    };
    for (int i = 0; i < n; ++i) {
      const int b = i & 1, sg = seg_of(i);
      if (q == 0 && lane == 0 && s_next == i) issue_s(i);
      const bool first = i == 0 || ti0 + i == a.NCH;       // a unit's first tile here
      const bool last = i == n - 1 || ti0 + i + 1 == a.NCH;  // a unit's last tile here
      (void)wait_bar(&bars[kBSReady + b], (uint32_t)(i >> 1) & 1u, abort_w);
      fence_after();
      uint32_t s[32];
      tmem_ld32(tq + kColS + 32 * b, s);
      tmem_wait_ld();
      fence_before();
      arrive(&bars[kBSFree + b]);
      // the next tile's scores go into the other buffer (released by the
      // softmax of tile i - 1), so they can be issued now if its K^ is ready
      if (q == 0 && lane == 0) try_issue_s(i + 1);
      float p[RP];
      float pm = 0.f;
#pragma unroll
      for (int r = 0; r < RP; r += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(msm + r);
        p[r] = ex2(__uint_as_float(s[r]) * a.scale_log2 - m4.x);
        p[r + 1] = ex2(__uint_as_float(s[r + 1]) * a.scale_log2 - m4.y);
        p[r + 2] = ex2(__uint_as_float(s[r + 2]) * a.scale_log2 - m4.z);
        p[r + 3] = ex2(__uint_as_float(s[r + 3]) * a.scale_log2 - m4.w);
        pm = fmaxf(fmaxf(pm, fmaxf(p[r], p[r + 1])), fmaxf(p[r + 2], p[r + 3]));
      }
      // vote of the four warps: does some weight of the tile exceed 2^8?
      // (a NaN weight counts: it only arises from a -inf maximum)
      const bool over = !(pm <= 0x1p8f);
      if (__any_sync(kFull, over) && lane == 0) misc[2 + i % 3] = 1u;
      asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");
      const bool raise = misc[2 + i % 3] != 0u;
      if (q == 0 && lane == 0) misc[2 + (i + 2) % 3] = 0u;   // next written at tile i + 2
      if (raise) {
        // the tile's row maxima over the 128 tokens: per warp by shuffles,
        // then across the four warps through shared memory
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          float v = __uint_as_float(s[r]) * a.scale_log2;
#pragma unroll
          for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
          if (lane == 0) red[q * RP + r] = v;
        }
        asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");
        if (q == 0) {   // lane r: the new maximum of row r and its factor
          const float mo = msm[lane];
          const float mn = fmaxf(fmaxf(mo, fmaxf(red[lane], red[RP + lane])),
                                 fmaxf(red[2 * RP + lane], red[3 * RP + lane]));
          fsm[lane] = ex2(mo - mn);   // 0 for a -inf maximum
          msm[lane] = mn;
        }
        asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");
        if (!first) {
          // rescale this lane's channel of the accumulator, hi then lo
          (void)wait_bar(&bars[kBODone], (uint32_t)(i - 1) & 1u, abort_w);
          o_waited = true;
          fence_after();
#pragma unroll
          for (int hl = 0; hl < 2; ++hl) {
            uint32_t o[32];
            tmem_ld32(tq + kColO + 32 * hl, o);
            tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < RP; r += 4) {
              const float4 f4 = *reinterpret_cast<const float4*>(fsm + r);
              o[r] = __float_as_uint(__uint_as_float(o[r]) * f4.x);
              o[r + 1] = __float_as_uint(__uint_as_float(o[r + 1]) * f4.y);
              o[r + 2] = __float_as_uint(__uint_as_float(o[r + 2]) * f4.z);
              o[r + 3] = __float_as_uint(__uint_as_float(o[r + 3]) * f4.w);
            }
            tmem_st32(tq + kColO + 32 * hl, o);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int r = 0; r < RP; r += 4) {
          const float4 f4 = *reinterpret_cast<const float4*>(fsm + r);
          const float4 m4 = *reinterpret_cast<const float4*>(msm + r);
          ls[r] *= f4.x;
          ls[r + 1] *= f4.y;
          ls[r + 2] *= f4.z;
          ls[r + 3] *= f4.w;
          p[r] = ex2(__uint_as_float(s[r]) * a.scale_log2 - m4.x);
          p[r + 1] = ex2(__uint_as_float(s[r + 1]) * a.scale_log2 - m4.y);
          p[r + 2] = ex2(__uint_as_float(s[r + 2]) * a.scale_log2 - m4.z);
          p[r + 3] = ex2(__uint_as_float(s[r + 3]) * a.scale_log2 - m4.w);
        }
      }
      // P^T: hi rows 0..31 then lo rows 32..63 of this token's column
      if (!o_waited) (void)wait_bar(&bars[kBODone], (uint32_t)(i - 1) & 1u, abort_w);
      uint8_t* pcol = smem + kP + (t >> 3) * 1024 + (t & 7) * 16;
#pragma unroll
      for (int jg = 0; jg < 4; ++jg) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = 8 * jg + 2 * k;
          ls[r] += p[r];
          ls[r + 1] += p[r + 1];
          hi[k] = f2_to_bf2(p[r], p[r + 1]);
          const f2 hf = bf2_to_f2(hi[k]);
          lo[k] = f2_to_bf2(p[r] - hf.x, p[r + 1] - hf.y);
        }
        *reinterpret_cast<uint4*>(pcol + jg * 128) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(pcol + (4 + jg) * 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async();
      fence_before();
      asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");   // P complete
      if (q == 0 && lane == 0) {
        // O^T += V^T [P_hi | P_lo]^T once V^ of the tile is complete; a unit's
        // first tile starts the accumulator
        (void)wait_bar(&bars[kBVFull + b], (uint32_t)(i >> 1) & 1u, abort_w);
        fence_after();
        const uint32_t va = smem_u32(smem + kStage + b * (2 * kTileBytes) + kTileBytes);
        const uint32_t pa = smem_u32(smem + kP);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma(tm + kColO, sdesc(va + 4096 * k, 2048, 128), sdesc(pa + 2048 * k, 1024, 128), kIdO,
               (k > 0 || !first) ? 1u : 0u);
        umma_commit(&bars[kBODone]);
        umma_commit(&bars[kBVEmpty + b]);
        // the next tile's scores, if not yet issued and its K^ is complete
        try_issue_s(i + 1);
      }
      o_waited = false;
      if (last) {
        // ---- the unit's partial: o (thread = channel t), l, m
        (void)wait_bar(&bars[kBODone], (uint32_t)i & 1u, abort_w);
        o_waited = true;
        fence_after();
        float* ps = a.part + (int64_t)(2 * cta + sg) * part_floats;
        {
          uint32_t oh[32], ol[32];
          tmem_ld32(tq + kColO, oh);
          tmem_ld32(tq + kColO + 32, ol);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < RP; ++r)
            ps[2 * RP + r * kD + t] = __uint_as_float(oh[r]) + __uint_as_float(ol[r]);
        }
        fence_before();
        // row sums over the 128 token threads, through the (now idle) P buffer
        float* lsm = reinterpret_cast<float*>(smem + kP);
#pragma unroll
        for (int r = 0; r < RP; r += 4)
          *reinterpret_cast<float4*>(lsm + t * RP + r) =
              make_float4(ls[r], ls[r + 1], ls[r + 2], ls[r + 3]);
        asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");
        if (q == 0) {
          float l = 0.f;
          for (int k = 0; k < kTile; ++k) l += lsm[k * RP + lane];
          ps[RP + lane] = l;
          ps[lane] = msm[lane];
          msm[lane] = -INFINITY;   // the next unit starts afresh
        }
        asm volatile("barrier.sync 2, %0;" :: "n"(kSoftThreads) : "memory");
#pragma unroll
        for (int r = 0; r < RP; ++r) ls[r] = 0.f;
      }
    }
    if (q == 0 && lane == 0) {
      // every commit's arrival has landed before tear-down (the last tile's
      // O was waited for in its epilogue)
      for (int i = n - 2 < 0 ? 0 : n - 2; i < n; ++i) {
        (void)wait_bar(&bars[kBVEmpty + (i & 1)], (uint32_t)(i >> 1) & 1u, abort_w);
        (void)wait_bar(&bars[kBKEmpty + (i & 1)], (uint32_t)(i >> 1) & 1u, abort_w);
      }
    }
  }

  // ---- tear-down: every MMA has completed (the softmax waited for the last
  // accumulation), so the tensor memory can go
  fence_before();
  __syncthreads();
  fence_after();
  if (w == kProdWarps)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tm),
                 "r"(kTmemCols) : "memory");
  // the split combine may launch now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ wait self-test

// This kernel's wait on mbarriers that nothing arrives on (the producer is
// absent): warp 0 waits with limit_ns and must give up, raise the abort word
// and record kFlagWaitTimeout; warp 1 starts half a limit later with the full
// limit and must return unsatisfied once the abort word is up, well before
// its own limit.  *status = 3 if both held, else 4.  The flag word is the
// CTA's own, not the library's.
__global__ void __launch_bounds__(64, 1)
tc_wait_selftest_kernel(uint64_t limit_ns, unsigned int* status) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t abort_w, good;
  __shared__ unsigned int flags;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_w = 0u;
    flags = 0u;
    good = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = global_ns();
  if (w == 0) {
    const bool ok = tc::wait_bar_for(&bars[0], 0, &abort_w, limit_ns, &flags);
    if (lane == 0 && !ok && abort_w) atomicAdd(&good, 1u);
  } else {
    while (global_ns() - t0 < limit_ns / 2) {
    }
    const uint64_t t1 = global_ns();
    const bool ok = tc::wait_bar_for(&bars[1], 0, &abort_w, kWaitNs, &flags);
    if (lane == 0 && !ok && global_ns() - t1 < 2 * limit_ns) atomicAdd(&good, 1u);
  }
  __syncthreads();
  if (threadIdx.x == 0) *status = (good == 2u && (flags & kFlagWaitTimeout)) ? 3u : 4u;
}

cudaError_t launch_tc_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t stream) {
  tc_wait_selftest_kernel<<<1, 64, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host

// One CTA per SM (capped at 256): equal shares of the flattened (unit, tile)
// space, at least one CTA per unit so that a share spans at most two units.
int attn_tc_ctas(int batch, int Hkv, int nrg, int64_t ntiles, int sms) {
  const int64_t units = (int64_t)batch * Hkv * nrg;
  const int64_t total = units * ntiles;
  int64_t n = sms < 256 ? sms : 256;
  if (n > total) n = total;
  if (n < units) n = units;
  return (int)n;
}

template <bool PAGED, bool C16>
static cudaError_t run_attn_tc(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  auto fn = attn_tc_kernel<PAGED, C16>;
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    int reserved = -1;
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    if (reserved != (int)kSmemBase) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  fn<<<(unsigned)prm.n_cta, tc::kThreads, tc::kSmem, stream>>>(prm, tab);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_attn_combine(prm, tc::kRows, stream);
}

cudaError_t launch_attn_tc(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream) {
  const bool c16 = prm.C < 32;
  if (prm.bt) return c16 ? run_attn_tc<true, true>(prm, tab, stream)
                         : run_attn_tc<true, false>(prm, tab, stream);
  return c16 ? run_attn_tc<false, true>(prm, tab, stream)
             : run_attn_tc<false, false>(prm, tab, stream);
}

}  // namespace lynx
