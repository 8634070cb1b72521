// spec.cu -- speculative verification and correction of "Lynx: Progressive
// Speculative KV Cache Transfer for Disaggregated LLM Inference" (technical
// review, Mechanism 3, Eq. 10 and Eq. 11), one cluster of CTAs per sequence.
//
// Draft token s_t (t = 1..T) is accepted with probability min(1, p_t(s_t) /
// q_t(s_t)) (Eq. 10), tested as u_t * q_t(s_t) < p_t(s_t) in float32; the
// accepted prefix ends at the first rejection.  The next token is drawn from
// max(0, p_{k+1} - q_{k+1}) at the first rejected position (Eq. 11), or from
// p_{T+1} when the whole draft is accepted.  The draw is an inverse CDF over
// integer weights W(x) = floor(w(x) * 2^40) with target floor(r * Z / 2^32),
// Z = sum W: the smallest x whose running sum exceeds the target.  Integer
// sums make the token independent of the summation order.
//
// A cluster of CTAs per sequence: every warp owns a contiguous segment of the
// vocabulary; one pass, with all of a lane's loads in flight at once, gives
// the segment totals in exact integer arithmetic, shared through distributed
// shared memory; one warp finds the segment holding the target with a prefix
// sum over the totals, and the CTA owning that segment rescans it, two tokens
// a thread, with a block-wide prefix sum.
#include "common.cuh"
#include "internal.h"

namespace lynx {

// A sequence is one cluster of kSpecCtas CTAs (thread-block cluster with
// distributed shared memory); CTA c owns vocabulary slice c, each of its
// warps a contiguous segment of the slice.
constexpr int kSpecCtas = 8;
constexpr int kSpecThreads = 512;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kSpecSegs = kSpecCtas * kSpecWarps;  // segments of the vocabulary
constexpr int kSpecPerLane = 32;  // tokens a lane loads at once

// Set when a draft token lay outside [0, V) (treated as rejected); read
// through read_spec_flags(), never reset.
__device__ unsigned int g_spec_flags = 0;

cudaError_t read_spec_flags(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_spec_flags, sizeof(unsigned int));
}

// Weights W(x) = floor(w * 2^40) of a float w, two ways.  spec_weight_int
// reads W off the bits of w: w = M * 2^(E - 150) with M the 24-bit significand
// (implicit bit included; subnormals have E = 1 and none), so W = M * 2^(E-110)
// (saturating at 2^64 - 1 from w = 2^24 on).  For 0 <= w < 8 the split form is
// cheaper: W = A * 2^20 + L with A = floor(w * 2^20) and L = floor(f * 2^20),
// f = w * 2^20 - A; each of A and L is read off the bits of 2^23 + (value)
// rounded toward zero, where one unit in the last place is 1, so their sums
// accumulate in 32-bit integers with the 2^23 bias taken out once.
__device__ __forceinline__ uint64_t spec_weight_int(float w) {
  if (!(w > 0.0f)) return 0ull;
  const uint32_t bits = __float_as_uint(w), e = bits >> 23;
  const uint32_t m = e ? (bits & 0x7fffffu) | 0x800000u : bits;
  const int sh = (int)(e ? e : 1u) - 110;
  if (sh >= 0) return sh > 40 ? ~0ull : (uint64_t)m << sh;
  return sh <= -24 ? 0ull : (uint64_t)(m >> -sh);
}
constexpr float kTwo20 = 1048576.0f, kTwo23 = 8388608.0f;
constexpr uint32_t kBias = 0x4B000000u;  // the bits of 2^23
constexpr float kSplitMax = 8.0f;        // the split form holds below this
// the biased bits of 2^23 + A and 2^23 + L for 0 <= w < kSplitMax
__device__ __forceinline__ void spec_parts(float w, uint32_t& ab, uint32_t& lb) {
  const float t1 = __fmaf_rz(w, kTwo20, kTwo23);
  const float f = __fmaf_rn(w, kTwo20, -__fsub_rn(t1, kTwo23));  // exact
  ab = __float_as_uint(t1);
  lb = __float_as_uint(__fmaf_rz(f, kTwo20, kTwo23));
}
__device__ __forceinline__ uint64_t spec_weight(float w) {
  if (!(w < kSplitMax)) return spec_weight_int(w);
  uint32_t ab, lb;
  spec_parts(fmaxf(w, 0.0f), ab, lb);
  return ((uint64_t)(ab - kBias) << 20) + (lb - kBias);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Read a 64-bit word at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ unsigned long long ld_peer_u64(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote) : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__global__ void __cluster_dims__(kSpecCtas, 1, 1) __launch_bounds__(kSpecThreads)
spec_verify_kernel(const float* __restrict__ p, const float* __restrict__ q,
                   const int32_t* __restrict__ s, const float* __restrict__ u,
                   const uint32_t* __restrict__ rs, const int T, const int64_t V,
                   int32_t* __restrict__ n_acc, int32_t* __restrict__ next_tok) {
  __shared__ unsigned long long wtot[2][kSpecWarps];  // per pass: this CTA's segment totals
  __shared__ unsigned long long all[kSpecSegs];
  static_assert(kSpecSegs % 32 == 0, "segments split evenly over a warp");
  __shared__ unsigned long long wsum[kSpecWarps];
  __shared__ int k_sh, seg_sh, done, found;
  __shared__ int32_t result_sh;
  __shared__ unsigned long long base_sh, target_sh;
  const uint32_t crank = cluster_rank();
  const int b = blockIdx.x / kSpecCtas, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;

  // ---- Eq. 10: the accepted prefix (warp 0 of every CTA, 32 positions at a time)
  if (w == 0) {
    int k = T;
    for (int t0 = 0; t0 < T; t0 += 32) {
      const int t = t0 + lane;
      bool reject = false;
      if (t < T) {
        const int64_t x = s[(int64_t)b * T + t];
        if (x < 0 || x >= V) {
          if (crank == 0) atomicOr(&g_spec_flags, kFlagBadToken);
          reject = true;
        } else {
          const float pv = p[((int64_t)b * (T + 1) + t) * V + x];
          const float qv = q[((int64_t)b * T + t) * V + x];
          reject = !(__fmul_rn(u[(int64_t)b * T + t], qv) < pv);
        }
      }
      const unsigned m = __ballot_sync(kFull, reject);
      if (m) {
        k = t0 + __ffs(m) - 1;
        break;
      }
    }
    if (lane == 0) k_sh = k;
  }
  __syncthreads();
  const int k = k_sh;
  const float* pk = p + ((int64_t)b * (T + 1) + k) * V;
  const float* qk = k < T ? q + ((int64_t)b * T + k) * V : nullptr;
  const uint32_t r = rs[b];
  const int64_t seg = (V + kSpecSegs - 1) / kSpecSegs;
  const int gseg = (int)crank * kSpecWarps + w;       // this warp's segment
  const int64_t x0 = (int64_t)gseg * seg < V ? (int64_t)gseg * seg : V;
  const int64_t x1 = x0 + seg < V ? x0 + seg : V;

  // A segment of up to 32 * kSpecPerLane tokens is read with all of a lane's
  // loads in flight at once; longer ones stream.
  const bool batched = seg <= 32 * kSpecPerLane;

  // ---- Eq. 11 (or p_{T+1}); with zero total weight, the weights of p
  bool have = false;
  for (int pass = 0; pass < 2 && !have; ++pass) {
    const bool resid = pass == 0 && qk;                // max(0, p - q) rather than p
    auto wval = [&](int64_t x) -> float {            // the float weight of token x
      const float pv = __ldg(pk + x), qv = resid ? __ldg(qk + x) : 0.0f;
      return resid ? fmaxf(__fsub_rn(pv, qv), 0.0f) : fmaxf(pv, 0.0f);
    };
    // this warp's segment total, split form; any weight past its range sends
    // the warp through the integer form
    unsigned long long acc = 0;
    float mx = 0.0f;
    if (batched) {
      // out-of-segment lanes read token 0 of the row and drop it
      float wv[kSpecPerLane];
      if (resid) {
        float qv[kSpecPerLane];
#pragma unroll
        for (int i = 0; i < kSpecPerLane; ++i) {
          const int64_t x = x0 + 32 * i + lane, xi = x < x1 ? x : 0;
          wv[i] = __ldg(pk + xi);
          qv[i] = __ldg(qk + xi);
        }
#pragma unroll
        for (int i = 0; i < kSpecPerLane; ++i)
          wv[i] = x0 + 32 * i + lane < x1 ? fmaxf(__fsub_rn(wv[i], qv[i]), 0.0f) : 0.0f;
      } else {
#pragma unroll
        for (int i = 0; i < kSpecPerLane; ++i) {
          const int64_t x = x0 + 32 * i + lane, xi = x < x1 ? x : 0;
          wv[i] = __ldg(pk + xi);
        }
#pragma unroll
        for (int i = 0; i < kSpecPerLane; ++i)
          wv[i] = x0 + 32 * i + lane < x1 ? fmaxf(wv[i], 0.0f) : 0.0f;
      }
      uint32_t sa = 0, sl = 0;
#pragma unroll
      for (int i = 0; i < kSpecPerLane; ++i) {
        mx = fmaxf(mx, wv[i]);
        uint32_t ab, lb;
        spec_parts(wv[i], ab, lb);
        sa += ab;
        sl += lb;
      }
      acc = ((unsigned long long)(sa - kSpecPerLane * kBias) << 20) + (sl - kSpecPerLane * kBias);
    } else {
      // (32-bit part sums fold into the total every 256 tokens a lane: A < 2^23)
      for (int64_t xb = x0 + lane; xb < x1; xb += 32 * 256) {
        const int64_t xe = xb + 32 * 256 < x1 ? xb + 32 * 256 : x1;
        uint32_t sa = 0, sl = 0, cnt = 0;
        for (int64_t x = xb; x < xe; x += 32) {
          const float wv = wval(x);
          mx = fmaxf(mx, wv);
          uint32_t ab, lb;
          spec_parts(wv, ab, lb);
          sa += ab;
          sl += lb;
          ++cnt;
        }
        acc += ((unsigned long long)(sa - cnt * kBias) << 20) + (sl - cnt * kBias);
      }
    }
    if (__any_sync(kFull, !(mx < kSplitMax))) {
      acc = 0;
      for (int64_t x = x0 + lane; x < x1; x += 32) acc += spec_weight(wval(x));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if (lane == 0) wtot[pass][w] = acc;
    cluster_sync_all();                                // every CTA's totals are written
    for (int i = tid; i < kSpecSegs; i += kSpecThreads)
      all[i] = ld_peer_u64(&wtot[pass][i % kSpecWarps], (uint32_t)(i / kSpecWarps));
    __syncthreads();
    if (w == 0) {
      // Lane l holds segments kPerLane*l .. kPerLane*l + kPerLane-1; a prefix
      // sum of the lane totals gives Z and the lane, then the segment, whose
      // running sum first exceeds the target.
      constexpr int kPerLane = kSpecSegs / 32;
      unsigned long long part[kPerLane], own = 0;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        part[i] = all[kPerLane * lane + i];
        own += part[i];
      }
      const unsigned long long inc = warp_incl_scan(own, lane);
      const unsigned long long Z = __shfl_sync(kFull, inc, 31);
      if (lane == 0) done = Z != 0;
      if (Z != 0) {
        // floor(r * Z / 2^32) exactly: r * Zhi + floor(r * Zlo / 2^32); below Z
        const unsigned long long target =
            (unsigned long long)r * (Z >> 32) + (((unsigned long long)r * (Z & 0xffffffffull)) >> 32);
        const int owner = __ffs(__ballot_sync(kFull, inc > target)) - 1;
        if (lane == owner) {
          unsigned long long run = inc - own;
          int sg = kPerLane * lane + kPerLane - 1;
#pragma unroll
          for (int i = 0; i < kPerLane; ++i) {
            if (run + part[i] > target) {
              sg = kPerLane * lane + i;
              break;
            }
            run += part[i];
          }
          seg_sh = sg;
          base_sh = run;
          target_sh = target;
        }
      }
    }
    __syncthreads();
    if (!done) continue;
    have = true;
    if ((int)crank != seg_sh / kSpecWarps) continue;
    // ---- the CTA holding the target segment rescans it, 2 tokens a thread
    // per round: the first token whose running sum exceeds the target
    const int64_t xs0 = (int64_t)seg_sh * seg < V ? (int64_t)seg_sh * seg : V;
    const int64_t xs1 = xs0 + seg < V ? xs0 + seg : V;
    const unsigned long long target = target_sh;
    unsigned long long base = base_sh;
    if (tid == 0) {
      result_sh = (int32_t)(xs1 - 1);
      found = 0;
    }
    for (int64_t c0 = xs0; c0 < xs1; c0 += 2 * kSpecThreads) {
      const int64_t xa = c0 + 2 * tid, xb = xa + 1;
      const unsigned long long wa = xa < xs1 ? spec_weight(wval(xa)) : 0ull;
      const unsigned long long wb = xb < xs1 ? spec_weight(wval(xb)) : 0ull;
      const unsigned long long inc = warp_incl_scan(wa + wb, lane);
      if (lane == 31) wsum[w] = inc;
      __syncthreads();
      unsigned long long before = base, total = 0;
#pragma unroll
      for (int i = 0; i < kSpecWarps; ++i) {
        const unsigned long long v = wsum[i];
        if (i < w) before += v;
        total += v;
      }
      const unsigned long long run = before + inc - (wa + wb);   // before token xa
      if (run <= target && target < run + wa + wb) {             // one thread at most
        result_sh = (int32_t)(target < run + wa ? xa : xb);
        found = 1;
      }
      __syncthreads();
      if (found) break;
      base += total;
    }
    if (tid == 0) {
      n_acc[b] = k;
      next_tok[b] = result_sh;
    }
  }
  if (!have && crank == 0 && tid == 0) {
    n_acc[b] = k;
    next_tok[b] = -1;
  }
  cluster_sync_all();  // peers may still read this CTA's totals
}

cudaError_t launch_spec_verify(const float* p, const float* q, const int32_t* s, const float* u,
                               const uint32_t* r, int batch, int T, int64_t V, int32_t* n_acc,
                               int32_t* next_tok, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  spec_verify_kernel<<<(unsigned)(batch * kSpecCtas), kSpecThreads, 0, stream>>>(
      p, q, s, u, r, T, V, n_acc, next_tok);
  return cudaGetLastError();
}

}  // namespace lynx
