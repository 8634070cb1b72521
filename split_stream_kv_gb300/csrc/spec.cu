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
// vocabulary; one coalesced pass gives the segment totals, shared through
// distributed shared memory; the warp whose segment holds the target rescans
// it 32 tokens at a time with a warp-wide prefix sum.
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

// Set when a draft token lay outside [0, V) (treated as rejected); read
// through read_spec_flags(), never reset.
__device__ unsigned int g_spec_flags = 0;

cudaError_t read_spec_flags(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_spec_flags, sizeof(unsigned int));
}

__device__ __forceinline__ uint64_t spec_weight(float w) {
  return w > 0.0f ? __float2ull_rz(w * 1099511627776.0f) : 0ull;  // floor(w * 2^40)
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

__global__ void __cluster_dims__(kSpecCtas, 1, 1) __launch_bounds__(kSpecThreads)
spec_verify_kernel(const float* __restrict__ p, const float* __restrict__ q,
                   const int32_t* __restrict__ s, const float* __restrict__ u,
                   const uint32_t* __restrict__ rs, const int T, const int64_t V,
                   int32_t* __restrict__ n_acc, int32_t* __restrict__ next_tok) {
  __shared__ unsigned long long wtot[2][kSpecWarps];  // per pass: this CTA's segment totals
  __shared__ unsigned long long all[kSpecSegs];
  __shared__ int k_sh, seg_sh, done;
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
  int32_t result = -1;
  bool have = false;

  // ---- Eq. 11 (or p_{T+1}); with zero total weight, the weights of p
  for (int pass = 0; pass < 2 && !have; ++pass) {
    const float* qw = pass == 0 ? qk : nullptr;
    auto weight = [&](int64_t x) -> uint64_t {
      const float pv = __ldg(pk + x);
      return spec_weight(qw ? fmaxf(__fsub_rn(pv, __ldg(qw + x)), 0.0f) : pv);
    };
    unsigned long long acc = 0;
    for (int64_t x = x0 + lane; x < x1; x += 32) acc += weight(x);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if (lane == 0) wtot[pass][w] = acc;
    cluster_sync_all();                                // every CTA's totals are written
    for (int i = tid; i < kSpecSegs; i += kSpecThreads)
      all[i] = ld_peer_u64(&wtot[pass][i % kSpecWarps], (uint32_t)(i / kSpecWarps));
    __syncthreads();
    if (tid == 0) {
      unsigned long long Z = 0;
      for (int i = 0; i < kSpecSegs; ++i) Z += all[i];
      done = Z != 0;
      if (Z != 0) {
        // floor(r * Z / 2^32) exactly: r * Zhi + floor(r * Zlo / 2^32)
        const unsigned long long target =
            (unsigned long long)r * (Z >> 32) + (((unsigned long long)r * (Z & 0xffffffffull)) >> 32);
        unsigned long long run = 0;
        int sg = kSpecSegs - 1;
        for (int i = 0; i < kSpecSegs; ++i) {
          if (run + all[i] > target) {
            sg = i;
            break;
          }
          run += all[i];
        }
        seg_sh = sg;
        base_sh = run;
        target_sh = target;
      }
    }
    __syncthreads();
    if (done) {
      have = true;
      if (gseg == seg_sh) {                           // this warp's segment holds the target
        const unsigned long long target = target_sh;
        unsigned long long run = base_sh;
        result = (int32_t)(x1 - 1);
        for (int64_t xs = x0; xs < x1; xs += 32) {
          const int64_t x = xs + lane;
          unsigned long long v = x < x1 ? weight(x) : 0ull;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {  // inclusive prefix sum over the lanes
            const unsigned long long n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
          }
          const unsigned hit = __ballot_sync(kFull, x < x1 && run + v > target);
          if (hit) {
            result = (int32_t)(xs + __ffs(hit) - 1);
            break;
          }
          run += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0) {
          n_acc[b] = k;
          next_tok[b] = result;
        }
      }
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
