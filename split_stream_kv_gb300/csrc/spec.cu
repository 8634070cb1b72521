// spec.cu -- speculative verification and correction of "Lynx: Progressive
// Speculative KV Cache Transfer for Disaggregated LLM Inference" (technical
// review, Mechanism 3, Eq. 10 and Eq. 11), one CTA per sequence.
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
// The 32 warps of the CTA each own a contiguous segment of the vocabulary:
// one coalesced pass gives the segment totals; the warp whose segment holds
// the target rescans it 32 tokens at a time with a warp-wide prefix sum.
#include "common.cuh"
#include "internal.h"

namespace lynx {

constexpr int kSpecThreads = 1024;
constexpr int kSpecWarps = kSpecThreads / 32;

// Set when a draft token lay outside [0, V) (treated as rejected); read
// through read_spec_flags(), never reset.
__device__ unsigned int g_spec_flags = 0;

cudaError_t read_spec_flags(unsigned int* flag) {
  return cudaMemcpyFromSymbol(flag, g_spec_flags, sizeof(unsigned int));
}

__device__ __forceinline__ uint64_t spec_weight(float w) {
  return w > 0.0f ? __float2ull_rz(w * 1099511627776.0f) : 0ull;  // floor(w * 2^40)
}

__global__ void __launch_bounds__(kSpecThreads)
spec_verify_kernel(const float* __restrict__ p, const float* __restrict__ q,
                   const int32_t* __restrict__ s, const float* __restrict__ u,
                   const uint32_t* __restrict__ rs, const int T, const int64_t V,
                   int32_t* __restrict__ n_acc, int32_t* __restrict__ next_tok) {
  __shared__ unsigned long long wtot[kSpecWarps];
  __shared__ int k_sh, seg_w, done;
  __shared__ unsigned long long base_sh, target_sh;
  const int b = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;

  // ---- Eq. 10: the accepted prefix (warp 0, 32 positions at a time)
  if (w == 0) {
    int k = T;
    for (int t0 = 0; t0 < T; t0 += 32) {
      const int t = t0 + lane;
      bool reject = false;
      if (t < T) {
        const int64_t x = s[(int64_t)b * T + t];
        if (x < 0 || x >= V) {
          atomicOr(&g_spec_flags, kFlagBadToken);
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
    if (lane == 0) {
      k_sh = k;
      done = 0;
    }
  }
  __syncthreads();
  const int k = k_sh;
  const float* pk = p + ((int64_t)b * (T + 1) + k) * V;
  const float* qk = k < T ? q + ((int64_t)b * T + k) * V : nullptr;
  const uint32_t r = rs[b];
  const int64_t seg = (V + kSpecWarps - 1) / kSpecWarps;
  const int64_t x0 = (int64_t)w * seg, x1 = x0 + seg < V ? x0 + seg : V;

  // ---- Eq. 11 (or p_{T+1}); with zero total weight, the weights of p
  for (int pass = 0; pass < 2; ++pass) {
    const float* qw = pass == 0 ? qk : nullptr;
    auto weight = [&](int64_t x) -> uint64_t {
      const float pv = __ldg(pk + x);
      return spec_weight(qw ? fmaxf(__fsub_rn(pv, __ldg(qw + x)), 0.0f) : pv);
    };
    unsigned long long acc = 0;
    for (int64_t x = x0 + lane; x < x1; x += 32) acc += weight(x);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if (lane == 0) wtot[w] = acc;
    __syncthreads();
    if (tid == 0) {
      unsigned long long Z = 0;
      for (int i = 0; i < kSpecWarps; ++i) Z += wtot[i];
      if (Z != 0) {
        // floor(r * Z / 2^32) exactly: r * Zhi + floor(r * Zlo / 2^32)
        const unsigned long long target =
            (unsigned long long)r * (Z >> 32) + (((unsigned long long)r * (Z & 0xffffffffull)) >> 32);
        unsigned long long run = 0;
        int ws = kSpecWarps - 1;
        for (int i = 0; i < kSpecWarps; ++i) {
          if (run + wtot[i] > target) {
            ws = i;
            break;
          }
          run += wtot[i];
        }
        seg_w = ws;
        base_sh = run;
        target_sh = target;
        done = 1;
      }
    }
    __syncthreads();
    if (done) {
      if (w == seg_w) {
        const unsigned long long target = target_sh;
        unsigned long long run = base_sh;
        int32_t tok = (int32_t)(x1 - 1);
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
            tok = (int32_t)(xs + __ffs(hit) - 1);
            break;
          }
          run += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0) {
          n_acc[b] = k;
          next_tok[b] = tok;
        }
      }
      return;
    }
  }
  if (tid == 0) {
    n_acc[b] = k;
    next_tok[b] = -1;
  }
}

cudaError_t launch_spec_verify(const float* p, const float* q, const int32_t* s, const float* u,
                               const uint32_t* r, int batch, int T, int64_t V, int32_t* n_acc,
                               int32_t* next_tok, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  spec_verify_kernel<<<(unsigned)batch, kSpecThreads, 0, stream>>>(p, q, s, u, r, T, V, n_acc,
                                                                    next_tok);
  return cudaGetLastError();
}

}  // namespace lynx
