// internal.h -- host-side interfaces between the C ABI and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lynx {

// Stage-3 tables for one alpha, built on the host in float64.
struct CompanderTable {
  float alpha;
  float c16;        // 65536 * 127 / log2(1 + alpha), float32
  float thr[128];   // thr[k] = smallest float32 a with Round(Y(a)) > k; thr[127] = +inf
};

// Reconstruction magnitudes X(I) = ((1+alpha)^(I/127) - 1)/alpha, I = 0..127.
struct ExpandTable {
  float x[128];
};

// Fast-path rounding window of the encoder, in units of 2^-16 of Y:
// results within this distance of a half-integer take the exact path.  The
// fast path's error grows with c16 = 65536 * 127 / log2(1 + alpha); over all
// float32 inputs it stays below 2 units for every alpha >= 1 checked (largest
// at alpha = 1), so the encoder accepts alpha >= 1 and keeps a window of
// twice that.
constexpr uint32_t kAmbiguityK = 4;
constexpr float kMinEncodeAlpha = 1.0f;

struct Shape {
  int64_t B, L;
  int H, D, page, C;
  int64_t NB() const { return L / page; }
  int64_t blocks() const { return B * NB() * H; }
  int NC() const { return page / C; }
};

// Page-block addressing of the streams: dense (no table; block (b, p, h) at
// index (b*NB + p)*H + h) or through a block table [B][NB] of physical pages
// in [0, nphys), each holding the H head blocks of one page.
struct Paging {
  const int32_t* table = nullptr;
  int64_t nphys = 0;
};

// Launchers: validated arguments, enqueue on `stream`, return a cudaError_t.
cudaError_t launch_encode(const void* kv, const Shape& s, const CompanderTable& tab,
                          void* anchor, void* residual, float* meta, cudaStream_t stream,
                          const Paging& pg = Paging());
cudaError_t launch_decode(const void* anchor, const void* residual, const float* meta,
                          const Shape& s, const ExpandTable& tab, void* out, bool bf16_out,
                          cudaStream_t stream, const Paging& pg = Paging());
// Anchor-only decode of a k-bit Anchor stream (3 <= k <= 6), see variants.cu.
cudaError_t launch_decode_anchor_bits(const void* anchor_k, const float* meta, const Shape& s,
                                      int k, const ExpandTable& tab, void* out, bool bf16_out,
                                      cudaStream_t stream);
// The Appendix A.1 variant (variants.cu): meta = m [D], then m_i [P/16][D]
// per block; residual may be null for the Anchor-only decode.
cudaError_t launch_a1_encode(const void* kv, const Shape& s, const CompanderTable& tab,
                             void* anchor, void* residual, float* meta, cudaStream_t stream);
cudaError_t launch_a1_decode(const void* anchor, const void* residual, const float* meta,
                             const Shape& s, const ExpandTable& tab, void* out, bool bf16_out,
                             cudaStream_t stream);
cudaError_t launch_compander_selfcheck(const CompanderTable& tab, uint64_t* counts,
                                       cudaStream_t stream);

struct AttnArgs {
  const void* q;
  int batch, T, H_q;
  const void *k_anchor, *k_residual;
  const float* k_meta;
  const void *v_anchor, *v_residual;
  const float* v_meta;
  Shape s;           // B = batch
  bool full;
  float* out;
  void* workspace;
  // optional: the draft tokens' own keys and values [batch][T][H_kv][D] BF16;
  // query token t then also attends to draft tokens 0..t
  const void* k_tail = nullptr;
  const void* v_tail = nullptr;
  Paging paging;  // of k_* and v_* (both use the same block table)
};
size_t attn_workspace_bytes(int batch, int T, int H_q, int H_kv, int64_t L);
cudaError_t launch_attn(const AttnArgs& a, const ExpandTable& tab, cudaStream_t stream);

// Record `msg` as this thread's last error and return `code`.
int report_error(int code, const char* msg);

// Host read of the device flag set when a bounded wait gave up.
cudaError_t read_wait_timeout(unsigned int* flag);
cudaError_t read_decode_wait_timeout(unsigned int* flag);
cudaError_t read_variant_wait_timeout(unsigned int* flag);
cudaError_t read_attn_flags(unsigned int* flag);
cudaError_t read_spec_flags(unsigned int* flag);
cudaError_t launch_spec_verify(const float* p, const float* q, const int32_t* s, const float* u,
                               const uint32_t* r, int batch, int T, int64_t V, int32_t* n_acc,
                               int32_t* next_tok, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int sm_count();

}  // namespace lynx
