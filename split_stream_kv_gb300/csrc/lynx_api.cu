// lynx_api.cu -- the extern "C" boundary declared in include/lynx.h: argument
// checks, the float64 alpha tables, and dispatch to the kernel launchers.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "lynx.h"

namespace lynx {

static thread_local char g_last_error[256] = "";

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }

static int cuda_fail(cudaError_t e, const char* what) {
  return fail(LYNX_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count() {
  static thread_local int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

// ---------------------------------------------------------- alpha tables

// Round(Y(a)) of Eq. 7 with Y in float64: 127 ln(1 + alpha a) / ln(1 + alpha).
static int round_code(float a, double al) {
  const double y = 127.0 * log1p(al * (double)a) / log1p(al);
  double r = floor(y + 0.5);
  if (r < 0.0) r = 0.0;
  if (r > 127.0) r = 127.0;
  return (int)r;
}

static void build_thresholds(float alpha, float thr[128]) {
  const double al = (double)alpha;
  const double lal = log1p(al);
  for (int k = 0; k < 127; ++k) {
    // smallest float a >= 0 with Round(Y(a)) >= k + 1: start at the real
    // boundary X(k + 1/2) and walk float neighbours until it is exact
    float c = (float)(expm1((k + 0.5) * lal / 127.0) / al);
    if (!(c >= 0.0f)) c = 0.0f;
    if (c > 1.0f) c = 1.0f;
    if (round_code(c, al) >= k + 1) {
      while (c > 0.0f) {
        const float prev = nextafterf(c, 0.0f);
        if (round_code(prev, al) >= k + 1) c = prev; else break;
      }
    } else {
      while (c < 1.0f && round_code(c, al) < k + 1) c = nextafterf(c, 2.0f);
    }
    thr[k] = c;
  }
  thr[127] = INFINITY;
}

static void build_expand(float alpha, float x[128]) {
  const double al = (double)alpha;
  for (int I = 0; I < 128; ++I) x[I] = (float)((pow(1.0 + al, (double)I / 127.0) - 1.0) / al);
}

// Per-thread cache of the last alpha's tables (building them costs a few us).
struct AlphaCache {
  uint32_t bits = 0xffffffffu;
  CompanderTable comp;
  ExpandTable expand;
};
static const AlphaCache& tables_for(float alpha) {
  static thread_local AlphaCache cache;
  uint32_t b;
  memcpy(&b, &alpha, 4);
  if (b != cache.bits) {
    cache.comp.alpha = alpha;
    cache.comp.c16 = (float)(65536.0 * 127.0 / log2(1.0 + (double)alpha));
    build_thresholds(alpha, cache.comp.thr);
    build_expand(alpha, cache.expand.x);
    cache.bits = b;
  }
  return cache;
}

// ---------------------------------------------------------- validation

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_alpha(float alpha) {
  if (!(alpha > 0.0f) || !isfinite(alpha)) return fail(LYNX_EINVAL, "alpha must be finite and > 0");
  return LYNX_OK;
}

// The encoder's fast Stage-3 rounding is exact (with its window) for alpha >= 1.
static int check_encode_alpha(float alpha) {
  int rc = check_alpha(alpha);
  if (rc) return rc;
  if (alpha < kMinEncodeAlpha)
    return fail(LYNX_EUNSUPPORTED, "alpha = %g: the encoder is built for alpha >= 1", alpha);
  return LYNX_OK;
}

// Pages of 64 ... 512 tokens for the Algorithm 1 codec (encode, both
// decoders, the k-bit Anchor decode); the attention kernel and the
// Appendix A.1 variant are built for pages up to 256.
static int check_codec_shape(int64_t B, int64_t L, int H, int D, int page, int C,
                             int max_page = 512) {
  if (B < 0 || L < 0 || H <= 0) return fail(LYNX_ESHAPE, "need B >= 0, L >= 0, H_kv >= 1");
  if (D != kD) return fail(LYNX_EUNSUPPORTED, "D = %d: only D = 128 is built", D);
  if ((page != 64 && page != 128 && page != 256 && page != 512) || page > max_page)
    return fail(LYNX_EUNSUPPORTED, "page = %d: built for 64 ... %d (powers of two)", page,
                max_page);
  if (C <= 0 || (C & (C - 1))) return fail(LYNX_ESHAPE, "C = %d must be a power of two", C);
  if (C < 16 || C > 128 || C > page)
    return fail(LYNX_EUNSUPPORTED, "C = %d: built for 16..128 and C <= page", C);
  if (L % page) return fail(LYNX_ESHAPE, "L = %lld is not a multiple of page = %d", (long long)L, page);
  if (B * L > (int64_t)0x7fffffff) return fail(LYNX_EUNSUPPORTED, "B*L must be < 2^31 tokens");
  return LYNX_OK;
}

static int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (!p) return fail(LYNX_EINVAL, "null pointer");
    if (!aligned16(p)) return fail(LYNX_EINVAL, "pointer not 16-byte aligned");
  }
  return LYNX_OK;
}

static void codec_sizes(int64_t B, int64_t L, int H, int D, int page, int C, size_t* a,
                        size_t* r, size_t* m) {
  const size_t elems = (size_t)B * (size_t)L * (size_t)H * (size_t)D;
  const size_t blocks = (size_t)B * (size_t)(L / page) * (size_t)H;
  if (a) *a = elems / 2;
  if (r) *r = elems / 2;
  if (m) *m = blocks * (size_t)(2 + 2 * (page / C)) * (size_t)D * sizeof(float);
}

}  // namespace lynx

using namespace lynx;

extern "C" {

const char* lynx_status_string(int code) {
  switch (code) {
    case LYNX_OK: return "ok";
    case LYNX_EINVAL: return "invalid argument";
    case LYNX_ESHAPE: return "inconsistent shape";
    case LYNX_EUNSUPPORTED: return "unsupported configuration";
    case LYNX_ECUDA: return "CUDA error";
    case LYNX_EWORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

const char* lynx_last_error(void) { return g_last_error; }

int lynx_encoded_sizes(int64_t B, int64_t L, int H_kv, int D, int page, int C,
                       size_t* anchor_bytes, size_t* residual_bytes, size_t* meta_bytes) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  codec_sizes(B, L, H_kv, D, page, C, anchor_bytes, residual_bytes, meta_bytes);
  return LYNX_OK;
}

int lynx_compander_thresholds(float alpha, float thresholds[127]) {
  if (!thresholds) return fail(LYNX_EINVAL, "null pointer");
  int rc = check_alpha(alpha);
  if (rc) return rc;
  const AlphaCache& t = tables_for(alpha);
  memcpy(thresholds, t.comp.thr, 127 * sizeof(float));
  return LYNX_OK;
}

int lynx_expand_table(float alpha, float table[128]) {
  if (!table) return fail(LYNX_EINVAL, "null pointer");
  int rc = check_alpha(alpha);
  if (rc) return rc;
  memcpy(table, tables_for(alpha).expand.x, 128 * sizeof(float));
  return LYNX_OK;
}

static int check_paging(const int32_t* block_table, int64_t num_blocks, Paging* pg) {
  if (num_blocks < 1 || num_blocks > INT32_MAX)
    return fail(LYNX_ESHAPE, "num_blocks = %lld: must be in [1, 2^31)", (long long)num_blocks);
  int rc = check_ptrs({block_table});
  if (rc) return rc;
  pg->table = block_table;
  pg->nphys = num_blocks;
  return LYNX_OK;
}

int lynx_encode_paged(const void* kv, int64_t B, int64_t L, int H_kv, int D, int page, int C,
                      float alpha, const int32_t* block_table, int64_t num_blocks,
                      void* anchor_pool, void* residual_pool, float* meta_pool, void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_encode_alpha(alpha))) return rc;
  if (B * L == 0) return LYNX_OK;
  Paging pg;
  if ((rc = check_paging(block_table, num_blocks, &pg))) return rc;
  if ((rc = check_ptrs({kv, anchor_pool, residual_pool, meta_pool}))) return rc;
  Shape s{B, L, H_kv, D, page, C};
  cudaError_t e = launch_encode(kv, s, tables_for(alpha).comp, anchor_pool, residual_pool,
                                meta_pool, static_cast<cudaStream_t>(stream), pg);
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_encode_paged");
}

int lynx_decode_paged(const void* anchor_pool, const void* residual_pool, const float* meta_pool,
                      const int32_t* block_table, int64_t num_blocks, int64_t B, int64_t L,
                      int H_kv, int D, int page, int C, float alpha, int mode, void* out,
                      int out_dtype, void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (mode != LYNX_ANCHOR && mode != LYNX_FULL)
    return fail(LYNX_EINVAL, "mode must be LYNX_ANCHOR or LYNX_FULL");
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return fail(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  if (B * L == 0) return LYNX_OK;
  Paging pg;
  if ((rc = check_paging(block_table, num_blocks, &pg))) return rc;
  if ((rc = check_ptrs({anchor_pool, meta_pool, out}))) return rc;
  if (mode == LYNX_FULL && (rc = check_ptrs({residual_pool}))) return rc;
  Shape s{B, L, H_kv, D, page, C};
  cudaError_t e = launch_decode(anchor_pool, mode == LYNX_FULL ? residual_pool : nullptr,
                                meta_pool, s, tables_for(alpha).expand, out,
                                out_dtype == LYNX_OUT_BF16, static_cast<cudaStream_t>(stream), pg);
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_decode_paged");
}

int lynx_encode(const void* kv, int64_t B, int64_t L, int H_kv, int D, int page, int C,
                float alpha, void* anchor, void* residual, float* meta, void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_encode_alpha(alpha))) return rc;
  if (B * L == 0) return LYNX_OK;  // nothing to encode; pointers are not examined
  if ((rc = check_ptrs({kv, anchor, residual, meta}))) return rc;
  Shape s{B, L, H_kv, D, page, C};
  cudaError_t e = launch_encode(kv, s, tables_for(alpha).comp, anchor, residual, meta,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_encode");
}

static int decode_common(const void* anchor, const void* residual, const float* meta, int64_t B,
                         int64_t L, int H_kv, int D, int page, int C, float alpha, void* out,
                         int out_dtype, void* stream, const char* what) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return fail(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  if (B * L == 0) return LYNX_OK;  // nothing to decode; pointers are not examined
  if ((rc = check_ptrs({anchor, meta, out}))) return rc;
  if (residual && (rc = check_ptrs({residual}))) return rc;
  Shape s{B, L, H_kv, D, page, C};
  cudaError_t e = launch_decode(anchor, residual, meta, s, tables_for(alpha).expand, out,
                                out_dtype == LYNX_OUT_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, what);
}

int lynx_decode_anchor(const void* anchor, const float* meta, int64_t B, int64_t L, int H_kv,
                       int D, int page, int C, float alpha, void* out, int out_dtype,
                       void* stream) {
  return decode_common(anchor, nullptr, meta, B, L, H_kv, D, page, C, alpha, out, out_dtype,
                       stream, "lynx_decode_anchor");
}

int lynx_decode_full(const void* anchor, const void* residual, const float* meta, int64_t B,
                     int64_t L, int H_kv, int D, int page, int C, float alpha, void* out,
                     int out_dtype, void* stream) {
  if (!residual && B * L != 0) return fail(LYNX_EINVAL, "null pointer");
  return decode_common(anchor, residual, meta, B, L, H_kv, D, page, C, alpha, out, out_dtype,
                       stream, "lynx_decode_full");
}

int lynx_decode_anchor_bits(const void* anchor_k, const float* meta, int64_t B, int64_t L,
                            int H_kv, int D, int page, int C, float alpha, int k, void* out,
                            int out_dtype, void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (k < 3 || k > 6) return fail(LYNX_EUNSUPPORTED, "k = %d: built for 3..6", k);
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return fail(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  if (B * L == 0) return LYNX_OK;
  if ((rc = check_ptrs({anchor_k, meta, out}))) return rc;
  Shape s{B, L, H_kv, D, page, C};
  cudaError_t e = launch_decode_anchor_bits(anchor_k, meta, s, k, tables_for(alpha).expand, out,
                                            out_dtype == LYNX_OUT_BF16,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_decode_anchor_bits");
}

int lynx_a1_encode(const void* kv, int64_t B, int64_t L, int H_kv, int D, int page, float alpha,
                   void* anchor, void* residual, float* meta, void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, 16, 512);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (B * L == 0) return LYNX_OK;
  if ((rc = check_ptrs({kv, anchor, residual, meta}))) return rc;
  Shape s{B, L, H_kv, D, page, 16};
  cudaError_t e = launch_a1_encode(kv, s, tables_for(alpha).comp, anchor, residual, meta,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_a1_encode");
}

int lynx_a1_decode(const void* anchor, const void* residual, const float* meta, int64_t B,
                   int64_t L, int H_kv, int D, int page, float alpha, void* out, int out_dtype,
                   void* stream) {
  int rc = check_codec_shape(B, L, H_kv, D, page, 16, 512);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return fail(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  if (B * L == 0) return LYNX_OK;
  if ((rc = check_ptrs({anchor, meta, out}))) return rc;
  if (residual && (rc = check_ptrs({residual}))) return rc;
  Shape s{B, L, H_kv, D, page, 16};
  cudaError_t e = launch_a1_decode(anchor, residual, meta, s, tables_for(alpha).expand, out,
                                   out_dtype == LYNX_OUT_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_a1_decode");
}

static int check_attn_shape(int batch, int T, int H_q, int64_t L, int H_kv, int D, int page,
                            int C) {
  int rc = check_codec_shape(batch, L, H_kv, D, page, C, 512);
  if (rc) return rc;
  if (batch < 1 || L < 1) return fail(LYNX_ESHAPE, "attention needs batch >= 1 and L >= 1");
  if (T < 1) return fail(LYNX_ESHAPE, "T = %d must be >= 1", T);
  if (H_q < 1 || H_q % H_kv) return fail(LYNX_ESHAPE, "H_q = %d is not a multiple of H_kv = %d", H_q, H_kv);
  if (T > 64) return fail(LYNX_EUNSUPPORTED, "T = %d: at most 64 query tokens", T);
  if ((H_q / H_kv) * T > 256)
    return fail(LYNX_EUNSUPPORTED, "(H_q/H_kv)*T = %d: at most 256 query rows per KV head", (H_q / H_kv) * T);
  return LYNX_OK;
}

int lynx_attn_workspace_bytes(int batch, int T, int H_q, int64_t L, int H_kv, int D, int page,
                              size_t* bytes) {
  if (!bytes) return fail(LYNX_EINVAL, "null pointer");
  int rc = check_attn_shape(batch, T, H_q, L, H_kv, D, page, page < 16 ? page : 16);
  if (rc) return rc;
  *bytes = attn_workspace_bytes(batch, T, H_q, H_kv, L);
  return LYNX_OK;
}

static int attn_common(const void* q, int batch, int T, int H_q, const void* k_anchor,
                       const void* k_residual, const float* k_meta, const void* v_anchor,
                       const void* v_residual, const float* v_meta, int64_t L, int H_kv, int D,
                       int page, int C, float alpha, int mode, const void* k_tail,
                       const void* v_tail, float* out, void* workspace, size_t workspace_bytes,
                       void* stream, const char* what, const Paging& pg = Paging()) {
  int rc = check_attn_shape(batch, T, H_q, L, H_kv, D, page, C);
  if (rc) return rc;
  if ((rc = check_alpha(alpha))) return rc;
  if (mode != LYNX_ANCHOR && mode != LYNX_FULL)
    return fail(LYNX_EINVAL, "mode must be LYNX_ANCHOR or LYNX_FULL");
  if ((rc = check_ptrs({q, k_anchor, k_meta, v_anchor, v_meta, out, workspace}))) return rc;
  if (mode == LYNX_FULL && (rc = check_ptrs({k_residual, v_residual}))) return rc;
  const size_t need = attn_workspace_bytes(batch, T, H_q, H_kv, L);
  if (workspace_bytes < need)
    return fail(LYNX_EWORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  AttnArgs a;
  a.q = q;
  a.batch = batch;
  a.T = T;
  a.H_q = H_q;
  a.k_anchor = k_anchor;
  a.k_residual = mode == LYNX_FULL ? k_residual : nullptr;
  a.k_meta = k_meta;
  a.v_anchor = v_anchor;
  a.v_residual = mode == LYNX_FULL ? v_residual : nullptr;
  a.v_meta = v_meta;
  a.s = Shape{batch, L, H_kv, D, page, C};
  a.full = mode == LYNX_FULL;
  a.out = out;
  a.workspace = workspace;
  a.k_tail = k_tail;
  a.v_tail = v_tail;
  a.paging = pg;
  cudaError_t e = launch_attn(a, tables_for(alpha).expand, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, what);
}

int lynx_attn_decode(const void* q, int batch, int T, int H_q, const void* k_anchor,
                     const void* k_residual, const float* k_meta, const void* v_anchor,
                     const void* v_residual, const float* v_meta, int64_t L, int H_kv, int D,
                     int page, int C, float alpha, int mode, float* out, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return attn_common(q, batch, T, H_q, k_anchor, k_residual, k_meta, v_anchor, v_residual,
                     v_meta, L, H_kv, D, page, C, alpha, mode, nullptr, nullptr, out, workspace,
                     workspace_bytes, stream, "lynx_attn_decode");
}

int lynx_attn_decode_tail(const void* q, int batch, int T, int H_q, const void* k_anchor,
                          const void* k_residual, const float* k_meta, const void* v_anchor,
                          const void* v_residual, const float* v_meta, int64_t L, int H_kv,
                          int D, int page, int C, float alpha, int mode, const void* k_tail,
                          const void* v_tail, float* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (batch > 0 && T > 0) {
    int rc = check_ptrs({k_tail, v_tail});
    if (rc) return rc;
  }
  return attn_common(q, batch, T, H_q, k_anchor, k_residual, k_meta, v_anchor, v_residual,
                     v_meta, L, H_kv, D, page, C, alpha, mode, k_tail, v_tail, out, workspace,
                     workspace_bytes, stream, "lynx_attn_decode_tail");
}

int lynx_attn_decode_paged(const void* q, int batch, int T, int H_q, const void* k_anchor_pool,
                           const void* k_residual_pool, const float* k_meta_pool,
                           const void* v_anchor_pool, const void* v_residual_pool,
                           const float* v_meta_pool, const int32_t* block_table,
                           int64_t num_blocks, int64_t L, int H_kv, int D, int page, int C,
                           float alpha, int mode, const void* k_tail, const void* v_tail,
                           float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if ((k_tail == nullptr) != (v_tail == nullptr))
    return fail(LYNX_EINVAL, "give both k_tail and v_tail, or neither");
  Paging pg;
  int rc = check_paging(block_table, num_blocks, &pg);
  if (rc) return rc;
  return attn_common(q, batch, T, H_q, k_anchor_pool, k_residual_pool, k_meta_pool,
                     v_anchor_pool, v_residual_pool, v_meta_pool, L, H_kv, D, page, C, alpha,
                     mode, k_tail, v_tail, out, workspace, workspace_bytes, stream,
                     "lynx_attn_decode_paged", pg);
}

int lynx_device_errors(unsigned int* bits) {
  if (!bits) return fail(LYNX_EINVAL, "null pointer");
  unsigned int enc = 0, dec = 0, att = 0, spc = 0, var = 0;
  cudaError_t e = read_wait_timeout(&enc);
  if (e == cudaSuccess) e = read_decode_wait_timeout(&dec);
  if (e == cudaSuccess) e = read_variant_wait_timeout(&var);
  if (e == cudaSuccess) e = read_attn_flags(&att);
  if (e == cudaSuccess) e = read_spec_flags(&spc);
  if (e != cudaSuccess) return cuda_fail(e, "lynx_device_errors");
  *bits = enc | dec | var | att | spc;
  return LYNX_OK;
}

int lynx_spec_verify(const float* p_target, const float* q_draft, const int32_t* draft_tokens,
                     const float* u_accept, const uint32_t* r_sample, int batch, int T,
                     int64_t V, int32_t* n_accepted, int32_t* next_token, void* stream) {
  if (batch < 0) return fail(LYNX_ESHAPE, "batch = %d < 0", batch);
  if (T < 1 || T > 64) return fail(LYNX_EUNSUPPORTED, "T = %d: 1..64 draft tokens", T);
  if (V < 1 || V > INT32_MAX) return fail(LYNX_ESHAPE, "V = %lld: must be in [1, 2^31)", (long long)V);
  if (batch == 0) return LYNX_OK;
  int rc = check_ptrs({p_target, q_draft, draft_tokens, u_accept, r_sample, n_accepted, next_token});
  if (rc) return rc;
  cudaError_t e = launch_spec_verify(p_target, q_draft, draft_tokens, u_accept, r_sample, batch, T,
                                     V, n_accepted, next_token, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_spec_verify");
}

int lynx_compander_selfcheck(float alpha, uint64_t* counts, void* stream) {
  int rc = check_alpha(alpha);
  if (rc) return rc;
  if ((rc = check_ptrs({counts}))) return rc;
  cudaError_t e = launch_compander_selfcheck(tables_for(alpha).comp, counts,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LYNX_OK : cuda_fail(e, "lynx_compander_selfcheck");
}

int lynx_wait_timeouts(unsigned int* flag) {
  if (!flag) return fail(LYNX_EINVAL, "null pointer");
  unsigned int enc = 0, dec = 0, var = 0;
  cudaError_t e = read_wait_timeout(&enc);
  if (e == cudaSuccess) e = read_decode_wait_timeout(&dec);
  if (e == cudaSuccess) e = read_variant_wait_timeout(&var);
  if (e != cudaSuccess) return cuda_fail(e, "lynx_wait_timeouts");
  *flag = ((enc | dec | var) & kFlagWaitTimeout) ? 1u : 0u;
  return LYNX_OK;
}

}  // extern "C"
