/*
 * lynx.h -- C ABI of the GB300 (sm_103a) split-stream KV codec and of decode
 * attention over its packed codes.
 *
 * Sources, cited by page title and section:
 *   [Review] "Lynx: Progressive Speculative KV Cache Transfer for
 *            Disaggregated LLM Inference" (technical review of the paper).
 *   [Digest] "Lynx: Progressive Speculative Quantization for accelerating KV
 *            Transfer in Long-Context Inference" (paper digest), "Method".
 *
 * Conventions shared by every call
 *   - Tensors are dense, row-major, in DEVICE memory owned by the caller.  The
 *     library allocates nothing on the device, keeps no state between calls
 *     except a per-thread copy of the last error text and a per-thread cache
 *     of the alpha tables, and is safe to call from several host threads.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is only enqueued: nothing synchronises, so results are
 *     ready when the stream reaches them.
 *   - Every argument is checked on the host before anything is enqueued; a
 *     failed check launches nothing and returns a negative lynx_status.  A
 *     codec call on an empty tensor (B * L == 0) enqueues nothing and returns
 *     LYNX_OK without examining the pointers.
 *     lynx_last_error() then holds a one-line reason.  A launch failure
 *     returns LYNX_ECUDA with the CUDA error text.  Device-side faults are not
 *     turned into status codes (they surface on the stream, as in CUDA).
 *   - Shapes: a KV tensor is kv[B][L][H_kv][D] BF16 with B = 2 * layers (or
 *     any batch of independent tensors), L tokens, H_kv heads, D = 128
 *     channels per head.  It is cut into page blocks of `page` tokens x D
 *     channels of one head, ordered (b, page index, head).
 *   - Encoded streams, per page block, contiguous, in block order:
 *       anchor   [B][L/page][H_kv][page][D/2] bytes   (4-bit Anchor codes)
 *       residual [B][L/page][H_kv][page][D/2] bytes   (4-bit Residual codes)
 *       meta     [B][L/page][H_kv][2 + 2*page/C][D] float32:
 *                gamma_min[D], gamma_scale[D], mu[page/C][D], sigma[page/C][D]
 *     Within a token row of D/2 bytes, byte 4G+k holds channel 8G+k in its low
 *     nibble and channel 8G+k+4 in its high nibble.  Anchor<<4 | Residual is
 *     the 8-bit two's-complement code Q8 = I*S + min(S, 0) of Eq. 9, I the
 *     7-bit magnitude code and S the sign.
 *   - Limits: D == 128; page in {64, 128, 256, 512} for the codec (encode,
 *     both decoders, the k-bit Anchor decode; the page sizes of the pages'
 *     ablation grid, [Review], "Concrete Improvement Suggestions", item 4)
 *     and for attention and the Appendix A.1 variant; C in
 *     {16, 32, 64, 128}, C <= page; L % page == 0; B * L < 2^31; alpha
 *     finite and > 0; every pointer 16-byte aligned.
 */
#ifndef LYNX_H
#define LYNX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LYNX_OK = 0,
    LYNX_EINVAL = -1,       /* null or misaligned pointer, bad alpha or enum */
    LYNX_ESHAPE = -2,       /* inconsistent sizes (L % page, C, T, heads ...) */
    LYNX_EUNSUPPORTED = -3, /* valid but not built: D != 128, page/C outside the list */
    LYNX_ECUDA = -4,        /* a CUDA call or launch failed */
    LYNX_EWORKSPACE = -5    /* workspace smaller than lynx_attn_workspace_bytes */
} lynx_status;

typedef enum { LYNX_ANCHOR = 0, LYNX_FULL = 1 } lynx_mode;
typedef enum { LYNX_OUT_BF16 = 0, LYNX_OUT_FP32 = 1 } lynx_dtype;

/* Host-only.  Byte sizes of the three encoded streams for a kv[B][L][H_kv][D]
 * tensor (see the layout above; meta holds 2 + 2*page/C float32 rows of D per
 * page block, [Review, "Why Not Global Grouped Quantization?"]).  Any output
 * pointer may be NULL.  Returns LYNX_OK or a shape/limit error. */
int lynx_encoded_sizes(int64_t B, int64_t L, int H_kv, int D, int page, int C,
                       size_t *anchor_bytes, size_t *residual_bytes,
                       size_t *meta_bytes);

/* Encode: Algorithm 1 [Review, Mechanism 1] on every page block.
 *   Stage 1: per channel, gamma_min = min over the page, gamma_scale =
 *            max - min, n = (x - gamma_min) * rn(1/(gamma_scale + 1e-6)).
 *   Stage 2: per chunk of C tokens and channel, mu = mean(n) (pairwise-halving
 *            sum), sigma = max|n - mu|, x_final = (n - mu) * rn(1/(sigma+1e-6)).
 *   Stage 3: I = Round(127 ln(1 + alpha|x_final|) / ln(1 + alpha)) (Eq. 7),
 *            S = sign(n - mu) (+1 at zero).
 *   Stage 4: Q8 = I*S + min(S,0) (Eq. 9); Anchor = Q8 >> 4, Residual = Q8 & 15.
 * Statistics are float32 with one rounding per operation in the order above;
 * Round is exact with respect to the float64 value of Eq. 7.  alpha must be
 * >= 1 (the pages use 100 to 2000); smaller values give LYNX_EUNSUPPORTED.
 *   kv        [B][L][H_kv][D] BF16, device, read only
 *   anchor    device, lynx_encoded_sizes() bytes, written
 *   residual  device, written
 *   meta      device float32, written                                      */
int lynx_encode(const void *kv, int64_t B, int64_t L, int H_kv, int D,
                int page, int C, float alpha, void *anchor, void *residual,
                float *meta, void *stream);

/* Anchor-only decode [Review, Mechanism 2, decode side Anchor Phase:
 * "Q_approx = dequant(Q_anc, gamma, mu, sigma)"]: the signed Anchor gives S
 * and V = I >> 4; the value is S * X(16V + 7), X(y) = ((1+alpha)^(y/127) - 1)
 * / alpha (the geometric-interval exponent of [Digest, Method]; Eq. 14), then
 *   n = fma(S*X, sigma + 1e-6, mu);  x = fma(n, gamma_scale + 1e-6, gamma_min)
 * with X(.) rounded once to float32 from float64.
 *   out  [B][L][H_kv][D], BF16 (round to nearest even) or FP32, device.     */
int lynx_decode_anchor(const void *anchor, const float *meta, int64_t B,
                       int64_t L, int H_kv, int D, int page, int C,
                       float alpha, void *out, int out_dtype, void *stream);

/* Full decode [Review, Mechanism 2, Residual Phase: "Q_full =
 * dequant(Q_anc + Q_res)"; Eq. 15]: Q8 = Anchor<<4 | Residual gives S and I
 * exactly; value S * X(I), then the same two fused multiply-adds.          */
int lynx_decode_full(const void *anchor, const void *residual,
                     const float *meta, int64_t B, int64_t L, int H_kv, int D,
                     int page, int C, float alpha, void *out, int out_dtype,
                     void *stream);

/* ---- Paged streams.  The pages' prototype keeps KV in pages aligned with
 * paged attention and scatters the decoded pages into device memory
 * [Review, Implementation Notes; Mechanism 2, Anchor Phase step 3].  Paged
 * variants keep the three streams in pools of num_blocks physical pages, each
 * holding the H_kv head blocks of one page exactly as the dense layout does
 * for one (b, page): anchor / residual pool [num_blocks][H_kv][page][D/2],
 * meta pool [num_blocks][H_kv][2 + 2*page/C][D] float32 (the sizes
 * lynx_encoded_sizes gives for B = 1, L = num_blocks * page).  A block table
 * block_table[B][L/page] (int32, device, 16-byte aligned) names the physical
 * page of each (sequence, logical page); K and V pools share one table.
 * Entries must lie in [0, num_blocks); an entry outside is replaced by 0 and
 * reported by lynx_device_errors (bit 2), so it gives wrong numbers, never a
 * stray memory access.  Distinct (sequence, page) pairs should name distinct
 * pages when encoding (pages written twice race). */

/* lynx_encode writing each page block to its physical page in the pools. */
int lynx_encode_paged(const void *kv, int64_t B, int64_t L, int H_kv, int D,
                      int page, int C, float alpha, const int32_t *block_table,
                      int64_t num_blocks, void *anchor_pool, void *residual_pool,
                      float *meta_pool, void *stream);

/* lynx_decode_anchor (mode LYNX_ANCHOR, residual_pool may be NULL) or
 * lynx_decode_full (LYNX_FULL) reading each page through the block table;
 * out is the dense [B][L][H_kv][D] tensor. */
int lynx_decode_paged(const void *anchor_pool, const void *residual_pool,
                      const float *meta_pool, const int32_t *block_table,
                      int64_t num_blocks, int64_t B, int64_t L, int H_kv, int D,
                      int page, int C, float alpha, int mode, void *out,
                      int out_dtype, void *stream);

/* ---------------------------------------------------------------------
 * Split-stream transfer [Review, Mechanism 2 (Figure 4, Implementation
 * Notes): the Anchor stream on a high-priority queue, the Residual stream on
 * a low-priority one, decoding as soon as the Anchor lands; Anchor buffers
 * are drained before Residual buffers at the page level; the serializer
 * quantises page i+1 while page i is in flight].
 *
 * The unit of transfer is a group of `pages_per_group` consecutive pages of
 * the flattened (b, page) order (H_kv page blocks each; the last group may be
 * shorter).  Because the three streams are stored in (b, page, head) order,
 * a group is one contiguous byte range of each stream (and of the BF16
 * tensor), so it moves with one copy per stream.
 *
 * A schedule is a list of operations on three queues:
 *   LYNX_Q_COPY     the one copy queue: every Anchor and meta copy of every
 *                   group comes before the first Residual copy (the drain
 *                   rule, taken strictly);
 *   LYNX_Q_HI       high-priority kernels: encode (sender) or anchor decode
 *                   (receiver);
 *   LYNX_Q_LO       low-priority kernels: the in-place upgrade to the full
 *                   decode (receiver).
 * An operation may wait for up to two earlier operations on other queues,
 * named by (kind, group); group -1 there means "every group of that kind". */
enum {
  LYNX_OP_ENCODE = 0,        /* sender: encode the group on the device       */
  LYNX_OP_COPY_ANCHOR = 1,   /* Anchor bytes of the group                    */
  LYNX_OP_COPY_META = 2,     /* metadata bytes of the group                  */
  LYNX_OP_COPY_RESIDUAL = 3, /* Residual bytes of the group                  */
  LYNX_OP_DECODE_ANCHOR = 4, /* receiver: Anchor-only decode into out        */
  LYNX_OP_UPGRADE = 5,       /* receiver: full decode over the same out      */
  LYNX_OP_NONE = -1
};
enum { LYNX_Q_COPY = 0, LYNX_Q_HI = 1, LYNX_Q_LO = 2 };

typedef struct {
  int32_t kind, queue;
  int64_t group;
  int64_t page0, n_pages;     /* flattened page range [page0, page0 + n_pages) */
  int64_t offset, bytes;      /* byte range of the copied stream (copies only) */
  int32_t wait_kind[2];       /* LYNX_OP_NONE when unused                       */
  int64_t wait_group[2];      /* -1: every group of wait_kind                   */
} lynx_split_op;

/* The schedule lynx_split_receive (send = 0) or lynx_split_send (send = 1)
 * enqueues, in issue order.  with_decode (receiver only): 1 adds the anchor
 * decode and upgrade kernels.  Host-only; writes at most max_ops entries and
 * sets *n_ops to the full count.  LYNX_EWORKSPACE if max_ops is too small. */
int lynx_split_plan(int64_t B, int64_t L, int H_kv, int D, int page, int C,
                    int64_t pages_per_group, int send, int with_decode,
                    lynx_split_op *ops, int64_t max_ops, int64_t *n_ops);

/* Receiver.  Copies the encoded streams from host memory (h_*, page-locked
 * for the copies to overlap) to the device (anchor, meta, residual), group
 * by group in the drain order above, on copy_stream.  If out is not NULL,
 * each group is decoded from its Anchor on hi_stream as soon as its Anchor
 * and meta have landed (lynx_decode_anchor of that page range), and, once
 * every Anchor group is decoded, upgraded in place on lo_stream as soon as
 * its Residual has landed (lynx_decode_full of that page range over the
 * same out).  Events (may be NULL): anchor_ready is recorded on hi_stream
 * when every Anchor and meta byte is on the device (and decoded, with out);
 * full_ready on lo_stream when every Residual byte is (and out holds the
 * full decode).  Streams may be NULL (the legacy default stream).  Returns
 * after enqueueing; sizes as lynx_encoded_sizes. */
int lynx_split_receive(const void *h_anchor, const float *h_meta,
                       const void *h_residual, void *anchor, float *meta,
                       void *residual, int64_t B, int64_t L, int H_kv, int D,
                       int page, int C, float alpha, int64_t pages_per_group,
                       void *out, int out_dtype, void *copy_stream,
                       void *hi_stream, void *lo_stream, void *anchor_ready,
                       void *full_ready);

/* Sender.  Encodes kv group by group on hi_stream into the device streams
 * (anchor, meta, residual) and copies each group's Anchor and meta to host
 * memory (h_*) on copy_stream as soon as it is encoded, so encoding group
 * g+1 overlaps the copy of group g; every Residual copy follows the last
 * Anchor copy.  Events (may be NULL): anchor_sent on copy_stream after the
 * last Anchor and meta byte, all_sent after the last Residual byte. */
int lynx_split_send(const void *kv, int64_t B, int64_t L, int H_kv, int D,
                    int page, int C, float alpha, void *anchor, float *meta,
                    void *residual, void *h_anchor, float *h_meta,
                    void *h_residual, int64_t pages_per_group,
                    void *hi_stream, void *copy_stream, void *anchor_sent,
                    void *all_sent);

/* Format header of a serialized request: header, then the Anchor stream,
 * the meta stream and the Residual stream, so the Anchor phase (codes and
 * the metadata needed to decode them) is one contiguous byte range.  All
 * integers little-endian as laid out here; 128 bytes. */
typedef struct {
  char magic[8];          /* "LYNXKV" 0 1                                  */
  uint32_t version;       /* 1                                             */
  uint32_t header_bytes;  /* 128                                           */
  int64_t B, L;
  int32_t H_kv, D, page, C;
  float alpha;
  uint32_t flags;         /* bit 0: Residual stream present                */
  uint64_t anchor_offset, anchor_bytes;
  uint64_t meta_offset, meta_bytes;
  uint64_t residual_offset, residual_bytes;
  uint64_t total_bytes;   /* header + the three streams                    */
  uint32_t reserved[3];   /* zero                                          */
  uint32_t header_crc;    /* CRC-32 (IEEE 802.3) of the 124 bytes before it */
} lynx_header;

/* Fill *h for these dimensions (validated as for lynx_encode). */
int lynx_header_init(lynx_header *h, int64_t B, int64_t L, int H_kv, int D,
                     int page, int C, float alpha, int with_residual);
/* LYNX_OK if *h is a well-formed version-1 header whose sizes and offsets
 * follow from its dimensions; LYNX_EINVAL (bad magic, version, CRC or
 * sizes) or the codes of lynx_encode for bad dimensions otherwise. */
int lynx_header_check(const lynx_header *h);

/* ---------------------------------------------------------------------
 * Comparison points.
 *
 * Linear INT-B baseline [Review, Prerequisites, Eq. 4: Q(x) = round(x/S +
 * Z), S = (x_max - x_min)/(2^B - 1)], the INT8 / INT4 of the pages' tables:
 * one (S, Z) per row of D = 128 channels (a token of one KV head), Z =
 * -x_min/S, Q = round((x - x_min) * rcp(S)) to nearest even, clamped to
 * [0, 2^B - 1] (rcp(0) = 0: a constant row codes to 0); a zero extreme
 * counts as +0.  Decode: x = fma(Q, S, x_min).
 *   kv     [rows][128] BF16 (a [B][L][H_kv][128] tensor has rows = B*L*H_kv)
 *   codes  [rows][128 * bits / 8] uint8; bits = 4: byte j holds channels 2j
 *          (low nibble) and 2j+1 (high nibble)
 *   meta   [rows][2] float32: (x_min, S)
 *   out    [rows][128] BF16 or float32 (out_dtype)
 * bits must be 4 or 8; device pointers, 16-byte aligned; one pass each,
 * enqueued on `stream`. */
int lynx_int_encode(const void *kv, int64_t rows, int D, int bits, void *codes,
                    float *meta, void *stream);
int lynx_int_decode(const void *codes, const float *meta, int64_t rows, int D,
                    int bits, void *out, int out_dtype, void *stream);

/* Other Anchor/Residual bit splits [Review, Concrete Improvement
 * Suggestions, items 4-5: 3+5, 4+4, 5+3, 6+2].  The code is the same signed
 * 8-bit Q8; a k-bit Anchor is its arithmetic top k bits and the Residual its
 * low 8-k bits.  Layout of a k-split: per token row and aligned group of 8
 * channels 8G..8G+7, k Anchor bytes and 8-k Residual bytes, channel 8G+j in
 * bits j*w .. j*w + w - 1 (w the field width) of the group's bytes read as
 * one little-endian integer; page blocks in the (b, page, head) order of the
 * 4+4 streams.  rows = B * L * H_kv token rows.
 * lynx_split_bits re-splits 4+4 streams; lynx_join_bits is its inverse.
 * Device pointers, 16-byte aligned (LYNX_EINVAL otherwise); D must be 128
 * and 3 <= k <= 6 (LYNX_EUNSUPPORTED), rows >= 0 (LYNX_ESHAPE); one pass,
 * enqueued on `stream`. */
int lynx_split_bits(const void *anchor, const void *residual, int64_t rows,
                    int D, int k, void *anchor_k, void *residual_k,
                    void *stream);
int lynx_join_bits(const void *anchor_k, const void *residual_k, int64_t rows,
                   int D, int k, void *anchor, void *residual, void *stream);
/* Anchor-only decode of a k-bit Anchor stream, 3 <= k <= 6: bucket point
 * I = 2^(8-k) V + 2^(7-k) - 1 (16 V + 7 for k = 4), then the
 * reconstruction of lynx_decode_anchor; out, shape checks and errors as
 * lynx_decode_anchor, and LYNX_EUNSUPPORTED for k outside 3..6. */
int lynx_decode_anchor_bits(const void *anchor_k, const float *meta, int64_t B,
                            int64_t L, int H_kv, int D, int page, int C,
                            float alpha, int k, void *out, int out_dtype,
                            void *stream);

/* The variant of [Review] Appendix A.1: x' = x / m (m = max |x| of the
 * channel over the page), x'' = x' / m_i (m_i = max |x'| over 16 consecutive
 * tokens), y = sgn(x'') ln(1 + alpha |x''|) / ln(1 + alpha), Q = sgn(x'')
 * Round(127 |y|) in [-127, 127] (exact, as Stage 3), Q_anc = Q >> 4
 * (arithmetic), Q_res = Q & 0xF.  Divisions are multiplications by correctly
 * rounded reciprocals, of 0 for a zero maximum.  Streams as lynx_encode
 * (same nibble pairing); meta [B][L/page][H_kv][1 + page/16][D] float32 =
 * m, then m_i per chunk.  Decode: x = (sgn X(|Q|) * m_i) * m (Eq. 14/15
 * inverse, two float32 products); with residual = NULL the Anchor-only
 * point Q = 16 Q_anc + 7.  A NaN element codes as 0 and is left out of
 * the maxima; an infinite page maximum makes the channel's scales 0.  The
 * pages use alpha = 100 for this variant.  Shape checks and errors as
 * lynx_encode / lynx_decode_full (C fixed at 16); alpha > 0 and finite. */
int lynx_a1_encode(const void *kv, int64_t B, int64_t L, int H_kv, int D,
                   int page, float alpha, void *anchor, void *residual,
                   float *meta, void *stream);
int lynx_a1_decode(const void *anchor, const void *residual, const float *meta,
                   int64_t B, int64_t L, int H_kv, int D, int page, float alpha,
                   void *out, int out_dtype, void *stream);

/* Speculative verification and correction [Review, Mechanism 3, Eq. 10 and
 * Eq. 11], for every sequence b of the batch, on distributions the caller's
 * verification pass (p, over the full KV) and draft steps (q, over the
 * Anchor-only KV) produced:
 *   p_target      [batch][T+1][V] float32, p(. | s_<t, Q_full), t = 1..T+1
 *   q_draft       [batch][T][V] float32, p(. | s_<t, Q_approx), t = 1..T
 *   draft_tokens  [batch][T] int32, s_1..s_T
 *   u_accept      [batch][T] float32 uniforms in [0, 1)
 *   r_sample      [batch] uint32 uniforms
 *   n_accepted    [batch] int32, written: k, the accepted prefix length
 *   next_token    [batch] int32, written: the token that follows s_k
 * s_t is accepted iff u_t * q_t(s_t) < p_t(s_t) (float32; i.e. with
 * probability min(1, p/q)) and every earlier one was.  The next token is
 * drawn from max(0, p_{k+1} - q_{k+1}) after a rejection, or from p_{T+1}
 * after a fully accepted draft, by inverse CDF over the integer weights
 * floor(w * 2^40) with target floor(r * Z / 2^32), Z their sum; if Z = 0 the
 * weights of p are used, and if they sum to 0 too the token is -1.  The
 * rows need not be normalised, but each row's weights must sum below 2^24
 * so that Z fits in 64 bits (distributions sum to 1); NaN and negative
 * weights count as 0.  A draft token outside [0, V) counts as rejected and
 * is reported by lynx_device_errors (bit 4).  1 <= T <= 64, 1 <= V < 2^31;
 * all device pointers, 16-byte aligned.  One cluster of 8 CTAs per sequence,
 * enqueued on `stream`. */
int lynx_spec_verify(const float *p_target, const float *q_draft,
                     const int32_t *draft_tokens, const float *u_accept,
                     const uint32_t *r_sample, int batch, int T, int64_t V,
                     int32_t *n_accepted, int32_t *next_token, void *stream);

/* Host call, synchronous: *bits = OR of the conditions any kernel of this
 * library in this process has reported: 1 = a bounded wait on an
 * asynchronous copy gave up (the kernel returned early, its outputs are
 * incomplete), 2 = a block-table entry was outside [0, num_blocks), 4 = a
 * draft token of lynx_spec_verify was outside [0, V), 8 = (checked build
 * only, liblynx_checked.so, the same sources compiled with -DLYNX_CHECKED) an
 * index that a kernel computed for a global access fell outside the extent the
 * call's shapes give; the index was replaced by 0, so the outputs are wrong
 * but nothing outside the buffers was touched. */
int lynx_device_errors(unsigned int *bits);

/* Host-only.  Device workspace (bytes) that lynx_attn_decode needs for these
 * sizes: split-K partial results, float32.  0 is never returned for valid
 * sizes.  Returns LYNX_OK or a shape/limit error. */
int lynx_attn_workspace_bytes(int batch, int T, int H_q, int64_t L, int H_kv,
                              int D, int page, size_t *bytes);

/* Decode attention over packed KV [Review, Prerequisites Eq. 1]:
 *   O = softmax(q K^T / sqrt(D)) V
 * for every sequence, query row and query head, grouped-query: query head hq
 * reads KV head hq / (H_q / H_kv).  K and V are reconstructed on the fly
 * (never written to global memory) as lynx_decode_anchor (mode LYNX_ANCHOR, the draft step of [Review,
 * Mechanism 2, Anchor Phase]) or lynx_decode_full (LYNX_FULL, the T-token
 * verification pass of [Review, Mechanism 3]) would with BF16 output, the
 * affine map applied as one fused multiply-add x = fma(v, A, B) with
 * A = (sigma + eps)(gamma_scale + eps), B = fma(mu, gamma_scale + eps,
 * gamma_min) per chunk and channel (the decoders use two; the BF16 operands
 * then differ from the decoders' on about 2e-4 of the values, by one BF16 ulp
 * or by 2^-22 of the channel's gamma_scale, far inside the attention
 * tolerance); every one of the T query rows attends to all L cached tokens.
 *   q          [batch][T][H_q][D] BF16, device
 *   k_*, v_*   the encode outputs of the K and V tensors [batch][L][H_kv][D]
 *              (B = batch); k_residual / v_residual may be NULL in ANCHOR mode
 *   out        [batch][T][H_q][D] float32, device, written
 *   workspace  device scratch of >= lynx_attn_workspace_bytes(...) bytes; its
 *              contents on entry do not matter and are clobbered
 * Limits: 1 <= T <= 64 (the pages' speculative cap), H_q % H_kv == 0,
 * (H_q / H_kv) * T <= 256, C >= 16, L >= 1.  Up to 8 query rows per KV head
 * take the single-warp shape (register-direct MMAs); more rows form groups of
 * up to 32, each of which reads the packed K and V once: in LYNX_FULL mode
 * with L a multiple of 128 on the tcgen05 path (tiles of 128 tokens rebuilt
 * in shared memory, scores and output accumulated in tensor memory), else
 * in the warp-pair shape. */
int lynx_attn_decode(const void *q, int batch, int T, int H_q,
                     const void *k_anchor, const void *k_residual,
                     const float *k_meta, const void *v_anchor,
                     const void *v_residual, const float *v_meta, int64_t L,
                     int H_kv, int D, int page, int C, float alpha, int mode,
                     float *out, void *workspace, size_t workspace_bytes,
                     void *stream);

/* lynx_attn_decode with the draft tokens' own keys and values: the single
 * parallel verification pass of [Review, Mechanism 3] runs one forward pass
 * over the whole draft s_1..s_T, so query token t (t = 0..T-1) attends to the
 * L cached tokens and, causally, to draft tokens 0..t, whose keys and values
 * that pass has just computed in BF16 (not quantised):
 *   O_t = softmax(q_t [K; Kt_0..t]^T / sqrt(D)) [V; Vt_0..t]
 *   k_tail, v_tail  [batch][T][H_kv][D] BF16, device, read only; token t of
 *                   sequence b for KV head h at ((b*T + t)*H_kv + h)*D
 * Everything else, the workspace size included, is as lynx_attn_decode; the
 * draft tokens are merged in the split combine.  Null tails: LYNX_EINVAL. */
int lynx_attn_decode_tail(const void *q, int batch, int T, int H_q,
                          const void *k_anchor, const void *k_residual,
                          const float *k_meta, const void *v_anchor,
                          const void *v_residual, const float *v_meta,
                          int64_t L, int H_kv, int D, int page, int C,
                          float alpha, int mode, const void *k_tail,
                          const void *v_tail, float *out, void *workspace,
                          size_t workspace_bytes, void *stream);

/* lynx_attn_decode_tail over paged streams: the K and V pools are read
 * through block_table (see the paged layout above).  k_tail and v_tail may
 * both be NULL (no draft tokens: the pass of lynx_attn_decode). */
int lynx_attn_decode_paged(const void *q, int batch, int T, int H_q,
                           const void *k_anchor_pool, const void *k_residual_pool,
                           const float *k_meta_pool, const void *v_anchor_pool,
                           const void *v_residual_pool, const float *v_meta_pool,
                           const int32_t *block_table, int64_t num_blocks,
                           int64_t L, int H_kv, int D, int page, int C,
                           float alpha, int mode, const void *k_tail,
                           const void *v_tail, float *out, void *workspace,
                           size_t workspace_bytes, void *stream);

/* lynx_attn_decode without a caller-provided workspace, for callers that
 * cannot allocate device memory: code that runs while a stream is being
 * captured into a CUDA graph, real-time or signal paths that must not enter an
 * allocator, and hosts whose memory manager forbids driver allocations after
 * start-up.  The split-K scratch is a fixed 8 MiB array in the library's
 * device image (static, one per GPU that loads the library, held until the
 * process exits); sizes that need more than that (lynx_attn_workspace_bytes
 * > 8 MiB) fail with LYNX_EWORKSPACE.  The paper has no counterpart: this is
 * an interface of this library only.
 * The first call on a device looks the array's address up (with that device
 * current; this also loads the library's device image, which places the
 * array) and caches it per device; a call that finds a different current
 * context than the cached address belongs to (after cudaDeviceReset) looks it
 * up again.  Make the first call on each device, and the first after a reset,
 * before any stream capture.  Nothing else is allocated or freed.  All calls share the one array
 * and it keeps the last call's contents (no state needs clearing: every
 * partial is written before it is read), so calls whose work overlaps on the
 * GPU race with each other: issue them on one stream, or order them.
 * Arguments, results and the other errors are those of lynx_attn_decode. */
int lynx_attn_decode_noalloc(const void *q, int batch, int T, int H_q,
                             const void *k_anchor, const void *k_residual,
                             const float *k_meta, const void *v_anchor,
                             const void *v_residual, const float *v_meta,
                             int64_t L, int H_kv, int D, int page, int C,
                             float alpha, int mode, float *out, void *stream);

/* Host-only.  The 127 rounding thresholds of Stage 3 for this alpha:
 * thresholds[k] is the smallest float32 a >= 0 whose Eq. 7 value (float64)
 * rounds to more than k, so Round(Y(a)) = #{k : a >= thresholds[k]}.
 * The encode kernel decides every code this way.  Returns LYNX_OK/EINVAL. */
int lynx_compander_thresholds(float alpha, float thresholds[127]);

/* Host-only.  The 128 reconstruction magnitudes X(I) = ((1+alpha)^(I/127)-1)
 * / alpha (Eq. 14/15), float64 rounded to float32, used by both decoders. */
int lynx_expand_table(float alpha, float table[128]);

/* Checks the encoder's fast Stage-3 rounding against the thresholds for every
 * float32 a in [0, 1] on the device, for this alpha.  counts (device, 4 x
 * uint64, zeroed by the call): [0] values checked, [1] values whose fast
 * result was not exact and was not flagged for the exact path (must be 0),
 * [2] values flagged for the exact path, [3] max |fast Y - exact Y| in units
 * of 2^-32 (an error bound of the approximation).  Enqueued on `stream`. */
int lynx_compander_selfcheck(float alpha, uint64_t *counts, void *stream);

/* Host call, synchronous: *flag = 1 if any kernel of this library in this
 * process gave up a bounded wait on an asynchronous copy (it then returned
 * early and its outputs are incomplete), else 0. */
int lynx_wait_timeouts(unsigned int *flag);

/* Check of the bounded wait every asynchronous-copy wait in the library
 * uses: one CTA initialises an mbarrier, arrives on it (arrive == 1) or not
 * (arrive == 0), and waits with a limit of limit_ns nanoseconds
 * (0 < limit_ns <= 1e9) on the global timer.  *status (device) = 1 if the
 * barrier completed, 2 if the wait gave up.  arrive == 2 runs the
 * verification pass's own wait (lynx_attn_decode on the tensor-memory path)
 * twice on barriers nothing arrives on: the first, limited to limit_ns, must
 * give up and raise the CTA's abort word; the second, started half a limit
 * later with the kernel's full limit (2 s), must then return at once;
 * *status = 3 if both held, 4 if not.  The library's error words are not
 * touched.  Nothing faults or hangs either way.  Enqueued on `stream`. */
int lynx_wait_selftest(uint64_t limit_ns, int arrive, unsigned int *status,
                       void *stream);

/* Text of a status code, and of the last failure on this host thread. */
const char *lynx_status_string(int code);
const char *lynx_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LYNX_H */
