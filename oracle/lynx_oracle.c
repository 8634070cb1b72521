/*
 * lynx_oracle.c -- plain, slow CPU oracle of the Lynx split-stream KV codec
 * and of decode attention over the reconstructed KV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no source, header, table or constant
 * generator with the CUDA library.
 *
 * Sources (web pages about one paper; cited by title and section):
 *   [Review] "Lynx: Progressive Speculative KV Cache Transfer for
 *            Disaggregated LLM Inference" (technical review of the paper),
 *            sections "Mechanism 1: Hierarchical Non-Linear Quantization
 *            (Algorithm 1)" Stages 1-4 with Eq. 7-9, "Mechanism 2" (decode
 *            side, Anchor and Residual phases), "Worked Example" Eq. 12-15,
 *            "Implementation Notes", "Appendix A.1", and "Prerequisites" Eq. 1.
 *   [Digest] "Lynx: Progressive Speculative Quantization for accelerating KV
 *            Transfer in Long-Context Inference" (paper digest), "Method".
 *
 * Arithmetic conventions (compiled with -ffp-contract=off -fno-fast-math):
 *   - Stage 1 and 2 statistics are IEEE binary32, one rounding per operation,
 *     in the order written below.  The pages store the metadata as float32
 *     ([Review], "Why Not Global Grouped Quantization?": "9 KB metadata per
 *     page in float32"), and a code is an integer decided from these values,
 *     so both this oracle and the GPU take that decision from the same
 *     float32 statistics.
 *   - The alpha-law value Y (Eq. 7) is evaluated in float64 from the float32
 *     magnitude, then rounded to the nearest integer.
 *   - Reconstruction tables and attention are float64.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   eps = 1e-6 in both divisions; a division by (s + eps) is a multiplication
 *   by the correctly rounded float32 reciprocal; the chunk mean sums its C
 *   values by a pairwise-halving tree (v[i] += v[i+h], h = C/2 ... 1), C a
 *   power of two; the sign S is the sign of the centred value (d >= 0 -> +1);
 *   Stage 4 applies Eq. 9 to the full 7-bit magnitude, giving one signed
 *   8-bit code whose arithmetic high nibble is the Anchor (Eq. 9 applied to
 *   V = I >> 4) and whose low nibble is the Residual (the extraction of
 *   [Review] Appendix A.1); Anchor-only reconstruction uses the bucket point
 *   16*V + 7 (the "+7 = 2^3 - 1" round-half-down bias of Stage 4).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EPS 1e-6f

/* ---------------------------------------------------------------- helpers */

static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float32 -> bfloat16 bit pattern, IEEE round to nearest, ties to even: the
 * decoders' BF16 output and every attention operand are the float32
 * reconstruction rounded this way.  Adding 0x7fff plus the lowest kept bit
 * and dropping the low 16 bits rounds ties to the even neighbour; a carry out
 * of the kept mantissa steps the exponent (past the largest finite bf16 it
 * lands on infinity, as round to nearest does).  A NaN stays a NaN: it keeps
 * its sign and top payload bits and is made quiet (the addition could carry
 * its payload into the exponent and return an infinity or a zero). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}

float oracle_bf16_to_f32(uint16_t h) { return bf16_bits_to_f32(h); }

/* ------------------------------------------------------ Stage 3 (Eq. 7) */

/* Y = ln(1 + alpha |x|) / ln(1 + alpha) * (2^7 - 1)   [Review, Stage 3, Eq. 7]
 * evaluated in float64 from the float32 magnitude a = |X_final|. */
double oracle_compand_y(float a, float alpha)
{
    double al = (double)alpha;
    return 127.0 * log1p(al * (double)a) / log1p(al);
}

/* I = Round(Y) in {0..127}                      [Review, Stage 3, after Eq. 7]
 * Round to nearest; Y >= 0 so floor(Y + 1/2) is nearest with ties upward. */
int oracle_round_code(float a, float alpha)
{
    double y = oracle_compand_y(a, alpha);
    double r = floor(y + 0.5);
    if (r < 0.0) r = 0.0;
    if (r > 127.0) r = 127.0;
    return (int)r;
}

/* Inverse compander |x^| = ((1 + alpha)^(I/127) - 1) / alpha, float64, then
 * rounded once to float32.            [Review, Worked Example, Eq. 14 and 15] */
float oracle_expand(int I, float alpha)
{
    double al = (double)alpha;
    return (float)((pow(1.0 + al, (double)I / 127.0) - 1.0) / al);
}

/* ------------------------------------------------------ Stage 4 (Eq. 9) */

/* Stage 4 exactly as the review prints it, for one element:
 *   I_bias = I + 7; V_mag = I_bias >> 4; V_recon = V_mag << 4;
 *   V_res = V_recon - I; Q_anc = V_mag * S + min(S, 0).
 * out[0..4] = I_bias, V_mag, V_recon, V_res, Q_anc.   [Review, Stage 4, Eq. 9]
 * Used only to check the worked example and to count the V_mag = 8 cases
 * that do not fit a 4-bit Anchor; the codec below uses the 8-bit reading. */
void oracle_stage4_literal(int I, int S, int *out)
{
    int I_bias = I + 7;
    int V_mag = I_bias >> 4;
    int V_recon = V_mag << 4;
    int V_res = V_recon - I;
    int Q_anc = V_mag * S + (S < 0 ? S : 0);
    out[0] = I_bias;
    out[1] = V_mag;
    out[2] = V_recon;
    out[3] = V_res;
    out[4] = Q_anc;
}

/* Eq. 9 applied to the full magnitude: Q8 = I*S + min(S, 0) in [-128, 127],
 * stored as its 8-bit two's-complement pattern.        [Review, Stage 4, Eq. 9] */
int oracle_code8(int I, int S)
{
    int q8 = I * S + (S < 0 ? S : 0);
    return q8 & 0xff;
}

/* Split of the signed 8-bit code: Anchor = Q8 >> 4 (arithmetic, a signed
 * 4-bit value = Eq. 9 applied to V = I >> 4), Residual = Q8 & 0xF.
 *                              [Review, Stage 4; Review, Appendix A.1] */
int oracle_anchor_nibble(int code8) { return (code8 >> 4) & 0xf; }
int oracle_residual_nibble(int code8) { return code8 & 0xf; }

/* --------------------------------------------------------------- encode */

/* Byte index within a token row and nibble shift for channel d (see the
 * packing note of oracle_encode_block). */
static size_t nib_byte(int d) { return (size_t)(d >> 3) * 4u + (size_t)(d & 3); }
static int nib_shift(int d) { return (d & 4) ? 4 : 0; }

/*
 * Algorithm 1 on one page block: P tokens x D channels of one KV head.
 *   x          BF16 bits, element (t, d) at x[t * row_stride + d]
 *   anchor     P x D/2 bytes, token-major.  Two 4-bit values per uint8
 *              ([Review, Implementation Notes]); the pages do not say which
 *              two, so within each aligned group of 8 channels 8G..8G+7,
 *              byte 4G + k holds channel 8G+k in its low nibble and channel
 *              8G+k+4 in its high nibble (k = 0..3).
 *   residual   same layout
 *   meta       (2 + 2 P/C) x D floats: gamma_min[D], gamma_scale[D],
 *              mu[P/C][D], sigma[P/C][D]
 * Returns 0, or -1 on a bad argument.
 */
int oracle_encode_block(const uint16_t *x, int64_t row_stride, int P, int D,
                        int C, float alpha, uint8_t *anchor, uint8_t *residual,
                        float *meta)
{
    if (P <= 0 || D <= 0 || (D & 7) || C <= 0 || (C & (C - 1)) || P % C)
        return -1;
    const int NC = P / C;
    float *g_min = meta;
    float *g_scale = meta + D;
    float *mu_rows = meta + 2 * D;
    float *sg_rows = meta + (size_t)(2 + NC) * D;
    float *n = (float *)malloc(sizeof(float) * (size_t)P);
    float *v = (float *)malloc(sizeof(float) * (size_t)C);
    if (!n || !v) {
        free(n);
        free(v);
        return -1;
    }
    memset(anchor, 0, (size_t)P * (size_t)(D / 2));
    memset(residual, 0, (size_t)P * (size_t)(D / 2));

    for (int d = 0; d < D; ++d) {
        /* Stage 1: gamma_min = min over the page, gamma_scale = max - min,
         * X <- (X - gamma_min) / (gamma_scale + eps)      [Review, Stage 1] */
        float lo = FLT_MAX, hi = -FLT_MAX;
        for (int t = 0; t < P; ++t) {
            float xv = bf16_bits_to_f32(x[(int64_t)t * row_stride + d]);
            if (xv < lo) lo = xv;
            if (xv > hi) hi = xv;
        }
        /* min and max do not order +0 and -0, so a zero extreme is given one
         * sign: the minimum becomes -0 (then x - gamma_min of any zero x is
         * +0, and no -0 reaches the sign test of Stage 3), the maximum +0. */
        if (lo == 0.0f) lo = -0.0f;
        if (hi == 0.0f) hi = 0.0f;
        float gs = hi - lo;
        float rg = 1.0f / (gs + ORACLE_EPS);
        for (int t = 0; t < P; ++t) {
            float xv = bf16_bits_to_f32(x[(int64_t)t * row_stride + d]);
            n[t] = (xv - lo) * rg;
        }
        g_min[d] = lo;
        g_scale[d] = gs;

        for (int c = 0; c < NC; ++c) {
            const float *nc = n + (size_t)c * C;
            /* Stage 2: mu = Mean over the C tokens of the chunk,
             * sigma = max |X - mu|, X_final = (X - mu) / (sigma + eps)
             *                                           [Review, Stage 2] */
            for (int i = 0; i < C; ++i) v[i] = nc[i];
            for (int h = C / 2; h >= 1; h /= 2)
                for (int i = 0; i < h; ++i) v[i] = v[i] + v[i + h];
            float mu = v[0] * (1.0f / (float)C);
            float sg = 0.0f;
            for (int i = 0; i < C; ++i) {
                float dd = nc[i] - mu;
                float ad = fabsf(dd);
                if (ad > sg) sg = ad;
            }
            float rs = 1.0f / (sg + ORACLE_EPS);
            mu_rows[(size_t)c * D + d] = mu;
            sg_rows[(size_t)c * D + d] = sg;

            for (int i = 0; i < C; ++i) {
                float dd = nc[i] - mu;
                int S = dd >= 0.0f ? 1 : -1;
                float xf = dd * rs;
                /* Stage 3: I = Round(Y(|X_final|))  [Review, Stage 3, Eq. 7] */
                int I = oracle_round_code(fabsf(xf), alpha);
                /* Stage 4: signed 8-bit code, split into two nibbles. */
                int code8 = oracle_code8(I, S);
                int t = c * C + i;
                size_t byte = (size_t)t * (size_t)(D / 2) + nib_byte(d);
                int sh = nib_shift(d);
                anchor[byte] |= (uint8_t)(oracle_anchor_nibble(code8) << sh);
                residual[byte] |= (uint8_t)(oracle_residual_nibble(code8) << sh);
            }
        }
    }
    free(n);
    free(v);
    return 0;
}

/*
 * Whole tensor kv[B][L][H][D] (BF16 bits), page blocks in the order
 * (b, page, h), for the blocks [blk_begin, blk_end) of that order.
 * Outputs are the full-size streams: anchor/residual [B][L/P][H][P][D/2],
 * meta [B][L/P][H][2 + 2P/C][D]; only the selected blocks are written.
 */
int oracle_encode_range(const uint16_t *kv, int64_t B, int64_t L, int H, int D,
                        int P, int C, float alpha, uint8_t *anchor,
                        uint8_t *residual, float *meta, int64_t blk_begin,
                        int64_t blk_end)
{
    if (B <= 0 || L <= 0 || H <= 0 || P <= 0 || L % P) return -1;
    const int64_t NB = L / P;
    const int NC = P / C;
    const size_t code_blk = (size_t)P * (size_t)(D / 2);
    const size_t meta_blk = (size_t)(2 + 2 * NC) * (size_t)D;
    for (int64_t blk = blk_begin; blk < blk_end; ++blk) {
        int64_t h = blk % H;
        int64_t p = (blk / H) % NB;
        int64_t b = blk / (H * NB);
        const uint16_t *x = kv + ((b * L + p * P) * H + h) * D;
        int rc = oracle_encode_block(x, (int64_t)H * D, P, D, C, alpha,
                                     anchor + blk * code_blk,
                                     residual + blk * code_blk,
                                     meta + blk * meta_blk);
        if (rc) return rc;
    }
    return 0;
}

/* --------------------------------------------------------------- decode */

/*
 * Decode one page block back to float32 values out[t * out_stride + d].
 * residual == NULL: Anchor-only reconstruction ("Q_approx = dequant(Q_anc,
 *   gamma, mu, sigma)" [Review, Mechanism 2, Anchor Phase]): the signed
 *   Anchor a gives S and V (a >= 0: S = +1, V = a; a < 0: S = -1,
 *   V = -a - 1) and the bucket point I = 16 V + 7.
 * residual != NULL: full reconstruction ("Q_full = dequant(Q_anc + Q_res)"
 *   [Review, Mechanism 2, Residual Phase]): Q8 = Anchor * 16 + Residual as a
 *   signed 8-bit value, S = sign, I = Q8 (S = +1) or -Q8 - 1 (S = -1).
 * Then |x_final| = ((1+alpha)^(I/127) - 1)/alpha (Eq. 14/15) with sign S, and
 * the two affine steps of Stages 2 and 1 are undone with fused multiply-adds:
 *   n = fma(x_final, sigma + eps, mu); x = fma(n, gamma_scale + eps, gamma_min).
 */
int oracle_decode_block(const uint8_t *anchor, const uint8_t *residual,
                        const float *meta, int P, int D, int C, float alpha,
                        float *out, int64_t out_stride)
{
    if (P <= 0 || D <= 0 || (D & 7) || C <= 0 || P % C) return -1;
    const int NC = P / C;
    const float *g_min = meta;
    const float *g_scale = meta + D;
    const float *mu_rows = meta + 2 * D;
    const float *sg_rows = meta + (size_t)(2 + NC) * D;
    float table[128];
    for (int I = 0; I < 128; ++I) table[I] = oracle_expand(I, alpha);

    for (int t = 0; t < P; ++t) {
        int c = t / C;
        for (int d = 0; d < D; ++d) {
            size_t byte = (size_t)t * (size_t)(D / 2) + nib_byte(d);
            int sh = nib_shift(d);
            int a = (anchor[byte] >> sh) & 0xf;
            int S, I;
            if (residual) {
                int r = (residual[byte] >> sh) & 0xf;
                int q8 = (a << 4) | r;
                if (q8 >= 128) q8 -= 256;
                S = q8 >= 0 ? 1 : -1;
                I = S > 0 ? q8 : -q8 - 1;
            } else {
                int qa = a >= 8 ? a - 16 : a;
                S = qa >= 0 ? 1 : -1;
                int V = S > 0 ? qa : -qa - 1;
                I = 16 * V + 7;
            }
            float xf = S > 0 ? table[I] : -table[I];
            float sg = sg_rows[(size_t)c * D + d];
            float mu = mu_rows[(size_t)c * D + d];
            float nv = fmaf(xf, sg + ORACLE_EPS, mu);
            float xv = fmaf(nv, g_scale[d] + ORACLE_EPS, g_min[d]);
            out[(int64_t)t * out_stride + d] = xv;
        }
    }
    return 0;
}

/* Whole-tensor decode into out[B][L][H][D] float32 for blocks
 * [blk_begin, blk_end) of the (b, page, h) order. */
int oracle_decode_range(const uint8_t *anchor, const uint8_t *residual,
                        const float *meta, int64_t B, int64_t L, int H, int D,
                        int P, int C, float alpha, float *out,
                        int64_t blk_begin, int64_t blk_end)
{
    if (B <= 0 || L <= 0 || H <= 0 || P <= 0 || L % P) return -1;
    const int64_t NB = L / P;
    const int NC = P / C;
    const size_t code_blk = (size_t)P * (size_t)(D / 2);
    const size_t meta_blk = (size_t)(2 + 2 * NC) * (size_t)D;
    for (int64_t blk = blk_begin; blk < blk_end; ++blk) {
        int64_t h = blk % H;
        int64_t p = (blk / H) % NB;
        int64_t b = blk / (H * NB);
        float *o = out + ((b * L + p * P) * H + h) * D;
        int rc = oracle_decode_block(anchor + blk * code_blk,
                                     residual ? residual + blk * code_blk : NULL,
                                     meta + blk * meta_blk, P, D, C, alpha, o,
                                     (int64_t)H * D);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------- bit-split variants */

/*
 * Other Anchor/Residual bit splits ([Review], "Concrete Improvement
 * Suggestions", items 4-5: the split 3+5, 4+4, 5+3 or 6+2 as one axis of an
 * ablation, and its Pareto frontier).  The code is
 * the same signed 8-bit Q8 of Stage 4; a k-bit Anchor is its arithmetic top
 * k bits and the Residual its low 8-k bits, so (Anchor << (8-k)) | Residual
 * == Q8, as for the 4+4 split (the extraction of [Review] Appendix A.1 with
 * a shift of 8-k).  The Anchor-only reconstruction point generalises the
 * 4+4 bucket point 16 V + 7: the round-half-down centre of the 2^(8-k)
 * codes of a bucket, I_rep = 2^(8-k) V + 2^(7-k) - 1, V = the Anchor's
 * magnitude (a >= 0 ? a : -a - 1).
 * Layout (a reading; the pages fix none): per token, the aligned group of 8
 * channels 8G..8G+7 fills k Anchor bytes and 8-k Residual bytes, channel
 * 8G+j in bits j*w .. j*w + w - 1 (w = the field width) of the group's
 * bytes read as one little-endian integer.  Blocks keep the (b, page, head)
 * order of the 4+4 streams.
 */
static int field_get(const uint8_t *p, int j, int w)
{
    int v = 0;
    for (int i = 0; i < w; ++i) {
        int b = j * w + i;
        v |= ((p[b >> 3] >> (b & 7)) & 1) << i;
    }
    return v;
}

static void field_put(uint8_t *p, int j, int w, int v)
{
    for (int i = 0; i < w; ++i) {
        int b = j * w + i;
        uint8_t m = (uint8_t)(1u << (b & 7));
        if ((v >> i) & 1) p[b >> 3] |= m; else p[b >> 3] &= (uint8_t)~m;
    }
}

/* Re-split `rows` token rows of D channels from the 4+4 streams (nibble
 * pairing of Stage 4) into a k / (8-k) split, 3 <= k <= 6. */
int oracle_split_bits(const uint8_t *anchor4, const uint8_t *residual4, int64_t rows, int D,
                      int k, uint8_t *ak, uint8_t *rk)
{
    if (k < 3 || k > 6 || D <= 0 || (D & 7)) return -1;
    const int rw = 8 - k;
    for (int64_t t = 0; t < rows; ++t) {
        for (int d = 0; d < D; ++d) {
            size_t byte = (size_t)t * (size_t)(D / 2) + nib_byte(d);
            int sh = nib_shift(d);
            int q8 = (((anchor4[byte] >> sh) & 0xf) << 4) | ((residual4[byte] >> sh) & 0xf);
            uint8_t *pa = ak + (size_t)t * (size_t)(D / 8) * (size_t)k + (size_t)(d / 8) * (size_t)k;
            uint8_t *pr = rk + (size_t)t * (size_t)(D / 8) * (size_t)rw + (size_t)(d / 8) * (size_t)rw;
            field_put(pa, d % 8, k, (q8 >> rw) & ((1 << k) - 1));
            field_put(pr, d % 8, rw, q8 & ((1 << rw) - 1));
        }
    }
    return 0;
}

/* Anchor-only decode of one page block from a k-bit Anchor stream. */
int oracle_decode_anchor_bits_block(const uint8_t *ak, const float *meta, int P, int D, int C,
                                    float alpha, int k, float *out, int64_t out_stride)
{
    if (k < 3 || k > 6 || P <= 0 || D <= 0 || (D & 7) || C <= 0 || P % C) return -1;
    const int NC = P / C;
    const float *g_min = meta;
    const float *g_scale = meta + D;
    const float *mu_rows = meta + 2 * D;
    const float *sg_rows = meta + (size_t)(2 + NC) * D;
    float table[128];
    for (int I = 0; I < 128; ++I) table[I] = oracle_expand(I, alpha);
    for (int t = 0; t < P; ++t) {
        int c = t / C;
        for (int d = 0; d < D; ++d) {
            const uint8_t *pa = ak + (size_t)t * (size_t)(D / 8) * (size_t)k + (size_t)(d / 8) * (size_t)k;
            int a = field_get(pa, d % 8, k);
            int qa = a >= (1 << (k - 1)) ? a - (1 << k) : a;
            int S = qa >= 0 ? 1 : -1;
            int V = S > 0 ? qa : -qa - 1;
            int I = (1 << (8 - k)) * V + (1 << (7 - k)) - 1;
            float xf = S > 0 ? table[I] : -table[I];
            float sg = sg_rows[(size_t)c * D + d];
            float mu = mu_rows[(size_t)c * D + d];
            float nv = fmaf(xf, sg + ORACLE_EPS, mu);
            out[(int64_t)t * out_stride + d] = fmaf(nv, g_scale[d] + ORACLE_EPS, g_min[d]);
        }
    }
    return 0;
}

/* The same over a whole [B][L][H][D] tensor (float32 out). */
int oracle_decode_anchor_bits_range(const uint8_t *ak, const float *meta, int64_t B, int64_t L,
                                    int H, int D, int P, int C, float alpha, int k, float *out)
{
    if (B <= 0 || L <= 0 || H <= 0 || P <= 0 || L % P || C <= 0 || P % C) return -1;
    const int64_t NB = L / P;
    const size_t code_blk = (size_t)P * (size_t)(D / 8) * (size_t)k;
    const size_t meta_blk = (size_t)(2 + 2 * (P / C)) * (size_t)D;
    for (int64_t blk = 0; blk < B * NB * H; ++blk) {
        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);
        int rc = oracle_decode_anchor_bits_block(ak + blk * code_blk, meta + blk * meta_blk, P, D,
                                                 C, alpha, k, out + ((b * L + p * P) * H + h) * D,
                                                 (int64_t)H * D);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------- Appendix A.1 variant */

/*
 * The variant of [Review] Appendix A.1 ("Hierarchical Quantization: Full
 * Derivation"), which differs from Algorithm 1: no centring, scaling by
 * magnitudes only.
 *   Step 1  x'  = x / m,    m   = max |x| of the channel over the page;
 *   Step 2  x'' = x' / m_i, m_i = max |x'| of the channel over a chunk of 16
 *           consecutive tokens;
 *   Step 3  y = sgn(x'') ln(1 + alpha |x''|) / ln(1 + alpha);
 *   Step 4  Q = clip(round(127 y), -127, 127); Q_anc = Q >> 4 (arithmetic),
 *           Q_res = Q & 0xF.
 * Readings: each division is a multiplication by the correctly rounded
 * float32 reciprocal, and a zero maximum gives 0 (its channel or chunk codes
 * to 0); |Q| = Round(Y(|x''|)) with Y of Eq. 7 in float64 (nearest, ties
 * up), so |Q| <= 127 and the clip never acts; Q keeps the sign of x'' (0 for
 * x'' = 0).  The nibbles are packed as the 4+4 streams of Stage 4 (byte 4G+j:
 * channels 8G+j low, 8G+j+4 high).  meta per block: m [D], then m_i
 * [P/16][D], float32.  Decode: |x''| = X(|Q|) (Eq. 14/15), x = sgn X m_i m
 * (two float32 products).  Anchor-only: Q is taken as 16 Q_anc + 7, the
 * round-half-down point of the bucket as in Stage 4.
 */
#define A1_CHUNK 16

int oracle_a1_encode_block(const uint16_t *x, int64_t row_stride, int P, int D, float alpha,
                           uint8_t *anchor, uint8_t *residual, float *meta)
{
    if (P <= 0 || P % A1_CHUNK || D <= 0 || (D & 7)) return -1;
    memset(anchor, 0, (size_t)P * (size_t)(D / 2));
    memset(residual, 0, (size_t)P * (size_t)(D / 2));
    for (int d = 0; d < D; ++d) {
        float m = 0.0f;
        for (int t = 0; t < P; ++t) {
            float a = fabsf(bf16_bits_to_f32(x[(int64_t)t * row_stride + d]));
            if (a > m) m = a;
        }
        float rm = m > 0.0f ? 1.0f / m : 0.0f;
        meta[d] = m;
        for (int c = 0; c < P / A1_CHUNK; ++c) {
            float xp[A1_CHUNK];
            float mi = 0.0f;
            for (int i = 0; i < A1_CHUNK; ++i) {
                int t = c * A1_CHUNK + i;
                xp[i] = bf16_bits_to_f32(x[(int64_t)t * row_stride + d]) * rm;
                float a = fabsf(xp[i]);
                if (a > mi) mi = a;
            }
            float rmi = mi > 0.0f ? 1.0f / mi : 0.0f;
            meta[(size_t)(1 + c) * D + d] = mi;
            for (int i = 0; i < A1_CHUNK; ++i) {
                int t = c * A1_CHUNK + i;
                float xpp = xp[i] * rmi;
                int I = oracle_round_code(fabsf(xpp), alpha);
                if (I > 127) I = 127;
                int Q = xpp > 0.0f ? I : (xpp < 0.0f ? -I : 0);
                int qa = Q >> 4;                    /* arithmetic shift */
                int qr = Q & 0xF;
                size_t byte = (size_t)t * (size_t)(D / 2) + nib_byte(d);
                anchor[byte] |= (uint8_t)((qa & 0xF) << nib_shift(d));
                residual[byte] |= (uint8_t)(qr << nib_shift(d));
            }
        }
    }
    return 0;
}

int oracle_a1_decode_block(const uint8_t *anchor, const uint8_t *residual, const float *meta,
                           int P, int D, float alpha, float *out, int64_t out_stride)
{
    if (P <= 0 || P % A1_CHUNK || D <= 0 || (D & 7)) return -1;
    float table[128];
    for (int I = 0; I < 128; ++I) table[I] = oracle_expand(I, alpha);
    for (int t = 0; t < P; ++t) {
        int c = t / A1_CHUNK;
        for (int d = 0; d < D; ++d) {
            size_t byte = (size_t)t * (size_t)(D / 2) + nib_byte(d);
            int a = (anchor[byte] >> nib_shift(d)) & 0xF;
            int qa = a >= 8 ? a - 16 : a;
            int Q = residual ? qa * 16 + ((residual[byte] >> nib_shift(d)) & 0xF) : qa * 16 + 7;
            int I = Q < 0 ? -Q : Q;
            if (I > 127) I = 127;
            float v = Q < 0 ? -table[I] : table[I];
            out[(int64_t)t * out_stride + d] = (v * meta[(size_t)(1 + c) * D + d]) * meta[d];
        }
    }
    return 0;
}

/* Whole [B][L][H][D] tensors, blocks in (b, page, h) order. */
int oracle_a1_encode_range(const uint16_t *kv, int64_t B, int64_t L, int H, int D, int P,
                           float alpha, uint8_t *anchor, uint8_t *residual, float *meta)
{
    if (B <= 0 || L <= 0 || H <= 0 || P <= 0 || L % P) return -1;
    const int64_t NB = L / P;
    const size_t code_blk = (size_t)P * (size_t)(D / 2);
    const size_t meta_blk = (size_t)(1 + P / A1_CHUNK) * (size_t)D;
    for (int64_t blk = 0; blk < B * NB * H; ++blk) {
        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);
        int rc = oracle_a1_encode_block(kv + ((b * L + p * P) * H + h) * D, (int64_t)H * D, P, D,
                                        alpha, anchor + blk * code_blk, residual + blk * code_blk,
                                        meta + blk * meta_blk);
        if (rc) return rc;
    }
    return 0;
}

int oracle_a1_decode_range(const uint8_t *anchor, const uint8_t *residual, const float *meta,
                           int64_t B, int64_t L, int H, int D, int P, float alpha, float *out)
{
    if (B <= 0 || L <= 0 || H <= 0 || P <= 0 || L % P) return -1;
    const int64_t NB = L / P;
    const size_t code_blk = (size_t)P * (size_t)(D / 2);
    const size_t meta_blk = (size_t)(1 + P / A1_CHUNK) * (size_t)D;
    for (int64_t blk = 0; blk < B * NB * H; ++blk) {
        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);
        int rc = oracle_a1_decode_block(anchor + blk * code_blk,
                                        residual ? residual + blk * code_blk : NULL,
                                        meta + blk * meta_blk, P, D, alpha,
                                        out + ((b * L + p * P) * H + h) * D, (int64_t)H * D);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------ linear INT-B baseline */

/*
 * The linear quantizer the pages compare against ([Review], Prerequisites,
 * "KV Cache Quantization and the Outlier Problem", Eq. 4):
 *   Q(x) = round(x / S + Z),  S = (x_max - x_min) / (2^B - 1).
 * Readings (the pages fix none of them): one (S, Z) per token and KV head,
 * over its D channels (the grouping in which an outlier channel sets the
 * scale of the others, Eq. 5); Z = -x_min / S, so Q = round((x - x_min)/S),
 * the division taken as a multiplication by the correctly rounded float32
 * reciprocal of S (of 0 for a constant row, S = 0: every code is then 0);
 * round to nearest, ties to even; Q clamped to [0, 2^B - 1]; a zero x_min
 * or x_max counts as +0 (so S of an all-zero row is +0).  Reconstruction
 * x = Q * S + x_min in one fused multiply-add.  B = 8: one byte a value;
 * B = 4: byte j holds channels 2j (low nibble) and 2j+1 (high nibble).
 * meta: (x_min, S) float32 per row.
 */
int oracle_int_encode_rows(const uint16_t *x, int64_t rows, int D, int bits, uint8_t *codes,
                           float *meta)
{
    if ((bits != 4 && bits != 8) || D <= 0 || (D & 1)) return -1;
    const int qmax = (1 << bits) - 1;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * D;
        float lo = bf16_bits_to_f32(xr[0]), hi = lo;
        for (int d = 1; d < D; ++d) {
            float v = bf16_bits_to_f32(xr[d]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        lo = lo + 0.0f;
        hi = hi + 0.0f;
        float S = (hi - lo) / (float)qmax;
        float rs = S > 0.0f ? 1.0f / S : 0.0f;
        uint8_t *cr = codes + r * (int64_t)(bits == 8 ? D : D / 2);
        if (bits == 4) memset(cr, 0, (size_t)(D / 2));
        for (int d = 0; d < D; ++d) {
            float dd = bf16_bits_to_f32(xr[d]) - lo;
            float qf = rintf(dd * rs);
            if (qf > (float)qmax) qf = (float)qmax;
            if (qf < 0.0f) qf = 0.0f;
            int q = (int)qf;
            if (bits == 8) cr[d] = (uint8_t)q;
            else cr[d / 2] |= (uint8_t)(q << ((d & 1) ? 4 : 0));
        }
        meta[2 * r] = lo;
        meta[2 * r + 1] = S;
    }
    return 0;
}

int oracle_int_decode_rows(const uint8_t *codes, const float *meta, int64_t rows, int D, int bits,
                           float *out)
{
    if ((bits != 4 && bits != 8) || D <= 0 || (D & 1)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t *cr = codes + r * (int64_t)(bits == 8 ? D : D / 2);
        float lo = meta[2 * r], S = meta[2 * r + 1];
        for (int d = 0; d < D; ++d) {
            int q = bits == 8 ? cr[d] : (cr[d / 2] >> ((d & 1) ? 4 : 0)) & 0xf;
            out[r * D + d] = fmaf((float)q, S, lo);
        }
    }
    return 0;
}

/* ------------------------------------------------------------ attention */

/*
 * One query row of O = softmax(q K^T / sqrt(d_k)) V   [Review, Eq. 1]
 * in float64 over L cached tokens: K[t * kv_stride + d], V likewise.
 * out[D] receives the float64 result.
 */
void oracle_attention_row(const float *q, const float *K, const float *V,
                          int64_t L, int D, int64_t kv_stride, double *out)
{
    double scale = 1.0 / sqrt((double)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    double m = -HUGE_VAL;
    for (int64_t t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += (double)q[d] * (double)K[t * kv_stride + d];
        s[t] = acc * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double w = exp(s[t] - m);
        l += w;
        for (int d = 0; d < D; ++d) out[d] += w * (double)V[t * kv_stride + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    free(s);
}

/* One query row of the verification pass with the draft tokens' own keys
 * and values [Review, Mechanism 3, "Single parallel verification pass": one
 * forward pass over the whole draft sequence]: the row of draft position t
 * attends to the L cached tokens (K, V, rows kv_stride apart) and to the
 * fresh tokens 0..t of the draft (Kt, Vt, rows tail_stride apart), i.e.
 * n_tail = t + 1 of them; one float64 softmax over all L + n_tail scores,
 * each scaled by 1/sqrt(D) [Eq. 1]. */
void oracle_attention_row_tail(const float *q, const float *K, const float *V,
                               int64_t L, const float *Kt, const float *Vt,
                               int n_tail, int D, int64_t kv_stride,
                               int64_t tail_stride, double *out)
{
    double scale = 1.0 / sqrt((double)D);
    int64_t n = L + n_tail;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -HUGE_VAL;
    for (int64_t t = 0; t < n; ++t) {
        const float *k = t < L ? K + t * kv_stride : Kt + (t - L) * tail_stride;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += (double)q[d] * (double)k[d];
        s[t] = acc * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        const float *v = t < L ? V + t * kv_stride : Vt + (t - L) * tail_stride;
        double w = exp(s[t] - m);
        l += w;
        for (int d = 0; d < D; ++d) out[d] += w * (double)v[d];
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    free(s);
}

/* ---------------------------------------------------------------- Eq. 10-11
 * Speculative verification and correction [Review, Mechanism 3, Eq. 10 and
 * Eq. 11], the draft-then-verify rule the pages adapt from Chen et al. 2023,
 * for one sequence:
 *   p  [T+1][V]  target distributions p(. | s_<t, Q_full), t = 1..T+1
 *   q  [T][V]    draft distributions p(. | s_<t, Q_approx), t = 1..T
 *   s  [T]       draft tokens, u [T] uniforms in [0, 1), r a uniform uint32.
 * Draft token s_t is accepted with probability min(1, p_t(s_t) / q_t(s_t))
 * (Eq. 10): with u_t uniform that is u_t * q_t(s_t) < p_t(s_t), one float32
 * product and compare.  k = the length of the accepted prefix.  At the first
 * rejected position k+1 the next token is drawn from
 * p'(x) ∝ max(0, p_{k+1}(x) - q_{k+1}(x)) (Eq. 11); when every draft token is
 * accepted it is drawn from p_{T+1} (the verification pass's next-token
 * distribution).  The draw is an inverse CDF over integer weights
 * W(x) = floor(w(x) * 2^40) (w the float32 weight), target floor(r * Z / 2^32)
 * with Z = sum W: the smallest x whose running sum of W exceeds the target.
 * If Z = 0 the weights of p at that position are used instead; if those sum
 * to 0 too, the token is -1.  Returns k; *token receives the drawn token. */
static uint64_t spec_weight(float w)
{
    return w > 0.0f ? (uint64_t)(w * 1099511627776.0f) : 0u;
}

/* float32 weight of token x: max(0, p - q) (Eq. 11) with a draft
 * distribution, p itself without one */
static float spec_w(const float *pk, const float *qk, int64_t x)
{
    return qk ? fmaxf(pk[x] - qk[x], 0.0f) : pk[x];
}

int oracle_spec_verify(const float *p, const float *q, const int32_t *s,
                       const float *u, uint32_t r, int T, int64_t V,
                       int32_t *token)
{
    int k = 0;
    while (k < T) {
        int64_t x = s[k];
        float pv = p[(int64_t)k * V + x], qv = q[(int64_t)k * V + x];
        if (!(u[k] * qv < pv)) break;
        ++k;
    }
    const float *pk = p + (int64_t)k * V;
    const float *qk = k < T ? q + (int64_t)k * V : NULL;
    for (int pass = 0; pass < 2; ++pass) {
        const float *qw = pass == 0 ? qk : NULL;
        uint64_t Z = 0;
        for (int64_t x = 0; x < V; ++x)
            Z += spec_weight(spec_w(pk, qw, x));
        if (Z == 0) continue;
        uint64_t target = (uint64_t)(((unsigned __int128)r * Z) >> 32);
        uint64_t run = 0;
        for (int64_t x = 0; x < V; ++x) {
            run += spec_weight(spec_w(pk, qw, x));
            if (run > target) {
                *token = (int32_t)x;
                return k;
            }
        }
    }
    *token = -1;
    return k;
}

/* oracle_spec_verify for each of `batch` sequences (arrays batch-major). */
void oracle_spec_verify_batch(const float *p, const float *q, const int32_t *s,
                              const float *u, const uint32_t *r, int batch, int T,
                              int64_t V, int32_t *k, int32_t *token)
{
    for (int b = 0; b < batch; ++b)
        k[b] = oracle_spec_verify(p + (int64_t)b * (T + 1) * V, q + (int64_t)b * T * V,
                                  s + (int64_t)b * T, u + (int64_t)b * T, r[b], T, V,
                                  token + b);
}
