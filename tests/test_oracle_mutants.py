"""The pins catch plausible mistakes in the oracle.

Each mutant is a copy of oracle/lynx_oracle.c with one planted mistake (a
dropped term, a wrong sign, index or constant, a transposed operand),
compiled on the CPU and swapped in for the real oracle; at least one pin of
tests/test_oracle_pins.py must then fail.  Nothing here touches a GPU.
"""
import inspect
import os
import tempfile

import pytest

import oracle

from . import test_oracle_pins as pins

MUTANTS = [
    ("INT-B minimum stored at row r, not 2r", '        meta[2 * r] = lo;',
     '        meta[r] = lo;'),
    ("INT-8 rows written at the 4-bit stride", '\n        uint8_t *cr = codes + r * (int64_t)(bits == 8 ? D : D / 2);',
     '\n        uint8_t *cr = codes + r * (int64_t)(D / 2);'),
    ("spec batch: p at stride T*V", 'k[b] = oracle_spec_verify(p + (int64_t)b * (T + 1) * V,',
     'k[b] = oracle_spec_verify(p + (int64_t)b * T * V,'),
    ("spec batch: every sequence seeded by r[0]", 's + (int64_t)b * T, u + (int64_t)b * T, r[b], T, V,',
     's + (int64_t)b * T, u + (int64_t)b * T, r[0], T, V,'),
    ('k-bit decode range: page and head swapped',
     '        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);\n        int rc = oracle_decode_anchor_bits_block(ak + blk * code_blk, meta + blk * meta_blk, P, D,',
     '        int64_t p = blk % NB, h = (blk / NB) % H, b = blk / (H * NB);\n        int rc = oracle_decode_anchor_bits_block(ak + blk * code_blk, meta + blk * meta_blk, P, D,'),
    ('A.1 encode range: page and head swapped',
     '        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);\n        int rc = oracle_a1_encode_block(kv + ((b * L + p * P) * H + h) * D, (int64_t)H * D, P, D,',
     '        int64_t p = blk % NB, h = (blk / NB) % H, b = blk / (H * NB);\n        int rc = oracle_a1_encode_block(kv + ((b * L + p * P) * H + h) * D, (int64_t)H * D, P, D,'),
    ('A.1 decode range: page and head swapped',
     '        int64_t h = blk % H, p = (blk / H) % NB, b = blk / (H * NB);\n        int rc = oracle_a1_decode_block(anchor + blk * code_blk,',
     '        int64_t p = blk % NB, h = (blk / NB) % H, b = blk / (H * NB);\n        int rc = oracle_a1_decode_block(anchor + blk * code_blk,'),
    ("range encode: page and head swapped",
     '        int64_t h = blk % H;\n        int64_t p = (blk / H) % NB;\n        int64_t b = blk / (H * NB);\n        const uint16_t *x',
     '        int64_t p = blk % NB;\n        int64_t h = (blk / NB) % H;\n        int64_t b = blk / (H * NB);\n        const uint16_t *x'),
    ("range encode: rows read at stride D", 'oracle_encode_block(x, (int64_t)H * D, P, D, C, alpha,',
     'oracle_encode_block(x, (int64_t)D, P, D, C, alpha,'),
    ("range decode: rows written at stride D", 'alpha, o,\n                                     (int64_t)H * D);',
     'alpha, o,\n                                     (int64_t)D);'),
    ("compander numerator 128 instead of 127",
     "return 127.0 * log1p(al * (double)a) / log1p(al);",
     "return 128.0 * log1p(al * (double)a) / log1p(al);"),
    ("round down instead of to nearest", "double r = floor(y + 0.5);", "double r = floor(y);"),
    ("inverse exponent over 128", "(double)I / 127.0) - 1.0) / al);",
     "(double)I / 128.0) - 1.0) / al);"),
    ("Eq. 9 without the min(S,0) term", "int q8 = I * S + (S < 0 ? S : 0);", "int q8 = I * S;"),
    ("anchor taken from the low nibble", "{ return (code8 >> 4) & 0xf; }",
     "{ return code8 & 0xf; }"),
    ("nibble pairing swapped", "{ return (d & 4) ? 4 : 0; }", "{ return (d & 4) ? 0 : 4; }"),
    ("page max as a min", "if (xv > hi) hi = xv;", "if (xv < hi) hi = xv;"),
    ("scale without eps", "float rg = 1.0f / (gs + ORACLE_EPS);", "float rg = 1.0f / (gs);"),
    ("normalise without subtracting gamma_min", "n[t] = (xv - lo) * rg;", "n[t] = xv * rg;"),
    ("tree sum off by one", "v[i] = v[i] + v[i + h];", "v[i] = v[i] + v[i + h - 1];"),
    ("mean over C+1", "float mu = v[0] * (1.0f / (float)C);",
     "float mu = v[0] * (1.0f / (float)(C + 1));"),
    ("sigma without abs", "float ad = fabsf(dd);", "float ad = dd;"),
    ("sign flipped", "int S = dd >= 0.0f ? 1 : -1;", "int S = dd >= 0.0f ? -1 : 1;"),
    ("decode chunk index wrong", "int c = t / C;\n        for (int d = 0; d < D; ++d) {\n            size_t byte",
     "int c = t % (P / C);\n        for (int d = 0; d < D; ++d) {\n            size_t byte"),
    ("k-bit decode chunk index wrong",
     "int c = t / C;\n        for (int d = 0; d < D; ++d) {\n            const uint8_t *pa",
     "int c = t % (P / C);\n        for (int d = 0; d < D; ++d) {\n            const uint8_t *pa"),
    ("anchor bucket point 16V", "I = 16 * V + 7;", "I = 16 * V;"),
    ("decode sigma without eps", "float nv = fmaf(xf, sg + ORACLE_EPS, mu);\n            float xv",
     "float nv = fmaf(xf, sg, mu);\n            float xv"),
    ("k-bit decode sigma without eps",
     "float nv = fmaf(xf, sg + ORACLE_EPS, mu);\n            out[(int64_t)t",
     "float nv = fmaf(xf, sg, mu);\n            out[(int64_t)t"),
    ("decode affine operands transposed",
     "float xv = fmaf(nv, g_scale[d] + ORACLE_EPS, g_min[d]);",
     "float xv = fmaf(nv, g_min[d] + ORACLE_EPS, g_scale[d]);"),
    ("attention scale 1/D",
     "double scale = 1.0 / sqrt((double)D);\n    double *s = (double *)malloc(sizeof(double) * (size_t)L);",
     "double scale = 1.0 / (double)D;\n    double *s = (double *)malloc(sizeof(double) * (size_t)L);"),
    ("softmax without the max shift",
     "double w = exp(s[t] - m);\n        l += w;\n        for (int d = 0; d < D; ++d) out[d] += w * (double)V[",
     "double w = exp(s[t]);\n        l += w;\n        for (int d = 0; d < D; ++d) out[d] += w * (double)V["),
    ("attention not normalised", "for (int d = 0; d < D; ++d) out[d] /= l;\n    free(s);\n}\n\n/* One query row",
     "for (int d = 0; d < D; ++d) out[d] /= 1.0;\n    free(s);\n}\n\n/* One query row"),
    ("verification row ignores the draft tokens", "int64_t n = L + n_tail;", "int64_t n = L;"),
    ("acceptance ratio inverted (q/p)", "if (!(u[k] * qv < pv)) break;",
     "if (!(u[k] * pv < qv)) break;"),
    ("correction from max(0, q - p)", "return qk ? fmaxf(pk[x] - qk[x], 0.0f) : pk[x];",
     "return qk ? fmaxf(qk[x] - pk[x], 0.0f) : pk[x];"),
    ("no bonus token: the last draft distribution is reused",
     "const float *pk = p + (int64_t)k * V;", "const float *pk = p + (int64_t)(k < T ? k : T - 1) * V;"),
    ("draft tokens take the cached values",
     "const float *v = t < L ? V + t * kv_stride : Vt + (t - L) * tail_stride;",
     "const float *v = t < L ? V + t * kv_stride : V + (t - L) * kv_stride;"),
    ("INT-B rounds down", "float qf = rintf(dd * rs);", "float qf = floorf(dd * rs);"),
    ("INT-B decode drops the minimum", "out[r * D + d] = fmaf((float)q, S, lo);",
     "out[r * D + d] = fmaf((float)q, S, 0.0f);"),
    ("INT-B with 2^B levels", "const int qmax = (1 << bits) - 1;", "const int qmax = (1 << bits);"),
    ("INT-4 nibbles swapped", "cr[d / 2] |= (uint8_t)(q << ((d & 1) ? 4 : 0));",
     "cr[d / 2] |= (uint8_t)(q << ((d & 1) ? 0 : 4));"),
    ("INT-B scale from the maximum alone", "float S = (hi - lo) / (float)qmax;",
     "float S = hi / (float)qmax;"),
    ("k-bit Anchor shifted by k", "field_put(pa, d % 8, k, (q8 >> rw) & ((1 << k) - 1));",
     "field_put(pa, d % 8, k, (q8 >> k) & ((1 << k) - 1));"),
    ("k-bit bucket point without the -1", "int I = (1 << (8 - k)) * V + (1 << (7 - k)) - 1;",
     "int I = (1 << (8 - k)) * V + (1 << (7 - k));"),
    ("bit fields written high bit first", "uint8_t m = (uint8_t)(1u << (b & 7));",
     "uint8_t m = (uint8_t)(1u << (7 - (b & 7)));"),
    ("A.1 sign dropped", "int Q = xpp > 0.0f ? I : (xpp < 0.0f ? -I : 0);", "int Q = I;"),
    ("A.1 decode without the page maximum",
     "out[(int64_t)t * out_stride + d] = (v * meta[(size_t)(1 + c) * D + d]) * meta[d];",
     "out[(int64_t)t * out_stride + d] = (v * meta[(size_t)(1 + c) * D + d]);"),
    ("A.1 page maximum without |.|", "float a = fabsf(bf16_bits_to_f32(x[(int64_t)t * row_stride + d]));",
     "float a = bf16_bits_to_f32(x[(int64_t)t * row_stride + d]);"),
    ("A.1 Anchor point 16 Q_anc + 8", "qa * 16 + 7;", "qa * 16 + 8;"),
    ("A.1 chunk maximum of x instead of x'", "float a = fabsf(xp[i]);",
     "float a = fabsf(bf16_bits_to_f32(x[(int64_t)t * row_stride + d]));"),
    ("bf16 rounds ties up", "    u += 0x7fffu + lsb;\n    return (uint16_t)(u >> 16);",
     "    u += 0x8000u + 0u * lsb;\n    return (uint16_t)(u >> 16);"),
    ("bf16 truncates", "    u += 0x7fffu + lsb;\n    return (uint16_t)(u >> 16);",
     "    u += 0u * lsb;\n    return (uint16_t)(u >> 16);"),
    ("bf16 tie parity from the dropped bit", "uint32_t lsb = (u >> 16) & 1u;",
     "uint32_t lsb = (u >> 15) & 1u;"),
    ("bf16 NaN not kept", "if ((u & 0x7fffffffu) > 0x7f800000u)\n        return",
     "if (0)\n        return"),
    ("Stage-1 eps 1e-3 in the encoder", "float rg = 1.0f / (gs + ORACLE_EPS);",
     "float rg = 1.0f / (gs + 1e-3f);"),
    ("Stage-2 eps 1e-3 in the encoder", "float rs = 1.0f / (sg + ORACLE_EPS);",
     "float rs = 1.0f / (sg + 1e-3f);"),
    ("Stage-2 eps 1e-5 in the encoder", "float rs = 1.0f / (sg + ORACLE_EPS);",
     "float rs = 1.0f / (sg + 1e-5f);"),
    ("decode Stage-2 eps 1e-3", "float nv = fmaf(xf, sg + ORACLE_EPS, mu);\n            float xv",
     "float nv = fmaf(xf, sg + 1e-3f, mu);\n            float xv"),
    ("decode Stage-1 eps 1e-3", "float xv = fmaf(nv, g_scale[d] + ORACLE_EPS, g_min[d]);",
     "float xv = fmaf(nv, g_scale[d] + 1e-3f, g_min[d]);"),
    ("A.1 chunk maximum + 1e-6 instead of the zero rule",
     "float rmi = mi > 0.0f ? 1.0f / mi : 0.0f;", "float rmi = 1.0f / (mi + 1e-6f);"),
    ("A.1 page maximum + 1e-6 instead of the zero rule",
     "float rm = m > 0.0f ? 1.0f / m : 0.0f;", "float rm = 1.0f / (m + 1e-6f);"),
    ("literal Stage 4 biased by 8", "int I_bias = I + 7;", "int I_bias = I + 8;"),
    ("literal Stage 4 residual sign flipped", "int V_res = V_recon - I;", "int V_res = I - V_recon;"),
    ("expansion without the division by alpha",
     "return (float)((pow(1.0 + al, (double)I / 127.0) - 1.0) / al);",
     "return (float)(pow(1.0 + al, (double)I / 127.0) - 1.0);"),
    ("compander normalised by log(alpha), not log1p(alpha)",
     "return 127.0 * log1p(al * (double)a) / log1p(al);",
     "return 127.0 * log1p(al * (double)a) / log(al);"),
    ("spec integer weights at 2^32", "(uint64_t)(w * 1099511627776.0f)",
     "(uint64_t)(w * 4294967296.0f)"),
]

# representative arguments for the parametrized pins
PARAMS = {"P": 256, "C": 32}


def _pin_functions():
    for name, fn in sorted(vars(pins).items()):
        if name.startswith("test_") and callable(fn):
            yield name, fn


def _run_pins():
    """Names of the pins that fail with the oracle currently swapped in."""
    failed = []
    for name, fn in _pin_functions():
        sig = inspect.signature(fn)
        kwargs = {}
        for p in sig.parameters:
            if p == "oracle_mod":
                kwargs[p] = oracle
            elif p in PARAMS:
                kwargs[p] = PARAMS[p]
            elif p == "alpha":
                kwargs[p] = 255.0
        try:
            fn(**kwargs)
        except Exception:          # noqa: BLE001 - any failure counts
            failed.append(name)
    return failed


def test_the_real_oracle_passes_every_pin():
    assert _run_pins() == []


@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(what, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site not unique: {old}"
    with tempfile.TemporaryDirectory() as d:
        lib = oracle.compile_variant(src.replace(old, new), os.path.join(d, "mutant.so"))
        with oracle.using_library(lib):
            failed = _run_pins()
    assert failed, f"no pin caught: {what}"
