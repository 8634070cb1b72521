"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code path: values printed
on the pages (tests/golden/), closed forms, hand-derived tiny cases,
invariants and error bounds.  Sources: "Lynx: Progressive Speculative KV Cache
Transfer for Disaggregated LLM Inference" (technical review, cited as Review)
and the paper digest page (cited as Digest).
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALPHA = 255.0


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32(x):
    return float(np.float32(x))


# ----------------------------------------------------------- worked example

def test_worked_example_stage3(oracle_mod):
    """Review, Worked Example, Eq. 12-13: x_final = 0.37/0.55, alpha = 255,
    Y ~ 117.9, I = 118."""
    g = golden("worked_example.json")
    xf = f32((g["x_view"] - g["mu"]) / g["sigma"])
    assert abs(xf - g["x_final_printed"]) < 5e-4
    y = oracle_mod.compand_y(xf, g["alpha"])
    # printed 117.9 comes from 4-digit intermediates (5.151/5.545*127 = 117.97)
    assert abs(y - g["Y_printed"]) < 0.1
    assert abs(math.log1p(g["alpha"] * xf) - g["ln_1_plus_alpha_x_printed"]) < 2e-3
    assert oracle_mod.round_code(xf, g["alpha"]) == g["I"]


def test_worked_example_stage4_literal(oracle_mod):
    """Review, Worked Example, Stage 4 trace: 125, 7, 112, -6, Q_anc = 7."""
    g = golden("worked_example.json")
    r = oracle_mod.stage4_literal(g["I"], g["S"])
    assert r == dict(I_bias=g["I_bias"], V_mag=g["V_mag"], V_recon=g["V_recon"],
                     V_res=g["V_res"], Q_anc=g["Q_anc"])
    # decode side of the trace: I = V_recon - V_res recovers 118
    assert r["V_recon"] - r["V_res"] == g["I_full_recovered"]


def test_worked_example_reconstructions(oracle_mod):
    """Review, Eq. 14-15: the closed forms of the printed expressions, and the
    page's claim that the full reconstruction is within 1%."""
    g = golden("worked_example.json")
    xf = f32((g["x_view"] - g["mu"]) / g["sigma"])
    full = oracle_mod.expand(g["I"], g["alpha"])
    assert abs(full - g["full_closed_form_I118"]) < 1e-4
    assert abs(full - xf) / xf < 0.01                       # "< 1%"
    assert abs(full - g["full_reconstruction_printed"]) / full < 0.01
    # Eq. 14's printed expression ((1+a)^(112/127) - 1)/a evaluated exactly
    anc = oracle_mod.expand(g["anchor_only_I_printed"], g["alpha"])
    assert abs(anc - g["anchor_only_closed_form_I112"]) < 1e-4
    assert abs(anc - g["anchor_only_printed"]) > 0.1        # the page's slip
    # 256^(112/127) = 132.98, not the printed 187
    assert abs((1 + g["alpha"]) ** (112 / 127) - 132.98) < 0.01


# ----------------------------------------------------------- Stage 4 / Eq. 9

def test_stage4_split_is_a_bijection(oracle_mod):
    """Review, Stage 4 and Eq. 9: the (sign, magnitude) code splits into an
    Anchor nibble and a Residual nibble with Anchor<<4 | Residual == code,
    every one of the 256 pairs used once; the Anchor is Eq. 9 applied to the
    top magnitude bits V = I >> 4 as a 4-bit two's complement."""
    seen = set()
    for S in (1, -1):
        for I in range(128):
            c8 = oracle_mod.code8(I, S)
            a = oracle_mod.anchor_nibble(c8)
            r = oracle_mod.residual_nibble(c8)
            assert 0 <= a < 16 and 0 <= r < 16
            assert (a << 4) | r == c8
            seen.add((a, r))
            a_signed = a - 16 if a >= 8 else a
            V = I >> 4
            assert a_signed == V * S + min(S, 0)            # Eq. 9
            if S > 0:
                assert 0 <= a_signed <= 7
            else:
                assert -8 <= a_signed <= -1
    assert len(seen) == 256
    # the page's special case: V_mag = 0 with S = -1 maps to Q_anc = -1
    assert oracle_mod.anchor_nibble(oracle_mod.code8(0, -1)) == 0xF


def test_literal_stage4_needs_a_fifth_bit(oracle_mod):
    """Review, Stage 4: with the +7 bias, I >= 121 gives V_mag = 8, so the
    Anchor as printed takes 18 values (it states [0,15] and [-16,-1]); the
    codec therefore applies Eq. 9 to the 8-bit code (the design's reading)."""
    vals = set()
    for S in (1, -1):
        for I in range(128):
            vals.add(oracle_mod.stage4_literal(I, S)["Q_anc"])
    assert len(vals) == 18
    assert oracle_mod.stage4_literal(121, 1)["V_mag"] == 8
    assert oracle_mod.stage4_literal(120, 1)["V_mag"] == 7
    # its residual always fits a signed nibble
    for I in range(128):
        assert -8 <= oracle_mod.stage4_literal(I, 1)["V_res"] <= 7


# ----------------------------------------------------------- Eq. 7 compander

def test_compander_closed_form(oracle_mod):
    """Eq. 7: Y(0) = 0, Y(1) = 127, strictly increasing."""
    assert oracle_mod.compand_y(0.0, ALPHA) == 0.0
    assert abs(oracle_mod.compand_y(1.0, ALPHA) - 127.0) < 1e-12
    xs = np.linspace(0, 1, 2001, dtype=np.float32)
    ys = [oracle_mod.compand_y(float(x), ALPHA) for x in xs]
    assert all(b > a for a, b in zip(ys, ys[1:]))
    assert oracle_mod.round_code(0.0, ALPHA) == 0
    assert oracle_mod.round_code(1.0, ALPHA) == 127


def test_compander_small_alpha_is_linear_quantizer(oracle_mod):
    """As alpha -> 0, ln(1+alpha x)/ln(1+alpha) -> x: the code becomes the
    textbook 7-bit linear magnitude quantizer round(127 |x|)."""
    rng = np.random.default_rng(1)
    xs = rng.random(4000).astype(np.float32)
    frac = (127 * xs.astype(np.float64)) % 1.0
    keep = np.abs(frac - 0.5) > 1e-3          # away from rounding boundaries
    for x in xs[keep]:
        assert oracle_mod.round_code(float(x), 1e-7) == int(np.rint(127 * float(x)))


def test_expand_inverts_compand(oracle_mod):
    """Eq. 14/15 is the inverse of Eq. 7: Round(Y(X(I))) == I for all I."""
    for alpha in (100.0, 255.0, 2000.0):
        for I in range(128):
            x = oracle_mod.expand(I, alpha)
            assert abs(oracle_mod.compand_y(x, alpha) - I) < 1e-3
            assert oracle_mod.round_code(x, alpha) == I
        assert oracle_mod.expand(0, alpha) == 0.0
        assert abs(oracle_mod.expand(127, alpha) - 1.0) < 1e-6


def test_anchor_levels_are_geometric(oracle_mod):
    """Digest, Method: the Anchor is a geometric-interval exponent,
    (1+alpha)^q.  With the bucket points 16V+7, (X + 1/alpha) grows by
    (1+alpha)^(16/127) per Anchor step."""
    for alpha in (100.0, 255.0):
        ratio = oracle_mod.anchor_ratio(alpha)
        for V in range(7):
            lo = oracle_mod.expand(16 * V + 7, alpha) + 1.0 / alpha
            hi = oracle_mod.expand(16 * V + 23, alpha) + 1.0 / alpha
            assert abs(hi / lo - ratio) < 1e-5 * ratio
    assert abs(oracle_mod.anchor_ratio(255.0) - 2.011) < 1e-3


# ----------------------------------------------------------- tiny hand cases

def _bf16_bits(vals):
    a = np.asarray(vals, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)   # exact for these values


def _hand_block():
    """P=4, D=8: channel 0 = [0,1,2,3], channels 1..7 constant."""
    cols = [_bf16_bits([0, 1, 2, 3])] + [_bf16_bits([5 + k] * 4) for k in range(7)]
    return np.stack(cols, axis=1)


def test_encode_hand_case(oracle_mod):
    """P=4, C=2, D=8.  Channel 0 = [0,1,2,3]: each chunk has two values, so
    after centring they sit at -sigma and +sigma, |X_final| ~ 1 - 1e-5 and
    I = 127: code8 = 128 (S=-1) then 127 (S=+1).  Channels 1..7 are constant:
    gamma_scale = 0, every value normalises to 0, so I = 0, S = +1, code 0.
    Channel 0 is the low nibble of byte 0 (it shares the byte with channel 4)."""
    anc, res, meta = oracle_mod.encode_block(_hand_block(), C=2, alpha=ALPHA)
    assert anc[:, 0].tolist() == [0x08, 0x07, 0x08, 0x07]
    assert res[:, 0].tolist() == [0x00, 0x0F, 0x00, 0x0F]
    assert (anc[:, 1:] == 0).all() and (res[:, 1:] == 0).all()
    assert meta[0].tolist() == [0.0] + [5.0 + k for k in range(7)]   # gamma_min
    assert meta[1].tolist() == [3.0] + [0.0] * 7                      # gamma_scale
    # mu per chunk: (0 + 1/3)/2 and (2/3 + 1)/2 ; sigma = 1/6
    assert abs(meta[2, 0] - 1 / 6) < 1e-6 and abs(meta[3, 0] - 5 / 6) < 1e-6
    assert abs(meta[4, 0] - 1 / 6) < 1e-6 and abs(meta[5, 0] - 1 / 6) < 1e-6
    assert (meta[2:, 1:] == 0).all()


def test_encode_nibble_pairing(oracle_mod):
    """The byte shared by channels 8G+k and 8G+k+4: moving the ramp of the hand
    case to channel 4 moves its code to the high nibble of byte 0, and to
    channel 9 the low nibble of byte 5."""
    base = _hand_block()
    flat = np.repeat(base[:, 1:2], 8, axis=1)          # constant channels
    x = np.concatenate([base, flat], axis=1)          # D = 16, ramp at 0
    x[:, [0, 4]] = x[:, [4, 0]]
    anc, res, _ = oracle_mod.encode_block(x, C=2, alpha=ALPHA)
    assert anc[:, 0].tolist() == [0x80, 0x70, 0x80, 0x70]
    assert res[:, 0].tolist() == [0x00, 0xF0, 0x00, 0xF0]
    x = np.concatenate([base, flat], axis=1)
    x[:, [0, 9]] = x[:, [9, 0]]
    anc, res, _ = oracle_mod.encode_block(x, C=2, alpha=ALPHA)
    assert anc[:, 5].tolist() == [0x08, 0x07, 0x08, 0x07]
    assert (np.delete(anc, 5, axis=1) == 0).all()


def test_negative_zero_extreme_is_canonical(oracle_mod):
    """A page whose minimum is a zero stores -0 whichever zero comes first,
    and zero values then centre to +0: S = +1, I = 0, code 0."""
    a = np.stack([_bf16_bits([-0.0, 0.0, 1.0, 2.0])] * 8, axis=1)
    b = np.stack([_bf16_bits([0.0, -0.0, 1.0, 2.0])] * 8, axis=1)
    ra = oracle_mod.encode_block(a, C=2, alpha=ALPHA)
    rb = oracle_mod.encode_block(b, C=2, alpha=ALPHA)
    for u, v in zip(ra, rb):
        assert u.tobytes() == v.tobytes()
    assert np.signbit(ra[2][0]).all()
    z = np.stack([_bf16_bits([-0.0, 0.0, -0.0, 0.0])] * 8, axis=1)
    anc, res, meta = oracle_mod.encode_block(z, C=2, alpha=ALPHA)
    assert (anc == 0).all() and (res == 0).all()


def test_decode_hand_case(oracle_mod):
    """Decode of the hand case.  Full: I = 127 decodes to |x_final| = 1, so the
    values come back within fp32 noise; the constant channels are exact.
    Anchor-only: V = 7 uses the bucket point 16*7+7 = 119."""
    x = _hand_block()
    anc, res, meta = oracle_mod.encode_block(x, C=2, alpha=ALPHA)
    full = oracle_mod.decode_block(anc, res, meta, C=2, alpha=ALPHA)
    assert np.allclose(full[:, 0], [0, 1, 2, 3], atol=1e-4)
    assert (full[:, 1:] == oracle_mod.bf16_bits_to_f32(x[:, 1:]).reshape(4, 7)).all()
    part = oracle_mod.decode_block(anc, None, meta, C=2, alpha=ALPHA)
    x119 = oracle_mod.expand(119, ALPHA)
    assert abs(x119 - 0.70402) < 1e-4
    half = (1 / 6 + 1e-6) * x119
    want = (3 + 1e-6) * np.array([1 / 6 - half, 1 / 6 + half,
                                  5 / 6 - half, 5 / 6 + half])
    assert np.allclose(part[:, 0], want, atol=1e-4), (part[:, 0], want)
    assert (part[:, 1:] == full[:, 1:]).all()


def test_decode_inverts_normalisation_at_chunk_extremes(oracle_mod):
    """At a chunk's extreme |d| = sigma the code is I = 127 and X(127) = 1
    exactly (Eq. 14/15), so the decoder must give back
    gamma_min + (gamma_scale + eps) * (mu +- (sigma + eps)): the exact inverse
    of dividing by (sigma + eps) and (gamma_scale + eps) (Stages 1-2)."""
    assert oracle_mod.expand(127, ALPHA) == 1.0
    anc, res, meta = oracle_mod.encode_block(_hand_block(), C=2, alpha=ALPHA)
    full = oracle_mod.decode_block(anc, res, meta, C=2, alpha=ALPHA)
    gm, gs = float(meta[0, 0]), float(meta[1, 0])
    eps = float(np.float32(1e-6))
    for t in range(4):
        c = t // 2
        mu, sg = float(meta[2 + c, 0]), float(meta[4 + c, 0])
        sign = -1.0 if t % 2 == 0 else 1.0
        want = gm + (np.float32(gs + eps)) * (mu + sign * float(np.float32(sg + eps)))
        assert abs(full[t, 0] - want) <= 2 * np.spacing(np.float32(abs(want)) + 1e-30), (t, full[t, 0], want)


# ----------------------------------------------------------- random blocks

def _random_block(seed, P=256, D=128, outliers=(3, 77)):
    rng = np.random.default_rng(seed)
    lap = rng.laplace(size=(P, D)).astype(np.float32)
    s = np.exp(0.5 * rng.standard_normal(D)).astype(np.float32)
    o = np.ones(D, np.float32)
    o[list(outliers)] = 100.0
    import oracle
    return oracle.f32_to_bf16_bits((lap * s * o).astype(np.float32))


def _signed_codes(anc, res):
    """Q8 as signed int8 for [P][D] from packed nibbles (Anchor<<4|Residual);
    byte 4G+k of a row holds channels 8G+k (low) and 8G+k+4 (high)."""
    P, half = anc.shape
    a = anc.reshape(P, half // 4, 4)
    r = res.reshape(P, half // 4, 4)
    c = np.empty((P, half // 4, 8), np.uint8)
    c[:, :, 0:4] = ((a & 0xF) << 4) | (r & 0xF)
    c[:, :, 4:8] = (a & 0xF0) | (r >> 4)
    return c.reshape(P, half * 2).view(np.int8).astype(np.int32)


def _magnitudes(q8):
    S = np.where(q8 >= 0, 1, -1)
    I = np.where(S > 0, q8, -q8 - 1)
    return S, I


@pytest.mark.parametrize("P,C", [(256, 32), (128, 32), (256, 64), (64, 16)])
def test_encode_invariants(oracle_mod, P, C):
    """Stage 1: gamma_min is the page minimum and gamma_scale the range.
    Stage 2: mu, sigma lie in [0, 1].  Each chunk-channel with sigma > 0
    reaches |X_final| ~ 1, i.e. I = 127.  Codes are monotone in x within a
    chunk-channel (the sign map of Eq. 9 keeps order)."""
    bits = _random_block(P + C, P=P)
    x = oracle_mod.bf16_bits_to_f32(bits).reshape(P, 128)
    anc, res, meta = oracle_mod.encode_block(bits.reshape(P, 128), C, ALPHA)
    NC = P // C
    assert np.array_equal(meta[0], x.min(axis=0))
    assert np.array_equal(meta[1], (x.max(axis=0) - x.min(axis=0)).astype(np.float32))
    mu, sg = meta[2:2 + NC], meta[2 + NC:]
    assert (mu >= 0).all() and (mu <= 1).all() and (sg >= 0).all() and (sg <= 1).all()
    q8 = _signed_codes(anc, res)
    S, I = _magnitudes(q8)
    for c in range(NC):
        blkI = I[c * C:(c + 1) * C]
        assert (blkI.max(axis=0)[sg[c] > 1e-3] == 127).all()
        for d in range(128):
            xs = x[c * C:(c + 1) * C, d]
            qs = q8[c * C:(c + 1) * C, d]
            order = np.argsort(xs, kind="stable")
            assert (np.diff(qs[order]) >= 0).all() or np.unique(xs).size < C
            # ties in x must share a code
            for v in np.unique(xs):
                assert np.unique(qs[xs == v]).size == 1



def test_range_layout_is_batch_page_head(oracle_mod):
    """encode() / decode() over a [B][L][H][D] tensor: block (b, p, h) of the
    streams is tokens p*P .. p*P + P - 1 of head h of batch b, encoded alone,
    and decode() writes it back to the same tokens and head."""
    B, NB, H, P, C = 2, 3, 2, 64, 16
    L = NB * P
    rng = np.random.default_rng(11)
    x = (rng.laplace(size=(B, L, H, 128)) *
         rng.uniform(0.5, 4.0, size=(1, 1, H, 128))).astype(np.float32)
    bits = oracle_mod.f32_to_bf16_bits(x).reshape(B, L, H, 128)
    anc, res, meta = oracle_mod.encode(bits, P, C, ALPHA)
    dec = oracle_mod.decode(anc, res, meta, L, P, C, ALPHA)
    for b in range(B):
        for p in range(NB):
            for h in range(H):
                a1, r1, m1 = oracle_mod.encode_block(bits[b, p * P:(p + 1) * P, h], C, ALPHA)
                assert np.array_equal(anc[b, p, h], a1), (b, p, h)
                assert np.array_equal(res[b, p, h], r1), (b, p, h)
                assert np.array_equal(meta[b, p, h], m1), (b, p, h)
                d1 = oracle_mod.decode_block(a1, r1, m1, C, ALPHA)
                assert np.array_equal(dec[b, p * P:(p + 1) * P, h], d1), (b, p, h)


def test_variant_range_layouts(oracle_mod):
    """The k-bit Anchor decode and the A.1 codec over a [B][L][H][D] tensor
    agree, block by block, with the same call on that block alone (a single
    block has no batch, page or head index to get wrong)."""
    B, NB, H, P, C, k = 2, 3, 2, 64, 16, 5
    L = NB * P
    rng = np.random.default_rng(13)
    x = (rng.laplace(size=(B, L, H, 128)) *
         rng.uniform(0.5, 4.0, size=(1, 1, H, 128))).astype(np.float32)
    bits = oracle_mod.f32_to_bf16_bits(x).reshape(B, L, H, 128)
    anc, res, meta = oracle_mod.encode(bits, P, C, ALPHA)
    ak, _ = oracle_mod.split_bits(anc, res, k)
    dk = oracle_mod.decode_anchor_bits(ak, meta, L, P, C, ALPHA, k)
    a1 = oracle_mod.a1_encode(bits, P)
    d1 = oracle_mod.a1_decode(*a1, L, P)
    for b in range(B):
        for p in range(NB):
            for h in range(H):
                blk = (slice(b, b + 1), slice(p, p + 1), slice(h, h + 1))
                tok = (b, slice(p * P, (p + 1) * P), h)
                one = oracle_mod.decode_anchor_bits(ak[blk], meta[blk], P, P, C, ALPHA, k)
                assert np.array_equal(dk[tok], one[0, :, 0]), (b, p, h)
                e1 = oracle_mod.a1_encode(bits[b:b + 1, p * P:(p + 1) * P, h:h + 1], P)
                for full, part in zip(a1, e1):
                    assert np.array_equal(full[blk], part), (b, p, h)
                assert np.array_equal(d1[tok], oracle_mod.a1_decode(*e1, P, P)[0, :, 0]), (b, p, h)

def _X(y, alpha=ALPHA):
    """Continuous inverse of Eq. 7 (for the half-code boundaries)."""
    return (np.power(1.0 + alpha, np.asarray(y, np.float64) / 127.0) - 1.0) / alpha


@pytest.mark.parametrize("P,C", [(256, 32), (128, 32), (256, 64)])
def test_full_decode_within_one_code_step(oracle_mod, P, C):
    """Full reconstruction error is at most one code step: x_final lies in
    [X(I-1/2), X(I+1/2)] and the decoder returns X(I), scaled back by
    (sigma+eps)(gamma_scale+eps) (plus float32 noise)."""
    bits = _random_block(11 + P + C, P=P).reshape(P, 128)
    x = oracle_mod.bf16_bits_to_f32(bits).reshape(P, 128).astype(np.float64)
    anc, res, meta = oracle_mod.encode_block(bits, C, ALPHA)
    xh = oracle_mod.decode_block(anc, res, meta, C, ALPHA).astype(np.float64)
    NC = P // C
    _, I = _magnitudes(_signed_codes(anc, res))
    gs = meta[1].astype(np.float64) + 1e-6
    sg = np.repeat(meta[2 + NC:].astype(np.float64), C, axis=0) + 1e-6
    step = _X(np.minimum(I + 0.5, 127.0)) - _X(np.maximum(I - 0.5, 0.0))
    bound = step * sg * gs + 4e-7 * (np.abs(x) + gs)
    assert (np.abs(xh - x) <= bound).all()


@pytest.mark.parametrize("P,C", [(256, 32), (128, 32)])
def test_anchor_decode_within_its_bucket(oracle_mod, P, C):
    """Anchor-only reconstruction lies in the same geometric bucket
    [X(16V - 1/2), X(16V + 15 + 1/2)] as the true value, and its error is
    never below the full reconstruction's for the same element."""
    bits = _random_block(23 + P, P=P).reshape(P, 128)
    x = oracle_mod.bf16_bits_to_f32(bits).reshape(P, 128).astype(np.float64)
    anc, res, meta = oracle_mod.encode_block(bits, C, ALPHA)
    xa = oracle_mod.decode_block(anc, None, meta, C, ALPHA).astype(np.float64)
    NC = P // C
    _, I = _magnitudes(_signed_codes(anc, res))
    V = I >> 4
    gs = meta[1].astype(np.float64) + 1e-6
    sg = np.repeat(meta[2 + NC:].astype(np.float64), C, axis=0) + 1e-6
    width = _X(np.minimum(16 * V + 15.5, 127.0)) - _X(np.maximum(16 * V - 0.5, 0.0))
    bound = width * sg * gs + 4e-7 * (np.abs(x) + gs)
    assert (np.abs(xa - x) <= bound).all()
    # anchor-only error is larger on average (it drops the residual bits)
    xf = oracle_mod.decode_block(anc, res, meta, C, ALPHA).astype(np.float64)
    assert np.abs(xa - x).mean() > 3 * np.abs(xf - x).mean()


def test_sign_flip_symmetry(oracle_mod):
    """x -> -x mirrors every chunk: S flips and I is kept, so Q8 -> -Q8 - 1,
    except where float32 rounding moves Y across a half-integer."""
    bits = _random_block(5).reshape(256, 128)
    neg = bits ^ np.uint16(0x8000)
    a1, r1, _ = oracle_mod.encode_block(bits, 32, ALPHA)
    a2, r2, _ = oracle_mod.encode_block(neg, 32, ALPHA)
    q1, q2 = _signed_codes(a1, r1), _signed_codes(a2, r2)
    S1, I1 = _magnitudes(q1)
    S2, I2 = _magnitudes(q2)
    same = (q2 == -q1 - 1)
    assert same.mean() > 0.99
    assert (np.abs(I1 - I2) <= 1).all()


def test_scale_invariance(oracle_mod):
    """Codes depend on x only through the two normalisations, so scaling a
    page by 2 keeps them (up to eps and float32 rounding near boundaries)."""
    bits = _random_block(9).reshape(256, 128)
    x = oracle_mod.bf16_bits_to_f32(bits).reshape(256, 128)
    bits2 = oracle_mod.f32_to_bf16_bits(x * 2)
    a1, r1, m1 = oracle_mod.encode_block(bits, 32, ALPHA)
    a2, r2, m2 = oracle_mod.encode_block(bits2, 32, ALPHA)
    assert np.array_equal(m2[0], 2 * m1[0]) and np.array_equal(m2[1], 2 * m1[1])
    q1, q2 = _signed_codes(a1, r1), _signed_codes(a2, r2)
    assert (q1 == q2).mean() > 0.99
    assert (np.abs(q1 - q2) <= 1).all()


def test_laplacian_mass_near_zero(oracle_mod):
    """Review, Stage 3: about half of the centred values have |x| < 0.17.
    I <= Round(Y(0.17)) counts them on synthetic Laplacian KV."""
    g = golden("size_examples.json")["laplacian_mass"]
    import torch
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(2, 512, 2, 128, seed=0)
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    anc, res, meta = oracle_mod.encode(bits, 128, 32, ALPHA)
    q8 = _signed_codes(anc.reshape(-1, 64), res.reshape(-1, 64))
    _, I = _magnitudes(q8)
    cut = oracle_mod.compand_y(g["threshold"], ALPHA)
    frac = (I < cut).mean()
    assert abs(frac - g["printed_fraction"]) < 0.08


# ----------------------------------------------------------- attention

def test_attention_single_token(oracle_mod):
    rng = np.random.default_rng(0)
    q, k, v = (rng.standard_normal((1, 128)).astype(np.float32) for _ in range(3))
    out = oracle_mod.attention_row(q[0], k, v)
    assert np.array_equal(out, v[0].astype(np.float64))


def test_attention_identical_keys_give_mean(oracle_mod):
    rng = np.random.default_rng(1)
    q = rng.standard_normal(128).astype(np.float32)
    k = np.tile(rng.standard_normal(128).astype(np.float32), (7, 1))
    v = rng.standard_normal((7, 128)).astype(np.float32)
    out = oracle_mod.attention_row(q, k, v)
    assert np.allclose(out, v.astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)


def test_attention_two_tokens_hand_weights(oracle_mod):
    """Scores differing by ln 3 give softmax weights 3/4 and 1/4 (Eq. 1)."""
    D = 128
    q = np.zeros(D, np.float32)
    q[0] = 1.0
    k = np.zeros((2, D), np.float32)
    k[0, 0] = np.float32(math.log(3.0) * math.sqrt(D))
    v = np.zeros((2, D), np.float32)
    v[0, :] = 4.0
    v[1, :] = 8.0
    out = oracle_mod.attention_row(q, k, v)
    w0 = 3.0 / 4.0
    assert np.allclose(out, w0 * 4.0 + (1 - w0) * 8.0, atol=1e-6)


def test_attention_invariances(oracle_mod):
    """Token order does not matter; adding one vector to every key shifts all
    scores equally and leaves the output unchanged."""
    rng = np.random.default_rng(2)
    L, D = 50, 128
    q = rng.standard_normal(D).astype(np.float32)
    k = rng.standard_normal((L, D)).astype(np.float32)
    v = rng.standard_normal((L, D)).astype(np.float32)
    out = oracle_mod.attention_row(q, k, v)
    perm = rng.permutation(L)
    assert np.allclose(oracle_mod.attention_row(q, k[perm], v[perm]), out,
                       atol=1e-12)
    shift = np.zeros(D, np.float32)
    shift[3] = 2.0  # exact in float32 addition for these magnitudes
    out2 = oracle_mod.attention_row(q, (k + shift).astype(np.float32), v)
    assert np.allclose(out2, out, atol=1e-6)


def test_attention_tail_is_the_concatenated_sequence(oracle_mod):
    """The verification row of draft position t attends to the cached tokens
    and to the draft's own tokens 0..t (Review, Mechanism 3, single parallel
    verification pass): the same as plain attention over the concatenation."""
    rng = np.random.default_rng(3)
    L, T, D = 20, 4, 128
    q = rng.standard_normal(D).astype(np.float32)
    k, v = (rng.standard_normal((L, D)).astype(np.float32) for _ in range(2))
    kt, vt = (rng.standard_normal((T, D)).astype(np.float32) for _ in range(2))
    for n in range(T + 1):
        got = oracle_mod.attention_row_tail(q, k, v, kt, vt, n)
        want = oracle_mod.attention_row(q, np.concatenate([k, kt[:n]]), np.concatenate([v, vt[:n]]))
        assert np.allclose(got, want, rtol=0, atol=1e-12), n


def test_attention_tail_is_causal(oracle_mod):
    """Draft tokens after the row's own position take no part: changing the
    later tail tokens leaves the row unchanged, and a dominant later token
    changes only the rows that see it."""
    rng = np.random.default_rng(4)
    L, T, D = 9, 3, 128
    q = rng.standard_normal(D).astype(np.float32)
    k, v = (rng.standard_normal((L, D)).astype(np.float32) for _ in range(2))
    kt, vt = (rng.standard_normal((T, D)).astype(np.float32) for _ in range(2))
    row1 = oracle_mod.attention_row_tail(q, k, v, kt, vt, 2)
    kt2, vt2 = kt.copy(), vt.copy()
    kt2[2] = (q * 50.0).astype(np.float32)      # dominant score for draft token 2
    vt2[2] = 7.0
    assert np.array_equal(oracle_mod.attention_row_tail(q, k, v, kt2, vt2, 2), row1)
    assert np.allclose(oracle_mod.attention_row_tail(q, k, v, kt2, vt2, 3), 7.0, atol=1e-9)


def test_attention_tail_hand_weights(oracle_mod):
    """One cached token with score 0 and one draft token with score ln 3:
    weights 1/4 and 3/4 (Eq. 1)."""
    D = 128
    q = np.zeros(D, np.float32)
    q[0] = 1.0
    k = np.zeros((1, D), np.float32)
    kt = np.zeros((1, D), np.float32)
    kt[0, 0] = np.float32(math.log(3.0) * math.sqrt(D))
    v = np.full((1, D), 4.0, np.float32)
    vt = np.full((1, D), 8.0, np.float32)
    out = oracle_mod.attention_row_tail(q, k, v, kt, vt, 1)
    assert np.allclose(out, 0.25 * 4.0 + 0.75 * 8.0, atol=1e-6)


# ---------------------------------------------------- Eq. 10-11 (Mechanism 3)

def _one(oracle_mod, p, q, s, u, r):
    k, tok = oracle_mod.spec_verify(np.array([p], np.float32), np.array([q], np.float32),
                                    np.array([s], np.int32), np.array([u], np.float32),
                                    np.array([r], np.uint32))
    return int(k[0]), int(tok[0])


def test_spec_inverse_cdf_on_exact_weights(oracle_mod):
    """Every draft token accepted (p = q), so the next token comes from
    p_{T+1} = (1/8, 3/8, 0, 1/2): r = j * 2^29 lands on the j/8 quantile."""
    same = [0.25, 0.25, 0.25, 0.25]
    last = [0.125, 0.375, 0.0, 0.5]
    got = [_one(oracle_mod, [same, last], [same], [2], [0.999], j << 29) for j in range(8)]
    assert got == [(1, t) for t in (0, 1, 1, 1, 3, 3, 3, 3)]


def test_spec_accept_rule(oracle_mod):
    """Eq. 10: accepted iff u < p(s)/q(s), decided as u*q < p in float32."""
    p = [0.2, 0.8]
    nxt = [1.0, 0.0]
    assert _one(oracle_mod, [p, nxt], [[0.4, 0.6]], [0], [0.5], 0)[0] == 0   # 0.5*0.4 = 0.2
    p_up = [float(np.nextafter(np.float32(0.2), np.float32(1))), 0.8]
    assert _one(oracle_mod, [p_up, nxt], [[0.4, 0.6]], [0], [0.5], 0)[0] == 1
    assert _one(oracle_mod, [[0.0, 1.0], nxt], [[0.5, 0.5]], [0], [0.0], 0)[0] == 0
    assert _one(oracle_mod, [[0.3, 0.7], nxt], [[0.3, 0.7]], [1], [0.99999994], 0)[0] == 1


def test_spec_correction_is_the_positive_part(oracle_mod):
    """Eq. 11: after a rejection only tokens with p > q can be drawn, with
    weight p - q."""
    p, q = [0.5, 0.5, 0.0, 0.0], [0.25, 0.75, 0.0, 0.0]
    for r in (0, 1 << 31, (1 << 32) - 1):
        assert _one(oracle_mod, [p, p], [q], [1], [0.9], r) == (0, 0)


def test_spec_output_follows_the_target_distribution(oracle_mod):
    """Losslessness (Mechanism 3): with drafts drawn from q, the emitted tokens
    follow p.  Two draft positions with independent distributions: the first
    emitted token ~ p_1, and the second (whenever the first draft was kept)
    ~ p_2.  200,000 seeded sequences, every frequency within 5 sigma."""
    rng = np.random.default_rng(12)
    V, T, N = 6, 2, 200_000
    p = rng.dirichlet(np.ones(V), size=T + 1).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=T).astype(np.float32)
    s = np.stack([rng.choice(V, size=N, p=q[t] / q[t].sum()) for t in range(T)], axis=1)
    u = rng.random((N, T), dtype=np.float32)
    r = rng.integers(0, 2 ** 32, size=N, dtype=np.uint64).astype(np.uint32)
    k, tok = oracle_mod.spec_verify(np.broadcast_to(p, (N, T + 1, V)),
                                    np.broadcast_to(q, (N, T, V)), s, u, r)
    first = np.where(k >= 1, s[:, 0], tok)
    kept = k >= 1
    second = np.where(k[kept] >= 2, s[kept, 1], tok[kept])
    for emitted, target in ((first, p[0]), (second, p[1])):
        n = emitted.size
        freq = np.bincount(emitted, minlength=V) / n
        pt = target.astype(np.float64) / target.sum()
        sigma = np.sqrt(pt * (1 - pt) / n)
        assert np.all(np.abs(freq - pt) <= 5 * sigma + 1e-12), (freq, pt)



def test_spec_batch_is_its_sequences(oracle_mod):
    """A batch of sequences with their own p, q, drafts, uniforms and seeds
    gives, sequence by sequence, what each gives alone (a batch of one has
    no stride or seed to get wrong)."""
    rng = np.random.default_rng(14)
    N, T, V = 24, 3, 7
    p = rng.dirichlet(np.ones(V), size=(N, T + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(N, T)).astype(np.float32)
    s = rng.integers(0, V, size=(N, T)).astype(np.int32)
    u = rng.random((N, T), dtype=np.float32)
    r = rng.integers(0, 2 ** 32, size=N, dtype=np.uint64).astype(np.uint32)
    k, tok = oracle_mod.spec_verify(p, q, s, u, r)
    for b in range(N):
        kb, tb = oracle_mod.spec_verify(p[b:b + 1], q[b:b + 1], s[b:b + 1], u[b:b + 1],
                                        r[b:b + 1])
        assert (k[b], tok[b]) == (kb[0], tb[0]), b
    assert len(set(zip(k.tolist(), tok.tolist()))) > 1   # the sequences differ

# ----------------------------------------------------------- size formulas

def test_kv_size_example(oracle_mod):
    """Review, Eq. 3: Qwen3-235B-A22B at 128K is about 23.5 (binary) GB;
    at 100 / 25 Gbps that takes about 1.9 / 7.5 s."""
    g = golden("size_examples.json")["kv_size"]
    n = oracle_mod.kv_size_bytes(g["k_factor"], g["L"], g["H_heads"] * g["D_head"],
                                 g["n_layers"], g["precision_bytes"])
    assert n == 25_232_932_864
    assert abs(n / 2 ** 30 - g["printed_size"]) < 0.01
    assert abs(23.5e9 * 8 / 100e9 - g["transfer_100gbps_printed_s"]) < 0.05
    assert abs(23.5e9 * 8 / 25e9 - g["transfer_25gbps_printed_s"]) < 0.05


def test_metadata_overhead_example(oracle_mod):
    """Review, grouped-quantization deep dive: 2304 scalars (9 KB float32) per
    H=128, P=256, C=32 page against a 65 KB BF16 page: 14%."""
    g = golden("size_examples.json")["metadata"]
    n = oracle_mod.metadata_scalars(g["H"], g["P"], g["C"])
    assert n == g["printed_scalars"]
    assert round(n * 4 / 1024) == g["printed_meta_kb"]
    page = g["H"] * g["P"] * 2
    assert page // 1000 == g["printed_page_kb"]       # 65,536 B printed as 65 KB
    assert round(100 * n * 4 / page) == g["printed_overhead_percent"]
    assert oracle_mod.meta_rows(g["P"], g["C"]) * g["H"] == n


def test_effective_bins_example(oracle_mod):
    g = golden("size_examples.json")["effective_bins"]
    assert abs(oracle_mod.effective_bins(g["B"], 1 / g["m_over_m_i"])
               - g["printed_bins"]) < 1e-12


# ----------------------------------------------------------- bit splits

def _fields(packed, w):
    """Little-endian w-bit fields of each aligned group of 8 channels:
    [rows][D*w/8] bytes -> [rows][D] unsigned values."""
    rows, nbytes = packed.shape
    groups = nbytes // w
    out = np.zeros((rows, groups * 8), np.int64)
    for g in range(groups):
        word = np.zeros(rows, np.int64)
        for i in range(w):
            word |= packed[:, g * w + i].astype(np.int64) << (8 * i)
        for j in range(8):
            out[:, g * 8 + j] = (word >> (j * w)) & ((1 << w) - 1)
    return out


def test_bit_splits_recompose_the_code(oracle_mod):
    """Concrete Improvement Suggestions, items 4-5 (splits 3+5 .. 6+2): for
    every split, Anchor << (8-k) | Residual is the same signed 8-bit code,
    the Anchor is its arithmetic top k bits, and k = 4 gives the 4+4
    Anchor of Stage 4."""
    P = 64
    bits = _random_block(11, P=P)
    anc, res, meta = oracle_mod.encode(bits.reshape(1, P, 1, 128), P, 16, ALPHA)
    q8 = _signed_codes(anc.reshape(P, 64), res.reshape(P, 64))
    assert set(np.unique(q8 & 0xFF)) == set(range(256)) or len(np.unique(q8)) > 200
    for k in (3, 4, 5, 6):
        ak, rk = oracle_mod.split_bits(anc, res, k)
        assert ak.shape[-1] == 128 * k // 8 and rk.shape[-1] == 128 * (8 - k) // 8
        a = _fields(ak.reshape(P, -1), k)
        r = _fields(rk.reshape(P, -1), 8 - k)
        a_signed = np.where(a >= 1 << (k - 1), a - (1 << k), a)
        assert np.array_equal(a_signed, q8 >> (8 - k))            # arithmetic shift
        assert np.array_equal(a_signed * (1 << (8 - k)) + r, q8)
        if k == 4:
            assert np.array_equal(a_signed, q8 >> 4)


def test_k_bit_anchor_decode_is_the_bucket_point(oracle_mod):
    """Anchor-only reconstruction of a k-bit Anchor is the full decode of the
    code whose residual is the bucket point: 2^(7-k) - 1 below a
    non-negative Anchor (I_rep = 2^(8-k) V + 2^(7-k) - 1), 2^(7-k) below a
    negative one (the same magnitude, Eq. 9's sign map).  k = 4 is the
    Anchor decode of Stage 4 (16 V + 7)."""
    P, C = 64, 16
    bits = _random_block(12, P=P)
    anc, res, meta = oracle_mod.encode(bits.reshape(1, P, 1, 128), P, C, ALPHA)
    q8 = _signed_codes(anc.reshape(P, 64), res.reshape(P, 64))
    for k in (3, 4, 5, 6):
        ak, _ = oracle_mod.split_bits(anc, res, k)
        got = oracle_mod.decode_anchor_bits(ak, meta, P, P, C, ALPHA, k)
        a = q8 >> (8 - k)
        rep = a * (1 << (8 - k)) + np.where(a >= 0, (1 << (7 - k)) - 1, 1 << (7 - k))
        u = (rep & 0xFF).astype(np.uint8)
        # back to the 4+4 nibble streams (byte 4G+j: channels 8G+j, 8G+j+4)
        u = u.reshape(P, 16, 8)
        a4 = ((u[:, :, 0:4] >> 4) | (u[:, :, 4:8] & 0xF0)).reshape(1, 1, 1, P, 64)
        r4 = ((u[:, :, 0:4] & 0xF) | ((u[:, :, 4:8] & 0xF) << 4)).reshape(1, 1, 1, P, 64)
        want = oracle_mod.decode(a4.astype(np.uint8), r4.astype(np.uint8), meta, P, P, C, ALPHA)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), k
        if k == 4:
            plain = oracle_mod.decode(anc, None, meta, P, P, C, ALPHA)
            assert np.array_equal(got.view(np.uint32), plain.view(np.uint32))


# ----------------------------------------------------------- INT-B baseline

def test_int_baseline_grid_rows_round_trip(oracle_mod):
    """Eq. 4 on rows whose range is exactly 2^B - 1: S = 1, Z = -x_min, so
    every integer value is its own code and decodes exactly; nibble j of a
    B = 4 row is channel 2j (low) then 2j + 1 (high)."""
    d = np.arange(128)
    # every value has at most 8 significant bits, so it is exact in BF16
    rows = {4: (d % 16).astype(np.float32) - 3.0,
            8: np.where(d == 127, 255, 2 * d).astype(np.float32) - 100.0}
    for B, x in rows.items():
        xb = oracle_mod.f32_to_bf16_bits(x).reshape(1, 128)
        codes, meta = oracle_mod.int_encode(xb, B)
        assert meta[0, 0] == x.min() and meta[0, 1] == 1.0
        q = codes[0] if B == 8 else np.stack([codes[0] & 0xF, codes[0] >> 4], 1).reshape(-1)
        assert np.array_equal(q.astype(np.float32), x - x.min())
        assert np.array_equal(oracle_mod.int_decode(codes, meta, B)[0], x)
    x = np.zeros(128, np.float32)
    x[0], x[1] = 15.0, 0.0
    x[2:] = 7.0
    codes, _ = oracle_mod.int_encode(oracle_mod.f32_to_bf16_bits(x).reshape(1, 128), 4)
    assert codes[0, 0] == 0x0F


def test_int_baseline_error_bound_and_extremes(oracle_mod):
    """|x^ - x| <= S/2 (+ float32 rounding); the row minimum codes to 0 and
    the maximum to 2^B - 1; a constant row (S = 0) codes to 0 and decodes
    exactly; a zero minimum is stored as +0."""
    rng = np.random.default_rng(3)
    x = (rng.laplace(size=(64, 128)) * np.exp(rng.standard_normal((64, 1)))).astype(np.float32)
    xb = oracle_mod.f32_to_bf16_bits(x)
    xf = oracle_mod.bf16_bits_to_f32(xb)
    for B in (4, 8):
        codes, meta = oracle_mod.int_encode(xb, B)
        y = oracle_mod.int_decode(codes, meta, B)
        S = meta[:, 1:2].astype(np.float64)
        err = np.abs(y.astype(np.float64) - xf)
        assert (err <= S / 2 * (1 + 1e-5) + np.abs(xf) * 2.0 ** -22).all()
        q = codes if B == 8 else np.stack([codes & 0xF, codes >> 4], -1).reshape(64, 128)
        assert (q[np.arange(64), xf.argmin(1)] == 0).all()
        assert (q[np.arange(64), xf.argmax(1)] == (1 << B) - 1).all()
    c = oracle_mod.f32_to_bf16_bits(np.full((2, 128), -2.5, np.float32))
    z = oracle_mod.f32_to_bf16_bits(np.where(np.arange(128) % 2 == 0, -0.0, 0.0)
                                    .astype(np.float32).reshape(1, 128))
    for B in (4, 8):
        codes, meta = oracle_mod.int_encode(c, B)
        assert (codes == 0).all() and meta[0, 1] == 0.0
        assert (oracle_mod.int_decode(codes, meta, B) == -2.5).all()
        _, mz = oracle_mod.int_encode(z, B)
        assert mz[0, 0].view(np.uint32) == 0 and mz[0, 1].view(np.uint32) == 0


def test_int_baseline_outlier_starves_ordinary_channels(oracle_mod):
    """Eq. 5: with one channel about 100x the others, the ordinary channels
    of a row share about 2^B m_i / m bins (2.56 for INT8 at m = 100 m_i)."""
    rng = np.random.default_rng(9)
    x = rng.uniform(-1, 1, size=(256, 128)).astype(np.float32)
    x[:, 5] = 100.0
    xb = oracle_mod.f32_to_bf16_bits(x)
    for B in (8, 4):
        codes, meta = oracle_mod.int_encode(xb, B)
        q = codes if B == 8 else np.stack([codes & 0xF, codes >> 4], -1).reshape(256, 128)
        ordinary = np.delete(q, 5, axis=1)
        used = np.array([len(np.unique(r)) for r in ordinary])
        span = (1 << B) * 2.0 / 101.0       # the ordinary range 2 of a row range ~101
        assert used.max() <= math.ceil(span) + 1
        assert used.min() >= 1
    assert abs(oracle_mod.effective_bins(8, 1 / 100) - 2.56) < 1e-12


# ----------------------------------------------------------- vNMSE

def test_vnmse_closed_forms(oracle_mod):
    rng = np.random.default_rng(4)
    r = rng.standard_normal((3, 5, 128))
    assert oracle_mod.vnmse(r, r) == 0.0
    assert abs(oracle_mod.vnmse(2 * r, r) - 1.0) < 1e-12
    assert abs(oracle_mod.vnmse(np.zeros_like(r), r) - 1.0) < 1e-12
    assert abs(oracle_mod.vnmse(r + 0.1 * r, r) - 0.01) < 1e-12


def test_attention_rows_gqa_mapping(oracle_mod):
    """Query head h reads KV head h // (H_q / H_kv): with each KV head's
    values constant (c_h), every output of query head j is c_{j // G}."""
    rng = np.random.default_rng(6)
    B, L, Hkv, G, T = 2, 16, 3, 2, 2
    K = rng.standard_normal((B, L, Hkv, 128)).astype(np.float32)
    c = np.arange(1, B * Hkv + 1, dtype=np.float32).reshape(B, 1, Hkv, 1)
    V = np.broadcast_to(c, (B, L, Hkv, 128)).astype(np.float32)
    q = rng.standard_normal((B, T, Hkv * G, 128)).astype(np.float32)
    o = oracle_mod.attention_rows(q, K, V)
    for b in range(B):
        for j in range(Hkv * G):
            assert np.allclose(o[b, :, j], c[b, 0, j // G, 0], rtol=0, atol=1e-12)


# ----------------------------------------------------------- Appendix A.1

def _a1_block(seed=5, P=128):
    """[1][P][1][128] bf16: Laplace channels, one all-negative channel, one
    zero channel, one channel of a repeated value."""
    rng = np.random.default_rng(seed)
    x = rng.laplace(size=(P, 128)).astype(np.float32) * np.exp(rng.standard_normal(128)).astype(np.float32)
    x[:, 3] = -np.abs(x[:, 3]) - 0.5
    x[:, 4] = 0.0
    x[:, 5] = 2.5
    import oracle
    return oracle.f32_to_bf16_bits(x).reshape(1, P, 1, 128)


def _a1_codes(anc, res):
    """Signed Q from the packed nibbles: Q = Q_anc * 16 + Q_res (Q_anc signed)."""
    a = _signed_codes(anc.reshape(anc.shape[-2], -1), res.reshape(res.shape[-2], -1))
    return a      # the nibble pairing of Stage 4 read back as one signed byte


def test_a1_chunk_maxima_and_signs(oracle_mod):
    """Appendix A.1: x'' = x / (m m_i) is +-1 at the largest |x| of each
    16-token chunk of a channel, so |Q| = 127 there with the sign of x; a zero
    channel codes to 0 and stores m = 0; Q = Q_anc * 16 + Q_res lies in
    [-127, 127] with Q_anc = Q >> 4 (arithmetic)."""
    P = 128
    x = _a1_block(P=P)
    anc, res, meta = oracle_mod.a1_encode(x, P)
    Q = _a1_codes(anc, res)
    xf = oracle_mod.bf16_bits_to_f32(x)[0, :, 0, :]
    assert Q.min() >= -127 and Q.max() <= 127
    for c in range(P // 16):
        blk = xf[16 * c:16 * (c + 1)]
        t = np.abs(blk).argmax(0)
        for d in range(128):
            v = blk[t[d], d]
            if v != 0:
                assert Q[16 * c + t[d], d] == (127 if v > 0 else -127), (c, d)
    assert (Q[:, 4] == 0).all() and meta[0, 0, 0, 0, 4] == 0
    assert (Q[:, 5] == 127).all()                 # a constant positive channel
    assert (Q[:, 3] <= 0).all()                   # the all-negative channel
    np.testing.assert_array_equal(meta[0, 0, 0, 0], np.abs(xf).max(0))


def test_a1_scale_invariance_and_small_alpha(oracle_mod):
    """Scaling a channel by a power of two leaves its codes unchanged (every
    step is a ratio); as alpha -> 0 the alpha-law is the identity and
    |Q| = round(127 |x''|), the textbook linear quantizer."""
    P = 64
    x = _a1_block(seed=8, P=P)
    xf = oracle_mod.bf16_bits_to_f32(x)
    anc, res, meta = oracle_mod.a1_encode(x, P)
    anc2, res2, meta2 = oracle_mod.a1_encode(oracle_mod.f32_to_bf16_bits(xf * 4.0), P)
    assert np.array_equal(anc, anc2) and np.array_equal(res, res2)
    np.testing.assert_array_equal(meta2[..., 0, :], 4 * meta[..., 0, :])
    a_s, r_s, m_s = oracle_mod.a1_encode(x, P, alpha=1e-7)
    Q = _a1_codes(a_s, r_s)
    xs = xf[0, :, 0, :].astype(np.float64)
    for c in range(P // 16):
        blk = xs[16 * c:16 * (c + 1)]
        mx = np.abs(blk).max(0)
        xpp = np.divide(blk, mx, out=np.zeros_like(blk), where=mx > 0)
        want = np.sign(xpp) * np.rint(127 * np.abs(xpp))
        frac = (127 * np.abs(xpp)) % 1.0
        keep = np.abs(frac - 0.5) > 1e-3
        assert np.array_equal(Q[16 * c:16 * (c + 1)][keep], want[keep].astype(int))


def test_a1_decode_error_bound_and_anchor_point(oracle_mod):
    """Full decode is within half a code step of x: |x - x^| <= m m_i
    max(X(|Q| + 1/2) - X(|Q|), X(|Q|) - X(|Q| - 1/2)) with X of Eq. 14/15 (the
    steps are geometric, so the two half-steps differ); the Anchor-only
    decode equals the full decode of Q = 16 Q_anc + 7."""
    P = 128
    alpha = 100.0
    x = _a1_block(seed=3, P=P)
    xf = oracle_mod.bf16_bits_to_f32(x).astype(np.float64)[0, :, 0, :]
    anc, res, meta = oracle_mod.a1_encode(x, P, alpha)
    y = oracle_mod.a1_decode(anc, res, meta, P, P, alpha)[0, :, 0, :].astype(np.float64)
    Q = _a1_codes(anc, res)
    I = np.abs(Q).astype(np.float64)

    def X(v):
        return ((1 + alpha) ** (np.clip(v, 0, 127) / 127.0) - 1) / alpha

    m = meta[0, 0, 0, 0].astype(np.float64)
    mi = np.repeat(meta[0, 0, 0, 1:].astype(np.float64), 16, axis=0)
    half = np.maximum(X(I + 0.5) - X(I), X(I) - X(I - 0.5))
    assert (np.abs(y - xf) <= m * mi * half * 1.001 + np.abs(xf) * 2.0 ** -20).all()
    r7 = np.full_like(res, 0x77)
    full7 = oracle_mod.a1_decode(anc, r7, meta, P, P, alpha)
    anchor_only = oracle_mod.a1_decode(anc, None, meta, P, P, alpha)
    assert np.array_equal(full7.view(np.uint32), anchor_only.view(np.uint32))


# ------------------------------------------ BF16 rounding of the reconstruction

# (float32 bit pattern, bf16 bit pattern) worked out by hand for IEEE round to
# nearest, ties to even.  A bf16 keeps the top 16 bits of the float32; the
# dropped 16 bits decide the rounding: below 0x8000 down, above it up, at
# exactly 0x8000 (a tie) towards the even kept pattern.
BF16_HAND = [
    (0x3F800000, 0x3F80),   # 1.0, exact
    (0x3F808000, 0x3F80),   # 1 + 2^-8: tie between 1 and 1 + 2^-7, 0x3F80 is even
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: tie between 0x3F81 (odd) and 0x3F82 (even)
    (0x3F808001, 0x3F81),   # one float ulp above a tie: up
    (0x3F807FFF, 0x3F80),   # one float ulp below a tie: down
    (0x3F817FFF, 0x3F81),   # below the tie that would round an odd pattern up
    (0x3FFF8000, 0x4000),   # tie from odd 0x3FFF: the carry steps the exponent, 2.0
    (0xBF818000, 0xBF82),   # negatives round by magnitude
    (0xBF808000, 0xBF80),
    (0x00000000, 0x0000),   # +0
    (0x80000000, 0x8000),   # -0 keeps its sign
    (0x00018000, 0x0002),   # subnormal tie from odd: up
    (0x00008000, 0x0000),   # subnormal tie from even (zero): down
    (0x7F7F7FFF, 0x7F7F),   # just below the tie above the largest finite bf16
    (0x7F7F8000, 0x7F80),   # that tie (0x7F7F odd) rounds up to +infinity
    (0xFF7FFFFF, 0xFF80),   # -FLT_MAX rounds to -infinity
    (0x7F800000, 0x7F80),   # infinities are exact
    (0xFF800000, 0xFF80),
]


def test_bf16_rounding_hand_values(oracle_mod):
    """The rounding that defines the decoders' BF16 output and every attention
    operand (the float32 reconstruction rounded to nearest even) on ties,
    near-ties, a carry into the exponent, signed zeros, subnormals and the
    overflow to infinity."""
    src = np.array([s for s, _ in BF16_HAND], np.uint32).view(np.float32)
    got = oracle_mod.f32_to_bf16_bits(src)
    assert got.tolist() == [d for _, d in BF16_HAND]


def test_bf16_rounding_keeps_nan(oracle_mod):
    """A NaN stays a NaN (all-ones exponent, non-zero mantissa) with its sign,
    for quiet and signalling payloads; none turns into an infinity or a zero."""
    src = np.array([0x7FC00000, 0x7F800001, 0x7FFFFFFF, 0xFFFFFFFF, 0xFF800001],
                   np.uint32).view(np.float32)
    got = oracle_mod.f32_to_bf16_bits(src).astype(np.uint32)
    assert ((got & 0x7F80) == 0x7F80).all() and ((got & 0x007F) != 0).all(), got
    assert (got >> 15).tolist() == [0, 0, 0, 1, 1]


def test_bf16_rounding_matches_the_ieee_bound(oracle_mod):
    """On random finite float32 values, each result is one of the two bf16
    neighbours and lies within half a bf16 ulp (a float64 check of the
    round-to-nearest bound)."""
    rng = np.random.default_rng(11)
    u = rng.integers(0, 0x7F7F0000, size=20000, dtype=np.uint32)
    u |= (rng.integers(0, 2, size=u.size, dtype=np.uint32) << 31)
    x = u.view(np.float32)
    h = oracle_mod.f32_to_bf16_bits(x)
    y = oracle_mod.bf16_bits_to_f32(h).astype(np.float64)
    down = (u & 0xFFFF0000).view(np.float32).astype(np.float64)
    up = ((u & 0xFFFF0000) + 0x10000).view(np.float32).astype(np.float64)
    xd = x.astype(np.float64)
    assert ((y == down) | (y == up)).all()
    assert (np.abs(y - xd) <= np.abs(up - down) / 2).all()


# ------------------------------------------------------------- the epsilons

def _eps_block():
    """P = 64, C = 32, D = 8, built so that both epsilons of Stages 1-2 (1e-6,
    the reading where the pages leave it open) move codes and metadata.
    Channel 0: token 0 = 2^20, tokens 1..31 = 0; chunk 1 alternates 0 (even
      t) and 1 (odd t).  gamma_scale = 2^20, and 2^20 + 1e-6 rounds to 2^20
      in float32, so n = x 2^-20: chunk 1 holds {0, 2^-20}, mu = 2^-21 and
      d = -+2^-21 exactly, sigma = 2^-21.  Then |X_final| = 2^-21 /
      (2^-21 + 1e-6) = 0.32288 and Y = 127 ln(1 + 255 * 0.32288) / ln 256 =
      101.296: I = 101 (sigma + eps = 1e-3 would give I = 3, eps = 2e-6
      I = 90, eps = 1e-7 I = 123).  Chunk 0: mu = 1/32, sigma = 31/32, the
      spike has |X_final| = 0.999999 (I = 127) and the zeros 1/31
      (Y = 50.89, I = 51).
    Channel 1: alternating 0 and 2^-20 over the whole page.  gamma_scale =
      2^-20 is comparable to eps: n = 2^-20 / (2^-20 + 1e-6) = 0.488144 on the
      non-zeros, so mu = 0.244072 in both chunks (eps = 0 would store 0.5).
      Both signs then sit at +-sigma: I = 127 everywhere.
    Channels 2..7 are zero."""
    P = 64
    x = np.zeros((P, 8), np.float32)
    x[0, 0] = 2.0 ** 20
    x[33:64:2, 0] = 1.0
    x[1::2, 1] = 2.0 ** -20
    return _bf16_bits(x.ravel()).reshape(P, 8), x


def test_epsilons_hand_block(oracle_mod):
    bits, _ = _eps_block()
    anc, res, meta = oracle_mod.encode_block(bits, C=32, alpha=ALPHA)
    Q = _signed_codes(anc, res).astype(int)
    # channel 0: signed codes Q8 = I (S = +1) or -I - 1 (S = -1)
    assert Q[0, 0] == 127 and (Q[1:32, 0] == -52).all()
    assert (Q[32:64:2, 0] == -102).all() and (Q[33:64:2, 0] == 101).all()
    # channel 1: every value at +-sigma of its chunk
    assert (Q[0::2, 1] == -128).all() and (Q[1::2, 1] == 127).all()
    assert (Q[:, 2:] == 0).all()
    # metadata rows: gamma_min, gamma_scale, mu[2], sigma[2]
    assert meta[1, 0] == 2.0 ** 20 and meta[1, 1] == 2.0 ** -20
    assert meta[2, 0] == 1 / 32 and meta[3, 0] == 2.0 ** -21
    assert meta[5, 0] == 2.0 ** -21
    mu1 = 0.5 * 2.0 ** -20 / (2.0 ** -20 + 1e-6)
    assert abs(meta[2, 1] - mu1) < 1e-6 * mu1 and abs(meta[3, 1] - mu1) < 1e-6 * mu1


def test_epsilons_round_trip(oracle_mod):
    """Encode and decode agree on both epsilons: the full decode of the hand
    block lies within half a code step of every value, the step taken from
    the closed form X(I) = ((1 + alpha)^(I/127) - 1) / alpha scaled by
    (sigma + 1e-6)(gamma_scale + 1e-6) from the hand derivation (at I = 101
    in channel 0's chunk 1 that is 0.0071 * 1.4768e-6 * 2^20 = 0.011).  A
    decoder with another epsilon lands orders of magnitude away (sigma + 1e-3
    instead of 2^-21 + 1e-6 scales the spread by 680)."""
    bits, x = _eps_block()
    anc, res, meta = oracle_mod.encode_block(bits, C=32, alpha=ALPHA)
    y = oracle_mod.decode_block(anc, res, meta, C=32, alpha=ALPHA).astype(np.float64)
    I = np.abs(_signed_codes(anc, res).astype(np.float64) + 0.5) - 0.5

    def X(v):
        return ((1 + ALPHA) ** (np.clip(v, 0, 127) / 127.0) - 1) / ALPHA

    half = np.maximum(X(I + 0.5) - X(I), X(I) - X(I - 0.5))
    # (sigma + eps)(gamma_scale + eps) per token, from the hand derivation
    scale = np.zeros((64, 8))
    scale[:32, 0] = (31 / 32 + 1e-6) * 2.0 ** 20
    scale[32:, 0] = (2.0 ** -21 + 1e-6) * 2.0 ** 20
    mu1 = 0.5 * 2.0 ** -20 / (2.0 ** -20 + 1e-6)
    scale[:, 1] = (mu1 + 1e-6) * (2.0 ** -20 + 1e-6)
    err = np.abs(y - x.astype(np.float64))
    assert (err <= half * scale * 1.001 + 1e-12).all(), err.max(0)
    assert abs(y[33, 0] - 1.0) < 0.011 and abs(y[1, 1] - 2.0 ** -20) < 1e-2 * 2.0 ** -20
    assert (y[:, 2:] == 0).all()


# ------------------------------------------------ Appendix A.1 zero maxima

def test_a1_zero_and_tiny_maxima(oracle_mod):
    """Appendix A.1 with maxima of 0 and maxima far below 1e-6 (P = 64, chunks
    of 16; reading: a zero maximum gives a zero reciprocal, any other maximum
    its exact reciprocal, nothing added).
    Channel 0: token 0 = 2^20 (the page maximum m), chunk 1 alternates +1 and
      -1, chunks 2-3 are zero.  rm = 2^-20 exactly, so chunk 1 has
      x' = +-2^-20 and m_1 = 2^-20, x'' = +-1: Q = +-127 (Anchor 7 / -8,
      Residual 15 / 1).  Chunks 2-3: m_i = 0 and Q = 0.
    Channel 1: token 0 = 2^-24 (the page maximum), the rest 0: rm = 2^24,
      x' = 1 at token 0, so m_0 = 1 exactly.
    Decode: chunk 1 is X(127) * 2^-20 * 2^20 = +-1 exactly, the zero chunks
    +0."""
    P = 64
    x = np.zeros((P, 128), np.float32)
    x[0, 0] = 2.0 ** 20
    x[16:32, 0] = np.where(np.arange(16) % 2 == 0, 1.0, -1.0)
    x[0, 1] = 2.0 ** -24
    bits = _bf16_bits(x.ravel()).reshape(1, P, 1, 128)
    anc, res, meta = oracle_mod.a1_encode(bits, P)
    Q = _a1_codes(anc, res).astype(int)
    m = meta[0, 0, 0]
    assert m[0, 0] == 2.0 ** 20 and m[1, 0] == 1.0 and m[2, 0] == 2.0 ** -20
    assert m[3, 0] == 0.0 and m[4, 0] == 0.0 and not np.signbit(m[3:, 0]).any()
    assert m[0, 1] == 2.0 ** -24 and m[1, 1] == 1.0
    assert Q[0, 0] == 127 and (Q[1:16, 0] == 0).all()
    assert Q[16:32, 0].tolist() == [127, -127] * 8
    assert (Q[32:, 0] == 0).all() and Q[0, 1] == 127 and (Q[1:, 1] == 0).all()
    y = oracle_mod.a1_decode(anc, res, meta, P, P)[0, :, 0, :]
    assert y[16:32, 0].tolist() == [1.0, -1.0] * 8
    assert (y[32:, 0] == 0).all() and not np.signbit(y[32:, 0]).any()
    assert y[0, 1] == 2.0 ** -24


# ------------------------------------------- Eq. 10-11 weights below 2^-32

def test_spec_tiny_weights_keep_their_share(oracle_mod):
    """The inverse CDF keeps weights down to 2^-40 (reading: integer weights
    floor(w 2^40)).  Both drafts accepted, next distribution
    (2^-36, 2^-36, 2^-35): integer weights 16, 16, 32, Z = 64, target
    floor(r 64 / 2^32).  r = 0, 2^30, 2^31, 3 2^30 give targets 0, 16, 32, 48:
    tokens 0, 1, 2, 2.  (At 2^32 every weight would floor to 0: no token.)
    A weight below 2^-40 floors to 0 and is never drawn."""
    same = [0.5, 0.25, 0.25]
    tiny = [2.0 ** -36, 2.0 ** -36, 2.0 ** -35]
    got = [_one(oracle_mod, [same, tiny], [same], [0], [0.0], r)
           for r in (0, 1 << 30, 1 << 31, 3 << 30)]
    assert got == [(1, 0), (1, 1), (1, 2), (1, 2)]
    below = [2.0 ** -41, 2.0 ** -36, 0.0]
    assert _one(oracle_mod, [same, below], [same], [0], [0.0], 0) == (1, 1)
