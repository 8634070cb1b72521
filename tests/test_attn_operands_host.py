"""The attention kernel's reconstruction of K and V against the decoders'.

The decoders rebuild x = fma(fma(v, sigma + eps, mu), gamma_scale + eps,
gamma_min) in float32 and round it to BF16.  Attention applies the same affine
map as one fused multiply-add, x1 = fma(v, A, B) with A = (sigma + eps)
(gamma_scale + eps) and B = fma(mu, gamma_scale + eps, gamma_min), built once
per chunk and channel.  This checks, on the CPU with float32 arithmetic and the
oracle's codes and metadata, over three (page, C) shapes and both modes:
- the emulated two-step form is the oracle's decode bit for bit;
- |x1 - x| <= 2^-22 (gamma_scale + eps): the two forms round differently, by a
  few float32 ulps of the channel's page range;
- the BF16 operands differ on fewer than 1e-3 of the values, and by at most one
  BF16 ulp (2^-7 of the value) plus 2^-21 (gamma_scale + eps): values that
  nearly cancel to zero inside their channel's range may differ by several
  ulps of a tiny value, still a few float32 ulps of the range;
- attention over the two operand sets differs by < 1e-5 after the R14
  normalisation, against the 2e-3 tolerance."""
import numpy as np

ALPHA = 255.0


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _fma(a, b, c):
    """float32 fused multiply-add: the float64 product of two float32 values
    is exact, so one rounding of a*b + c to float32 (via float64) is the fma
    except in double-rounding ties, which do not occur at this scale."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _block(seed, P=128):
    from split_stream_kv_gb300 import synth
    import torch
    kv = synth.kv_cache(2, P * 16, 1, 128, seed=seed, device="cpu")
    return kv.view(torch.int16).numpy().view(np.uint16)


import pytest


@pytest.mark.parametrize("seed,P,C", [(3, 128, 32), (5, 256, 64), (7, 64, 16)])
def test_one_fma_operands_against_the_decoders(oracle_mod, seed, P, C):
    bits = _block(seed, P)
    anc, res, meta = oracle_mod.encode(bits, P, C, ALPHA)
    L = bits.shape[1]
    eps = np.float32(1e-6)
    tab = oracle_mod.expand_table(ALPHA)
    a4 = anc.reshape(2, L // P, P, 64)
    r4 = res.reshape(2, L // P, P, 64)
    ch = np.arange(128)
    byte = (ch >> 3) * 4 + (ch & 3)
    sh = np.where(ch & 4, 4, 0)
    an = (a4[..., byte] >> sh) & 0xF                                      # [2][NB][P][128]
    m = meta.reshape(2, L // P, 2 + 2 * (P // C), 128)
    chunk = np.arange(P) // C
    gm = m[:, :, None, 0, :]
    gs = _f32(m[:, :, None, 1, :] + eps)
    mu = m[:, :, 2 + chunk, :]
    sg = _f32(m[:, :, 2 + P // C + chunk, :] + eps)
    A = _f32(sg * gs)
    B = _fma(mu, gs, gm)
    gs_b = np.broadcast_to(gs, an.shape).astype(np.float64)
    q = np.random.default_rng(seed).standard_normal((4, 128)).astype(np.float32)
    for residual in (None, res):
        exact = oracle_mod.decode(anc, residual, meta, L, P, C, ALPHA)   # [2][L][1][128]
        # the decoders' table value v of every code
        if residual is None:
            qa = np.where(an >= 8, an.astype(np.int32) - 16, an)
            S = np.where(qa >= 0, 1, -1)
            I = 16 * np.where(qa >= 0, qa, -qa - 1) + 7
        else:
            q8 = (an.astype(np.int32) << 4) | ((r4[..., byte] >> sh) & 0xF)
            q8 = np.where(q8 >= 128, q8 - 256, q8)
            S = np.where(q8 >= 0, 1, -1)
            I = np.where(q8 >= 0, q8, -q8 - 1)
        v = _f32(S * tab[I])
        two = _fma(_fma(v, sg, mu), gs, gm)
        assert np.array_equal(two.reshape(exact.shape), exact)        # the decoders' path
        one = _fma(v, A, B)
        assert (np.abs(one.astype(np.float64) - two) <= 2.0 ** -22 * gs_b).all()
        e16 = oracle_mod.f32_to_bf16_bits(two)
        o16 = oracle_mod.f32_to_bf16_bits(one)
        assert float((e16 != o16).mean()) < 1e-3
        be = oracle_mod.bf16_bits_to_f32(e16).reshape(two.shape).astype(np.float64)
        bo = oracle_mod.bf16_bits_to_f32(o16).reshape(two.shape).astype(np.float64)
        bound = 2.0 ** -7 * np.maximum(np.abs(be), np.abs(bo)) + 2.0 ** -21 * gs_b
        assert (np.abs(be - bo) <= bound).all()
        # attention over the two operand sets (K = layer row 0, V = row 1)
        K, V = be.reshape(exact.shape)[0, :, 0], be.reshape(exact.shape)[1, :, 0]
        K1, V1 = bo.reshape(exact.shape)[0, :, 0], bo.reshape(exact.shape)[1, :, 0]
        norm = np.maximum(1.0, np.abs(V).max(axis=0))
        for r in range(4):
            d = np.abs(oracle_mod.attention_row(q[r], _f32(K1), _f32(V1))
                       - oracle_mod.attention_row(q[r], _f32(K), _f32(V)))
            assert (d / norm).max() < 1e-5
