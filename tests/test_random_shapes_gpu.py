"""Parity with the oracle over seeded random shapes: the codec bit for bit
(pages 64 ... 512, every chunk size, alpha from 1 to 2000, odd batch and head
counts) and attention within the 2e-3 normalised bound (dense and paged
streams, both modes, query groups of 1 ... 16 heads, T up to 64, draft-token
tails).  Each case draws its shape from a generator seeded by its index, so a
failure names a reproducible shape."""
import random

import numpy as np
import pytest
import torch

from .test_attn_gpu import ALPHA, TOL, _decode_seq_head
from .test_codec_gpu import assert_same, bits_of
from .test_paged_gpu import _gather, _table

pytestmark = pytest.mark.gpu


def _codec_shape(i):
    rng = random.Random(9100 + i)
    P = rng.choice([64, 128, 256, 512])
    C = rng.choice([c for c in (16, 32, 64, 128) if c <= P])
    return dict(B=rng.randint(1, 4), H=rng.choice([1, 2, 3, 5, 8]), P=P, C=C,
                L=P * rng.randint(1, 3), alpha=rng.choice([1.0, 30.0, 255.0, 2000.0]))


def _attn_shape(i):
    rng = random.Random(9200 + i)
    P = rng.choice([64, 128, 256, 512])
    C = rng.choice([c for c in (16, 32, 64, 128) if c <= P])
    G = rng.choice([1, 2, 4, 8, 16])
    # the mix is fixed by the index (two thirds Anchor+Residual, a third
    # paged, every fourth full case with a draft-token tail); the shape is drawn
    full = i % 3 != 0
    return dict(P=P, C=C, G=G, batch=rng.randint(1, 3), Hkv=rng.choice([1, 2, 4]),
                T=rng.choice([t for t in (1, 2, 3, 5, 8, 13, 16, 33, 64) if t * G <= 256]),
                L=P * rng.randint(1, max(1, 1536 // P)), full=full,
                paged=i % 3 == 2, tail=full and i % 4 == 1,
                pairs_seed=rng.randrange(1 << 30))


@pytest.mark.parametrize("i", range(12))
def test_random_codec_shape(lynx_lib, oracle_mod, cuda_dev, i):
    from split_stream_kv_gb300 import synth
    s = _codec_shape(i)
    B, L, H, P, C, alpha = s["B"], s["L"], s["H"], s["P"], s["C"], s["alpha"]
    kv = synth.kv_cache(B, L, H, 128, seed=500 + i, device=cuda_dev,
                        n_outlier=max(1, H * 128 // 100))
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, alpha)
    torch.cuda.synchronize()
    oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, alpha)
    assert_same(anc, oa, f"anchor {s}")
    assert_same(res, orr, f"residual {s}")
    assert_same(meta, om, f"meta {s}")
    ref = oracle_mod.decode(oa, orr, om, L, P, C, alpha)
    assert_same(lynx_lib.lynx_decode_full(anc, res, meta, L, P, C, alpha, torch.float32), ref,
                f"full decode {s}")
    ref = oracle_mod.decode(oa, None, om, L, P, C, alpha)
    assert_same(lynx_lib.lynx_decode_anchor(anc, meta, L, P, C, alpha, torch.float32), ref,
                f"anchor decode {s}")


@pytest.mark.parametrize("i", range(16))
def test_random_attention_shape(lynx_lib, oracle_mod, cuda_dev, i):
    from split_stream_kv_gb300 import synth
    s = _attn_shape(i)
    batch, L, Hkv, G, T, P, C = s["batch"], s["L"], s["Hkv"], s["G"], s["T"], s["P"], s["C"]
    full, Hq = s["full"], s["G"] * s["Hkv"]
    kv = synth.kv_cache(2 * batch, L, Hkv, 128, seed=600 + i, device=cuda_dev)
    k, v = kv[0::2].contiguous(), kv[1::2].contiguous()
    q = synth.queries(batch, T, Hq, 128, seed=700 + i, device=cuda_dev)
    mode = lynx_lib.LYNX_FULL if full else lynx_lib.LYNX_ANCHOR
    kt = vt = None
    if s["tail"]:
        tl = synth.kv_cache(2 * batch, T, Hkv, 128, seed=800 + i, device=cuda_dev)
        kt, vt = tl[0::2].contiguous(), tl[1::2].contiguous()

    def use(st):
        return st if full else (st[0], None, st[2])
    if s["paged"]:
        table, nb = _table(batch, L // P, spare=3, seed=i, dev=cuda_dev)
        kp = lynx_lib.lynx_encode_paged(k, P, C, ALPHA, table, nb)
        vp = lynx_lib.lynx_encode_paged(v, P, C, ALPHA, table, nb)
        out = lynx_lib.lynx_attn_decode_paged(q, use(kp), use(vp), table, L, P, C, ALPHA, mode,
                                              k_tail=kt, v_tail=vt)
        ks = tuple(_gather(t, table).numpy() for t in kp)
        vs = tuple(_gather(t, table).numpy() for t in vp)
    else:
        kd = lynx_lib.lynx_encode(k, P, C, ALPHA)
        vd = lynx_lib.lynx_encode(v, P, C, ALPHA)
        out = lynx_lib.lynx_attn_decode(q, use(kd), use(vd), L, P, C, ALPHA, mode,
                                        k_tail=kt, v_tail=vt)
        ks = tuple(t.cpu().numpy() for t in kd)
        vs = tuple(t.cpu().numpy() for t in vd)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all(), s
    rng = random.Random(s["pairs_seed"])
    pairs = sorted({(rng.randrange(batch), rng.randrange(Hkv)) for _ in range(2)})
    qf, o = q.float().cpu().numpy(), out.cpu().numpy()
    for b, h in pairs:
        K = _decode_seq_head(oracle_mod, ks, b, h, L, P, C, full)
        V = _decode_seq_head(oracle_mod, vs, b, h, L, P, C, full)
        norm = np.maximum(1.0, np.abs(V).max(axis=0))
        if s["tail"]:
            ktf = kt.float().cpu().numpy()[b, :, h]
            vtf = vt.float().cpu().numpy()[b, :, h]
            norm = np.maximum(norm, np.abs(vtf).max(axis=0))
        for t in range(T):
            for g in range(G):
                hq = h * G + g
                ref = (oracle_mod.attention_row_tail(qf[b, t, hq], K, V, ktf, vtf, t + 1)
                       if s["tail"] else oracle_mod.attention_row(qf[b, t, hq], K, V))
                rel = (np.abs(o[b, t, hq].astype(np.float64) - ref) / norm).max()
                assert rel <= TOL, (s, b, t, hq, rel)
    assert lynx_lib.lynx_device_errors() & 1 == 0
