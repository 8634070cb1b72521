"""Parity of the packed-KV decode attention (through the C ABI) with the
oracle: float64 softmax(q K^T / sqrt(128)) V over the oracle's own decode of
the same packed streams, rounded to BF16 (the values the kernel sees).

Tolerance: outputs can be as large as the outlier channels of V (|v| up to
~1e3), so the 2e-3 max-abs bound is applied to the error divided by
max(1, max_t |V_t,d|) per (sequence, head, channel), and to the raw error of
the channels whose values stay below 16.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0
TOL = 2e-3


def _decode_seq_head(oracle_mod, streams, b, h, L, P, C, full):
    """Oracle decode of all pages of (sequence b, head h) -> float32 [L][128]
    holding BF16-rounded values."""
    anc, res, meta = streams
    NB = L // P
    out = np.empty((L, 128), np.float32)
    for p in range(NB):
        x = oracle_mod.decode_block(anc[b, p, h], res[b, p, h] if full else None,
                                    meta[b, p, h], C, ALPHA)
        out[p * P:(p + 1) * P] = oracle_mod.bf16_bits_to_f32(
            oracle_mod.f32_to_bf16_bits(x)).reshape(P, 128)
    return out


def _check(oracle_mod, q, k_np, v_np, out, L, P, C, full, pairs, H_q, H_kv, T):
    G = H_q // H_kv
    qf = q.float().cpu().numpy()
    o = out.cpu().numpy()
    worst = 0.0
    for b, h in pairs:
        K = _decode_seq_head(oracle_mod, k_np, b, h, L, P, C, full)
        V = _decode_seq_head(oracle_mod, v_np, b, h, L, P, C, full)
        norm = np.maximum(1.0, np.abs(V).max(axis=0))
        small = np.abs(V).max(axis=0) < 16
        for t in range(T):
            for gq in range(G):
                hq = h * G + gq
                ref = oracle_mod.attention_row(qf[b, t, hq], K, V)
                err = np.abs(o[b, t, hq].astype(np.float64) - ref)
                rel = (err / norm).max()
                worst = max(worst, rel)
                assert rel <= TOL, (b, t, hq, rel)
                if small.any():
                    assert err[small].max() <= TOL, (b, t, hq, err[small].max())
    return worst


def _run(lynx_lib, oracle_mod, dev, batch, L, H_kv, H_q, T, P, C, pairs, seed=0, T_anchor=1):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=seed, device=dev)
    k = kv[0::2].contiguous()
    v = kv[1::2].contiguous()
    ks = lynx_lib.lynx_encode(k, P, C, ALPHA)
    vs = lynx_lib.lynx_encode(v, P, C, ALPHA)
    k_np = tuple(t.cpu().numpy() for t in ks)
    v_np = tuple(t.cpu().numpy() for t in vs)
    results = {}
    for mode, TT in ((lynx_lib.LYNX_ANCHOR, T_anchor), (lynx_lib.LYNX_FULL, T)):
        q = synth.queries(batch, TT, H_q, 128, seed=seed + TT, device=dev)
        full = mode == lynx_lib.LYNX_FULL
        ksm = ks if full else (ks[0], None, ks[2])
        vsm = vs if full else (vs[0], None, vs[2])
        out = lynx_lib.lynx_attn_decode(q, ksm, vsm, L, P, C, ALPHA, mode)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        results[mode] = _check(oracle_mod, q, k_np, v_np, out, L, P, C, full, pairs, H_q, H_kv, TT)
    return results


def test_tiny_single_head(lynx_lib, oracle_mod, cuda_dev):
    """1 layer, 1 KV head, 1 query head, L=256, page 256, C 32."""
    r = _run(lynx_lib, oracle_mod, cuda_dev, 1, 256, 1, 1, 8, 256, 32, [(0, 0)])
    print(r)


def test_gqa_groups_and_row_groups(lynx_lib, oracle_mod, cuda_dev):
    """4 query heads per KV head; T=8 gives 32 query rows (4 row groups)."""
    pairs = [(0, 0), (0, 1), (1, 0), (1, 1)]
    r = _run(lynx_lib, oracle_mod, cuda_dev, 2, 1024, 2, 8, 8, 128, 32, pairs, seed=3)
    print(r)


@pytest.mark.parametrize("P,C,L", [(64, 16, 1024), (256, 64, 2048), (128, 128, 512),
                                   (128, 16, 640)])
def test_page_and_chunk_sizes(lynx_lib, oracle_mod, cuda_dev, P, C, L):
    _run(lynx_lib, oracle_mod, cuda_dev, 1, L, 2, 4, 2, P, C, [(0, 0), (0, 1)], seed=P + C)


@pytest.mark.parametrize("P,C,L,H_kv,H_q,T,Ta", [
    (64, 16, 1024, 2, 8, 3, 2),      # 12 rows: padded warp-pair pass, two chunks per 32 tokens
    (256, 64, 2048, 1, 8, 4, 1),     # 32 rows
    (128, 16, 1024, 1, 3, 3, 3),     # 9 rows both modes
    (128, 32, 768, 1, 16, 2, 1),     # 16 query heads per KV head: anchor mode with 16 rows
    (128, 32, 1024, 2, 8, 16, 2),    # 64 rows: two row groups of 32
    (128, 128, 1024, 2, 8, 8, 1),    # 32 rows, chunks of 128 (one per verification tile)
    (64, 32, 1088, 1, 4, 8, 1),      # L not a multiple of 128: the register-direct pair shape
    (128, 32, 128, 4, 16, 8, 1),     # one 128-token tile per (KV head, row group): one CTA each
    (512, 64, 2048, 2, 8, 8, 1),     # pages of 512 (the codec's largest): tensor-memory pass
    (512, 16, 1536, 1, 4, 8, 2),     # pages of 512, chunks of 16 (32 chunks a page)
])
def test_row_counts_and_pairs(lynx_lib, oracle_mod, cuda_dev, P, C, L, H_kv, H_q, T, Ta):
    pairs = [(0, h) for h in range(H_kv)]
    _run(lynx_lib, oracle_mod, cuda_dev, 1, L, H_kv, H_q, T, P, C, pairs, seed=L + T, T_anchor=Ta)


def test_rising_maxima_rescale_every_tile(lynx_lib, oracle_mod, cuda_dev):
    """Keys whose channel 0 grows by 1 per token and queries that weight it:
    each 128-token tile raises every row's running maximum by about
    16 (log2 units), more than the 2^8 a weight may reach before the maximum is
    raised, so the verification pass rescales its accumulators on every tile
    (and its split partials carry maxima far apart)."""
    from split_stream_kv_gb300 import synth
    batch, L, H_kv, H_q, T, P, C = 1, 1024, 1, 4, 8, 128, 32
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=31, device=cuda_dev)
    ramp = torch.arange(L, device=cuda_dev, dtype=torch.float32)
    kv[0::2, :, :, 0] = (kv[0::2, :, :, 0].float() + ramp[None, :, None]).to(kv.dtype)
    k = kv[0::2].contiguous()
    v = kv[1::2].contiguous()
    ks = lynx_lib.lynx_encode(k, P, C, ALPHA)
    vs = lynx_lib.lynx_encode(v, P, C, ALPHA)
    q = synth.queries(batch, T, H_q, 128, seed=32, device=cuda_dev)
    q[..., 0] = 1.0
    out = lynx_lib.lynx_attn_decode(q, ks, vs, L, P, C, ALPHA, lynx_lib.LYNX_FULL)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert lynx_lib.lynx_device_errors() == 0
    k_np = tuple(t.cpu().numpy() for t in ks)
    v_np = tuple(t.cpu().numpy() for t in vs)
    _check(oracle_mod, q, k_np, v_np, out, L, P, C, True, [(0, 0)], H_q, H_kv, T)


def test_decode_attention_full_size_sampled(lynx_lib, oracle_mod, cuda_dev):
    """8 sequences x 32768 tokens, 32 query heads over 8 KV heads: draft step
    (T=1, Anchor) and verification (T=8, Anchor+Residual); three sampled
    (sequence, KV head) pairs checked on every query row."""
    pairs = [(0, 0), (3, 5), (7, 7)]
    r = _run(lynx_lib, oracle_mod, cuda_dev, 8, 32768, 8, 32, 8, 128, 32, pairs, seed=5)
    print(r)


def test_shares_straddling_units_all_heads(lynx_lib, oracle_mod, cuda_dev):
    """4 sequences x 4 KV heads x 10240 tokens: 5120 chunks of 32 tokens over
    304 CTAs, so most CTA shares (16-17 chunks) start or end inside a head and
    one work unit of such a CTA carries its state across; every (sequence, KV
    head) is checked, draft (T=1 Anchor) and verification (T=8 full)."""
    pairs = [(b, h) for b in range(4) for h in range(4)]
    r = _run(lynx_lib, oracle_mod, cuda_dev, 4, 10240, 4, 16, 8, 128, 32, pairs, seed=11)
    print(r)


def test_more_units_than_sms(lynx_lib, oracle_mod, cuda_dev):
    """4 sequences x 8 KV heads x 8 row groups of 32 (T = 64, 4 query heads per
    KV head) = 256 work units of two 128-token tiles: more units than a GB300
    has SMs, so the verification pass runs one unit per CTA over more than one
    wave and the combine maps every unit to its own CTA.  Four (sequence, KV
    head) pairs checked on all 256 rows."""
    pairs = [(0, 0), (1, 7), (2, 3), (3, 5)]
    r = _run(lynx_lib, oracle_mod, cuda_dev, 4, 256, 8, 32, 64, 128, 32, pairs, seed=13)
    print(r)


def _run_tail(lynx_lib, oracle_mod, dev, batch, L, H_kv, H_q, T, P, C, pairs, mode, seed):
    """Attention with the draft tokens' own keys and values (causal tail)."""
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=seed, device=dev)
    k = kv[0::2].contiguous()
    v = kv[1::2].contiguous()
    tail = synth.kv_cache(2 * batch, T, H_kv, 128, seed=seed + 1, device=dev)
    kt = tail[0::2].contiguous()
    vt = tail[1::2].contiguous()
    ks = lynx_lib.lynx_encode(k, P, C, ALPHA)
    vs = lynx_lib.lynx_encode(v, P, C, ALPHA)
    full = mode == lynx_lib.LYNX_FULL
    q = synth.queries(batch, T, H_q, 128, seed=seed + 2, device=dev)
    out = lynx_lib.lynx_attn_decode_tail(q, ks if full else (ks[0], None, ks[2]),
                                         vs if full else (vs[0], None, vs[2]),
                                         L, P, C, ALPHA, mode, kt, vt)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    k_np = tuple(t.cpu().numpy() for t in ks)
    v_np = tuple(t.cpu().numpy() for t in vs)
    qf, o = q.float().cpu().numpy(), out.cpu().numpy()
    ktf, vtf = kt.float().cpu().numpy(), vt.float().cpu().numpy()
    G = H_q // H_kv
    worst = 0.0
    for b, h in pairs:
        K = _decode_seq_head(oracle_mod, k_np, b, h, L, P, C, full)
        V = _decode_seq_head(oracle_mod, v_np, b, h, L, P, C, full)
        norm = np.maximum(1.0, np.maximum(np.abs(V).max(axis=0), np.abs(vtf[b, :, h]).max(axis=0)))
        for t in range(T):
            for gq in range(G):
                hq = h * G + gq
                ref = oracle_mod.attention_row_tail(qf[b, t, hq], K, V, ktf[b, :, h], vtf[b, :, h],
                                                    t + 1)
                rel = (np.abs(o[b, t, hq].astype(np.float64) - ref) / norm).max()
                worst = max(worst, rel)
                assert rel <= TOL, (b, t, hq, rel)
    return worst


@pytest.mark.parametrize("mode_name,batch,L,H_kv,H_q,T,P,C", [
    ("full", 2, 1024, 2, 8, 8, 128, 32),     # 32 rows: warp-pair shape, draft length 8
    ("anchor", 1, 2048, 2, 4, 2, 256, 64),   # 4 rows: single shape
    ("full", 1, 768, 1, 3, 3, 128, 16),      # 9 rows, C = 16
    ("anchor", 2, 512, 2, 2, 1, 64, 16),     # T = 1: the draft step sees its own token
    ("full", 1, 1024, 2, 8, 64, 128, 32),    # T = 64, the pages' cap: 256 rows, 8 row groups
    ("full", 1, 768, 1, 1, 40, 256, 32),     # 40 rows: a full and a partial row group
])
def test_attention_with_draft_tokens(lynx_lib, oracle_mod, cuda_dev, mode_name, batch, L, H_kv,
                                     H_q, T, P, C):
    mode = lynx_lib.LYNX_FULL if mode_name == "full" else lynx_lib.LYNX_ANCHOR
    pairs = [(b, h) for b in range(batch) for h in range(H_kv)]
    r = _run_tail(lynx_lib, oracle_mod, cuda_dev, batch, L, H_kv, H_q, T, P, C, pairs, mode,
                  seed=L + T)
    print(r)


def test_attention_with_draft_tokens_full_size_sampled(lynx_lib, oracle_mod, cuda_dev):
    """The verification step of the bench workload (8 x 32768 tokens, 32
    query heads over 8 KV heads, T = 8) with the draft tokens' own keys and
    values; two sampled (sequence, KV head) pairs."""
    r = _run_tail(lynx_lib, oracle_mod, cuda_dev, 8, 32768, 8, 32, 8, 128, 32, [(1, 2), (6, 7)],
                  lynx_lib.LYNX_FULL, seed=9)
    print(r)
