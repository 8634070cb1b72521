"""Paged streams (pools of physical pages behind a block table) through the C
ABI, against the oracle: the pages' prototype keeps KV in pages aligned with
paged attention and scatters decoded pages into device memory.  The pools
are gathered back into the dense (b, page, h) order on the host and compared
with the oracle's encode (bit-exact), decode (bit-exact) and attention
(2e-3, normalised as in test_attn_gpu.py)."""
import numpy as np
import pytest
import torch

from .test_attn_gpu import TOL, _decode_seq_head
from .test_codec_gpu import THREADS, assert_same, bits_of

pytestmark = pytest.mark.gpu

ALPHA = 255.0


def _table(B, NB, spare, seed, dev):
    """A block table naming distinct physical pages in scattered order, with
    `spare` unused pages in the pool."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(B * NB + spare, generator=g)[: B * NB]
    return perm.view(B, NB).to(torch.int32).to(dev), B * NB + spare


def _gather(pool, table):
    """Pool [num_blocks][H][...] -> dense [B][NB][H][...] in table order."""
    t = table.long().cpu()
    return pool.cpu()[t.view(-1)].view(t.shape[0], t.shape[1], *pool.shape[1:])


@pytest.mark.parametrize("B,L,H,P,C", [(2, 1024, 2, 128, 32), (3, 512, 1, 256, 64),
                                       (1, 640, 3, 64, 16)])
def test_paged_encode_decode_match_oracle(lynx_lib, oracle_mod, cuda_dev, B, L, H, P, C):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(B, L, H, 128, seed=L + P + C, device=cuda_dev)
    NB = L // P
    table, nblocks = _table(B, NB, spare=5, seed=B + NB, dev=cuda_dev)
    pa, pr, pm = lynx_lib.lynx_encode_paged(kv, P, C, ALPHA, table, nblocks)
    torch.cuda.synchronize()
    oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, ALPHA, threads=THREADS)
    assert_same(_gather(pa, table), oa, "anchor")
    assert_same(_gather(pr, table), orr, "residual")
    assert_same(_gather(pm, table), om, "meta")
    for mode, name in ((lynx_lib.LYNX_FULL, "full"), (lynx_lib.LYNX_ANCHOR, "anchor")):
        ref = oracle_mod.decode(oa, orr if name == "full" else None, om, L, P, C, ALPHA,
                                threads=THREADS)
        f32 = lynx_lib.lynx_decode_paged(pa, pr if name == "full" else None, pm, table, L, P, C,
                                         ALPHA, mode, torch.float32)
        b16 = lynx_lib.lynx_decode_paged(pa, pr if name == "full" else None, pm, table, L, P, C,
                                         ALPHA, mode, torch.bfloat16)
        torch.cuda.synchronize()
        assert_same(f32, ref, f"paged decode {name} fp32")
        assert np.array_equal(bits_of(b16), oracle_mod.f32_to_bf16_bits(ref)), name
    assert lynx_lib.lynx_device_errors() == 0


@pytest.mark.parametrize("mode_name,T,H_q,tail,P,C", [
    ("anchor", 1, 8, False, 128, 32), ("full", 8, 8, True, 128, 32), ("full", 2, 4, False, 128, 32),
    # 16 rows per KV head over pages of 64 and chunks of 16 (two chunks per
    # 32-token producer range on the tensor-memory path)
    ("full", 4, 8, False, 64, 16),
    # pages of 512 (four per sequence) behind the table, draft and verification
    ("anchor", 1, 8, False, 512, 64), ("full", 8, 8, False, 512, 32)])
def test_paged_attention_matches_oracle(lynx_lib, oracle_mod, cuda_dev, mode_name, T, H_q,
                                        tail, P, C):
    from split_stream_kv_gb300 import synth
    batch, L, H_kv = 2, 2048, 2
    NB = L // P
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=T + H_q, device=cuda_dev)
    k, v = kv[0::2].contiguous(), kv[1::2].contiguous()
    table, nblocks = _table(batch, NB, spare=3, seed=T, dev=cuda_dev)
    kp = lynx_lib.lynx_encode_paged(k, P, C, ALPHA, table, nblocks)
    vp = lynx_lib.lynx_encode_paged(v, P, C, ALPHA, table, nblocks)
    full = mode_name == "full"
    mode = lynx_lib.LYNX_FULL if full else lynx_lib.LYNX_ANCHOR
    q = synth.queries(batch, T, H_q, 128, seed=T, device=cuda_dev)
    kt = vt = None
    if tail:
        tl = synth.kv_cache(2 * batch, T, H_kv, 128, seed=T + 50, device=cuda_dev)
        kt, vt = tl[0::2].contiguous(), tl[1::2].contiguous()
    out = lynx_lib.lynx_attn_decode_paged(q, kp if full else (kp[0], None, kp[2]),
                                          vp if full else (vp[0], None, vp[2]), table, L, P, C,
                                          ALPHA, mode, k_tail=kt, v_tail=vt)
    torch.cuda.synchronize()
    ks = tuple(_gather(t, table).numpy() for t in kp)
    vs = tuple(_gather(t, table).numpy() for t in vp)
    qf, o = q.float().cpu().numpy(), out.cpu().numpy()
    G = H_q // H_kv
    for b in range(batch):
        for h in range(H_kv):
            K = _decode_seq_head(oracle_mod, ks, b, h, L, P, C, full)
            V = _decode_seq_head(oracle_mod, vs, b, h, L, P, C, full)
            norm = np.maximum(1.0, np.abs(V).max(axis=0))
            if tail:
                vtf = vt.float().cpu().numpy()[b, :, h]
                norm = np.maximum(norm, np.abs(vtf).max(axis=0))
            for t in range(T):
                for gq in range(G):
                    hq = h * G + gq
                    if tail:
                        ref = oracle_mod.attention_row_tail(qf[b, t, hq], K, V,
                                                            kt.float().cpu().numpy()[b, :, h],
                                                            vtf, t + 1)
                    else:
                        ref = oracle_mod.attention_row(qf[b, t, hq], K, V)
                    rel = (np.abs(o[b, t, hq].astype(np.float64) - ref) / norm).max()
                    assert rel <= TOL, (b, t, hq, rel)
    assert lynx_lib.lynx_device_errors() == 0


def test_out_of_range_table_entry_is_reported(lynx_lib, cuda_dev):
    """An entry outside [0, num_blocks) is caught by the kernels' own range
    check: it is replaced by page 0 and reported (bit 2), with no stray access."""
    from split_stream_kv_gb300 import synth
    B, L, H, P, C = 1, 512, 1, 128, 32
    kv = synth.kv_cache(B, L, H, 128, seed=3, device=cuda_dev)
    table = torch.tensor([[0, 1, 2, 7]], dtype=torch.int32, device=cuda_dev)  # 7 >= num_blocks
    pa, pr, pm = lynx_lib.lynx_encode_paged(kv, P, C, ALPHA, table, 4)
    torch.cuda.synchronize()
    assert lynx_lib.lynx_device_errors() & 2
    assert lynx_lib.lynx_wait_timeouts() == 0
