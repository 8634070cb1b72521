"""Cases run by tests/test_checked_gpu.py on both builds of the library (the
library a process uses is chosen by LYNX_LIBRARY before the binding loads):
every codec page size, paged streams, the k-bit Anchor decode and the four
attention passes.  Returns {name: numpy array}; inputs are seeded, so both
processes see the same tensors."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

ALPHA = 255.0
CODEC = [(2, 1024, 3, 512, 32), (2, 1024, 2, 256, 64), (3, 1024, 3, 128, 32),
         (2, 512, 2, 64, 16), (1, 1024, 2, 512, 16)]


def run_cases():
    import torch

    from split_stream_kv_gb300 import lynx, synth
    dev = torch.device("cuda:0")
    out = {}

    def keep(name, t):
        out[name] = t.contiguous().view(torch.uint8).cpu().numpy()

    for B, L, H, P, C in CODEC:
        tag = f"{B}x{L}x{H}_p{P}c{C}"
        kv = synth.kv_cache(B, L, H, 128, seed=B + L + P + C, device=dev)
        anc, res, meta = lynx.lynx_encode(kv, P, C, ALPHA)
        keep("enc_" + tag, torch.cat([anc.view(-1), res.view(-1), meta.view(torch.uint8).view(-1)]))
        keep("full_" + tag, lynx.lynx_decode_full(anc, res, meta, L, P, C, ALPHA))
        keep("anc_" + tag, lynx.lynx_decode_anchor(anc, meta, L, P, C, ALPHA))
        if P == 512 and C == 32:
            for k in (3, 6):
                ak, _ = lynx.lynx_split_bits(anc, res, k)
                keep(f"bits{k}_" + tag, lynx.lynx_decode_anchor_bits(ak, meta, L, P, C, ALPHA, k))
    # paged codec: pools behind a scattered table
    B, L, H, P, C = 2, 1024, 2, 128, 32
    kv = synth.kv_cache(B, L, H, 128, seed=77, device=dev)
    NB = L // P
    g = torch.Generator().manual_seed(3)
    table = torch.randperm(B * NB + 5, generator=g)[: B * NB].view(B, NB).to(torch.int32).to(dev)
    pools = lynx.lynx_encode_paged(kv, P, C, ALPHA, table, B * NB + 5)
    keep("paged_full", lynx.lynx_decode_paged(*pools, table, L, P, C, ALPHA, lynx.LYNX_FULL))
    # attention: draft, verify, verify with draft tokens, paged verify, 64 tokens
    batch, L, Hkv, Hq, P, C = 2, 2048, 2, 8, 128, 32
    kvv = synth.kv_cache(2 * batch, L, Hkv, 128, seed=21, device=dev)
    ks = lynx.lynx_encode(kvv[0::2].contiguous(), P, C, ALPHA)
    vs = lynx.lynx_encode(kvv[1::2].contiguous(), P, C, ALPHA)
    for T, mode in ((1, lynx.LYNX_ANCHOR), (8, lynx.LYNX_FULL), (64, lynx.LYNX_FULL)):
        q = synth.queries(batch, T, Hq, 128, seed=T, device=dev)
        k_use = ks if mode == lynx.LYNX_FULL else (ks[0], None, ks[2])
        v_use = vs if mode == lynx.LYNX_FULL else (vs[0], None, vs[2])
        keep(f"attn_T{T}", lynx.lynx_attn_decode(q, k_use, v_use, L, P, C, ALPHA, mode))
    q8 = synth.queries(batch, 8, Hq, 128, seed=8, device=dev)
    tail = synth.kv_cache(2 * batch, 8, Hkv, 128, seed=5, device=dev)
    keep("attn_tail", lynx.lynx_attn_decode(q8, ks, vs, L, P, C, ALPHA, lynx.LYNX_FULL,
                                            k_tail=tail[0::2].contiguous(),
                                            v_tail=tail[1::2].contiguous()))
    NB = L // P
    table = torch.randperm(batch * NB + 7, generator=g)[: batch * NB].view(batch, NB)
    table = table.to(torch.int32).to(dev)
    idx = table.view(-1).long()

    def pool(t):
        p = torch.zeros((batch * NB + 7,) + tuple(t.shape[2:]), dtype=t.dtype, device=dev)
        p[idx] = t.reshape((-1,) + tuple(t.shape[2:]))
        return p
    keep("attn_paged", lynx.lynx_attn_decode_paged(q8, tuple(pool(t) for t in ks),
                                                   tuple(pool(t) for t in vs), table, L, P, C,
                                                   ALPHA, lynx.LYNX_FULL))
    # the same verification, dense and paged, over pages of 64 and chunks of 16
    P, C = 64, 16
    ks = lynx.lynx_encode(kvv[0::2].contiguous(), P, C, ALPHA)
    vs = lynx.lynx_encode(kvv[1::2].contiguous(), P, C, ALPHA)
    keep("attn_T8_c16", lynx.lynx_attn_decode(q8, ks, vs, L, P, C, ALPHA, lynx.LYNX_FULL))
    NB = L // P
    table = torch.randperm(batch * NB + 7, generator=g)[: batch * NB].view(batch, NB)
    table = table.to(torch.int32).to(dev)
    idx = table.view(-1).long()
    keep("attn_paged_c16", lynx.lynx_attn_decode_paged(q8, tuple(pool(t) for t in ks),
                                                       tuple(pool(t) for t in vs), table, L, P,
                                                       C, ALPHA, lynx.LYNX_FULL))
    # pages of 512: draft and verification
    P, C = 512, 64
    ks = lynx.lynx_encode(kvv[0::2].contiguous(), P, C, ALPHA)
    vs = lynx.lynx_encode(kvv[1::2].contiguous(), P, C, ALPHA)
    q1 = synth.queries(batch, 1, Hq, 128, seed=1, device=dev)
    keep("attn_T1_p512", lynx.lynx_attn_decode(q1, (ks[0], None, ks[2]), (vs[0], None, vs[2]),
                                               L, P, C, ALPHA, lynx.LYNX_ANCHOR))
    keep("attn_T8_p512", lynx.lynx_attn_decode(q8, ks, vs, L, P, C, ALPHA, lynx.LYNX_FULL))
    torch.cuda.synchronize()
    out["device_errors"] = __import__("numpy").array([lynx.lynx_device_errors()])
    out["library"] = __import__("numpy").frombuffer(
        os.path.basename(lynx.LIB_PATH).encode(), dtype="uint8")
    return out


if __name__ == "__main__":
    import numpy as np
    np.savez(sys.argv[1], **run_cases())
