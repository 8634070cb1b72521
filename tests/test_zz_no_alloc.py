"""The allocation-free attention entry point against the regular one.

lynx_attn_decode_noalloc serves callers that cannot allocate device memory
(stream capture, real-time paths, hosts that forbid driver allocations): its
split-K scratch is a fixed array inside the library.  It runs the same
kernels with the same split as lynx_attn_decode with a caller workspace, so
its output must equal that one bit for bit, call after call, although the
array is shared and keeps the previous call's contents.  This file sorts last
so that a run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0
TOL = 2e-3   # the attention tests' bound (normalised by max(1, max|V|))
P, C = 128, 32


def _streams(lynx_lib, cuda_dev, batch, L, H_kv, seed):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=seed, device=cuda_dev)
    ks = lynx_lib.lynx_encode(kv[0::2].contiguous(), P, C, ALPHA)
    vs = lynx_lib.lynx_encode(kv[1::2].contiguous(), P, C, ALPHA)
    return ks, vs


def _use(lynx_lib, mode, s):
    return s if mode == lynx_lib.LYNX_FULL else (s[0], None, s[2])


def test_noalloc_matches_workspace_variant_bitwise(lynx_lib, cuda_dev):
    """A larger call first (twice the chunks, so more split-K partials in the
    shared array, from other data), then the draft and the verify shape twice
    each: every output equals the workspace variant's bit for bit, so nothing
    left in the array by an earlier call is ever read."""
    from split_stream_kv_gb300 import synth
    bk, bv = _streams(lynx_lib, cuda_dev, 2, 4096, 2, seed=99)
    big_q = synth.queries(2, 8, 8, 128, seed=3, device=cuda_dev)
    need_big = lynx_lib.lynx_attn_workspace_bytes(2, 8, 8, 4096, 2, 128, P)
    lynx_lib.lynx_attn_decode_noalloc(big_q, bk, bv, 4096, P, C, ALPHA, lynx_lib.LYNX_FULL)

    batch, L, H_kv, H_q = 2, 2048, 2, 8
    ks, vs = _streams(lynx_lib, cuda_dev, batch, L, H_kv, seed=21)
    for mode, T in ((lynx_lib.LYNX_ANCHOR, 1), (lynx_lib.LYNX_FULL, 8)):
        assert lynx_lib.lynx_attn_workspace_bytes(batch, T, H_q, L, H_kv, 128, P) < need_big
        q = synth.queries(batch, T, H_q, 128, seed=T, device=cuda_dev)
        k_use, v_use = _use(lynx_lib, mode, ks), _use(lynx_lib, mode, vs)
        ref = lynx_lib.lynx_attn_decode(q, k_use, v_use, L, P, C, ALPHA, mode)
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            lynx_lib.lynx_attn_decode_noalloc(q, k_use, v_use, L, P, C, ALPHA, mode, out=out)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            assert torch.equal(out, ref), (out - ref).abs().max().item()


def test_noalloc_matches_the_oracle(lynx_lib, oracle_mod, cuda_dev):
    """One verification pass through the allocation-free entry point against
    float64 oracle attention over the oracle's decode of the same codes
    (rounded to BF16), every (sequence, head) of a small case."""
    from split_stream_kv_gb300 import synth
    batch, L, H_kv, H_q, T = 2, 1024, 2, 8, 8
    ks, vs = _streams(lynx_lib, cuda_dev, batch, L, H_kv, seed=5)
    q = synth.queries(batch, T, H_q, 128, seed=11, device=cuda_dev)
    out = torch.empty((batch, T, H_q, 128), dtype=torch.float32, device=cuda_dev)
    lynx_lib.lynx_attn_decode_noalloc(q, ks, vs, L, P, C, ALPHA, lynx_lib.LYNX_FULL, out=out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    qf = q.float().cpu().numpy()
    hat = []
    for s in (ks, vs):
        x = oracle_mod.decode(s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(), L, P,
                              C, ALPHA)
        hat.append(oracle_mod.bf16_bits_to_f32(oracle_mod.f32_to_bf16_bits(x)).reshape(x.shape))
    K, V = hat
    ref = oracle_mod.attention_rows(qf, K, V)
    G = H_q // H_kv
    norm = np.maximum(1.0, np.abs(V).max(axis=1))                 # [batch][H_kv][128]
    norm = np.repeat(norm, G, axis=1)[:, None]                     # [batch][1][H_q][128]
    err = (np.abs(o - ref) / norm).max()
    assert err <= TOL, err


def test_noalloc_rejects_sizes_beyond_its_scratch(lynx_lib, cuda_dev):
    """More split-K partials than the built-in array holds is an error, not a
    fault: 64 sequences x 32 KV heads x 4 row groups need > 8 MiB."""
    lib = lynx_lib.lib()
    need = lynx_lib.lynx_attn_workspace_bytes(64, 8, 128, 4096, 32, 128, 128)
    assert need > (8 << 20)
    import ctypes
    p = ctypes.c_void_p(0x10000)
    rc = lib.lynx_attn_decode_noalloc(p, 64, 8, 128, p, p, p, p, p, p, 4096, 32, 128, 128, 32,
                                      ALPHA, 1, p, None)
    assert rc == lynx_lib.LYNX_EWORKSPACE
    assert "scratch" in lynx_lib.lynx_last_error()
