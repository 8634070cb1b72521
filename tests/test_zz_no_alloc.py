"""The allocation-free attention entry point against the regular one.

lynx_attn_decode_noalloc serves callers that cannot allocate device memory
(stream capture, real-time paths, hosts that forbid driver allocations): its
split-K scratch is a fixed array inside the library.  It must give the same
output as lynx_attn_decode with a caller workspace, call after call, since the
array is shared and keeps the previous call's contents.  This file sorts last
so that a run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0
TOL = 2e-3   # the attention tests' bound (normalised by max(1, max|V|))


def test_noalloc_matches_workspace_variant_twice(lynx_lib, cuda_dev):
    from split_stream_kv_gb300 import synth
    batch, L, H_kv, H_q, P, C = 2, 2048, 2, 8, 128, 32
    kv = synth.kv_cache(2 * batch, L, H_kv, 128, seed=21, device=cuda_dev)
    ks = lynx_lib.lynx_encode(kv[0::2].contiguous(), P, C, ALPHA)
    vs = lynx_lib.lynx_encode(kv[1::2].contiguous(), P, C, ALPHA)
    vmax = kv[1::2].float().abs().amax(dim=1).clamp_min(1.0)        # [batch][H_kv][128]
    for mode, T in ((lynx_lib.LYNX_ANCHOR, 1), (lynx_lib.LYNX_FULL, 8)):
        q = synth.queries(batch, T, H_q, 128, seed=T, device=cuda_dev)
        k_use = ks if mode == lynx_lib.LYNX_FULL else (ks[0], None, ks[2])
        v_use = vs if mode == lynx_lib.LYNX_FULL else (vs[0], None, vs[2])
        ref = lynx_lib.lynx_attn_decode(q, k_use, v_use, L, P, C, ALPHA, mode)
        outs = []
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            lynx_lib.lynx_attn_decode_noalloc(q, k_use, v_use, L, P, C, ALPHA, mode, out=out)
            outs.append(out)
        torch.cuda.synchronize()
        norm = vmax.repeat_interleave(H_q // H_kv, dim=1)[:, None]   # [batch][1][H_q][128]
        for out in outs:
            assert torch.isfinite(out).all()
            err = ((out - ref).abs() / norm).max().item()
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
