"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/lynx.h declares, sizes follow the stated layout,
arguments are rejected before anything is enqueued, and the float64 tables
the kernels use agree with the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "lynx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lynx_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lynx_lib):
    lib = lynx_lib.lib()
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each one under the same name
    for n in names:
        assert hasattr(lynx_lib, n), n


def test_checked_build_exports_every_declared_symbol(lynx_lib):
    """liblynx_checked.so (the same sources with in-kernel index checks) is
    built beside the regular library and exports the same C ABI."""
    import ctypes

    from split_stream_kv_gb300 import _build
    lib = ctypes.CDLL(_build.LIB_CHECKED)
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_encoded_sizes(lynx_lib):
    # Llama-3-8B-shaped: 32 layers x K,V, L=16384, 8 heads, page 128, C 32
    a, r, m = lynx_lib.lynx_encoded_sizes(64, 16384, 8, 128, 128, 32)
    assert a == r == 512 * 2 ** 20
    assert m == 64 * 128 * 8 * (2 + 8) * 128 * 4 == 320 * 2 ** 20
    # meta is (2 + 2P/C) floats per channel per block (14% of BF16 at P=256, C=32)
    a, r, m = lynx_lib.lynx_encoded_sizes(1, 256, 1, 128, 256, 32)
    assert m == 2304 * 4


BAD = ctypes.c_void_p(0x1001)     # misaligned, never dereferenced
OK = ctypes.c_void_p(0x10000)     # aligned, never dereferenced: every call below fails first


@pytest.mark.parametrize("args,code", [
    (dict(D=64), -3),
    (dict(page=96), -3),
    (dict(page=1024), -3),
    (dict(C=48), -2),
    (dict(C=8), -3),
    (dict(C=512, page=256), -3),
    (dict(L=1000), -2),
    (dict(alpha=0.0), -1),
    (dict(alpha=float("nan")), -1),
    (dict(alpha=float("inf")), -1),
    (dict(alpha=0.5), -3),            # the encoder is built for alpha >= 1
    (dict(kv=None), -1),
    (dict(kv=BAD), -1),
    (dict(H=0), -2),
])
def test_encode_rejects(lynx_lib, args, code):
    lib = lynx_lib.lib()
    a = dict(kv=OK, B=2, L=1024, H=2, D=128, page=128, C=32, alpha=255.0)
    a.update(args)
    rc = lib.lynx_encode(a["kv"], a["B"], a["L"], a["H"], a["D"], a["page"], a["C"], a["alpha"],
                         OK, OK, OK, None)
    assert rc == code, lynx_lib.lynx_last_error()
    assert lynx_lib.lynx_last_error()


def test_decode_rejects(lynx_lib):
    lib = lynx_lib.lib()
    assert lib.lynx_decode_full(OK, None, OK, 1, 128, 1, 128, 128, 32, 255.0, OK, 0, None) == -1
    assert lib.lynx_decode_anchor(OK, OK, 1, 128, 1, 128, 128, 32, 255.0, OK, 7, None) == -1
    assert lib.lynx_decode_anchor(OK, BAD, 1, 128, 1, 128, 128, 32, 255.0, OK, 0, None) == -1


def test_attention_rejects(lynx_lib):
    lib = lynx_lib.lib()

    def call(batch=1, T=1, Hq=4, L=256, Hkv=1, D=128, page=128, C=32, mode=0, ws=1 << 30,
             kres=None):
        return lib.lynx_attn_decode(OK, batch, T, Hq, OK, kres, OK, OK, None, OK, L, Hkv, D,
                                    page, C, 255.0, mode, OK, OK, ws, None)

    assert call(Hq=6, Hkv=4) == -2            # H_q % H_kv
    assert call(T=0) == -2
    assert call(T=65, Hq=1) == -3             # more than 64 query tokens
    assert call(T=64, Hq=8, Hkv=1) == -3      # 512 rows > 256
    assert call(mode=1) == -1                 # full mode needs residuals
    assert call(mode=3) == -1
    assert call(ws=0) == -5
    assert call(L=100) == -2
    assert call(page=1024, L=2048) == -3      # pages up to 512, like the codec
    assert call(page=96, L=192) == -3         # pages are powers of two from 64
    assert lynx_lib.lynx_attn_workspace_bytes(1, 8, 4, 1024, 1, 128, 512) > 0
    need = lynx_lib.lynx_attn_workspace_bytes(1, 1, 4, 256, 1, 128, 128)
    assert need > 0
    assert call(ws=need - 1) == -5


def test_status_strings(lynx_lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lynx_lib.lynx_status_string(code)


@pytest.mark.parametrize("alpha", [255.0, 100.0, 2000.0, 1.0])
def test_thresholds_match_oracle_rounding(lynx_lib, oracle_mod, alpha):
    """thresholds[k] is the smallest float32 whose Eq. 7 code exceeds k: the
    oracle gives k+1 there and k at the next float below."""
    thr = np.array(lynx_lib.lynx_compander_thresholds(alpha), dtype=np.float32)
    assert (np.diff(thr) > 0).all()
    for k, t in enumerate(thr):
        assert oracle_mod.round_code(float(t), alpha) == k + 1
        below = np.nextafter(np.float32(t), np.float32(0))
        assert oracle_mod.round_code(float(below), alpha) == k


@pytest.mark.parametrize("alpha", [255.0, 100.0, 2000.0])
def test_expand_table_matches_oracle(lynx_lib, oracle_mod, alpha):
    lib_tab = np.array(lynx_lib.lynx_expand_table(alpha), dtype=np.float32)
    ora_tab = oracle_mod.expand_table(alpha)
    assert lib_tab.tobytes() == ora_tab.tobytes()


def test_binding_rejects_cpu_tensors(lynx_lib):
    import torch
    kv = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lynx_lib.lynx_encode(kv, 128, 32, 255.0)


def test_binding_rejects_mis_sized_buffers(lynx_lib):
    """The C ABI sees pointers only, so the binding checks every caller
    tensor against the sizes the call implies before anything is launched
    (these checks run before any device work, so meta tensors suffice)."""
    import torch

    from split_stream_kv_gb300 import lynx
    dev = torch.device("meta")

    def streams(B, L, H, P=128, C=32):
        a, r, m = lynx.stream_shapes(B, L, H, 128, P, C)
        return (torch.empty(a, dtype=torch.uint8, device=dev),
                torch.empty(r, dtype=torch.uint8, device=dev),
                torch.empty(m, dtype=torch.float32, device=dev))

    q = torch.empty((2, 1, 8, 128), dtype=torch.bfloat16, device=dev)
    ks, vs = streams(2, 256, 2), streams(2, 256, 2)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    good_out = torch.empty((2, 1, 8, 128), dtype=torch.float32, device=dev)
    check = lynx._check_attn_io
    check("t", q, ks, vs, 256, 128, 32, lynx.LYNX_FULL, good_out, ws, 1024)
    bad = [
        dict(out=torch.empty((2, 1, 8, 64), dtype=torch.float32, device=dev)),
        dict(out=torch.empty((2, 1, 8, 128), dtype=torch.bfloat16, device=dev)),
        dict(L=512),                                   # streams hold 256 tokens
        dict(vs=streams(2, 256, 4)),                   # V with other heads
        dict(ks=(ks[0], None, ks[2])),                 # full mode without residuals
        dict(ks=(ks[0], ks[1], torch.empty(1, device=dev))),
        dict(need=1 << 21),                            # workspace too small
    ]
    for b in bad:
        a = dict(q=q, ks=ks, vs=vs, L=256, out=good_out, need=1024)
        a.update(b)
        with pytest.raises(ValueError):
            check("t", a["q"], a["ks"], a["vs"], a["L"], 128, 32, lynx.LYNX_FULL, a["out"], ws,
                  a["need"])
    with pytest.raises(ValueError):
        lynx._expect(torch.empty((4,), device=dev), (4,), torch.float32,
                     torch.device("cuda", 0), "device")
