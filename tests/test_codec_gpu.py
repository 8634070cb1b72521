"""Parity of the CUDA codec (through the C ABI) with the CPU oracle.

Acceptance: packed codes and metadata bit-exact; decoded values bit-exact in
float32 (the oracle uses the same float32 reconstruction), and the BF16
output equal to the oracle's float32 rounded to nearest even.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0
THREADS = max(1, min(16, os.cpu_count() or 1))


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_same(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = gpu.cpu().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    if g.tobytes() != ref.tobytes():
        gv = g.reshape(-1).view(np.uint8) if g.dtype == np.uint8 else g.reshape(-1)
        rv = ref.reshape(-1).view(np.uint8) if ref.dtype == np.uint8 else ref.reshape(-1)
        bad = np.nonzero(gv != rv)[0]
        raise AssertionError(f"{what}: {bad.size} of {gv.size} differ; first at {bad[:8]}: "
                             f"gpu {gv[bad[:8]]} oracle {rv[bad[:8]]}")


@pytest.mark.parametrize("alpha", [255.0, 100.0, 2000.0, 1.0])
def test_compander_fast_path_exhaustive(lynx_lib, cuda_dev, alpha):
    """Every float32 in [0, 1]: the encoder's fast Stage-3 rounding either
    equals the threshold rule or is flagged and sent to the exact path."""
    n, bad, amb, maxerr = lynx_lib.lynx_compander_selfcheck(alpha, cuda_dev)
    assert n == 0x3F800001
    assert bad == 0
    assert amb < n * 1e-3                       # the exact path stays rare
    print(f"alpha={alpha}: flagged {amb / n:.2e}, max |Y'-Y| = {maxerr / 2**32:.3e}")


# (B, L, H, page, C): several blocks per CTA, ragged grid tails, every (page, C)
CASES = [
    (2, 256, 1, 256, 32),      # the tiny configuration: 1 layer, 1 head
    (3, 1024, 3, 128, 32),
    (2, 512, 2, 64, 16),
    (2, 1024, 2, 256, 64),
    (1, 512, 4, 128, 128),
    (2, 512, 1, 256, 16),
    (1, 256, 2, 64, 64),
    (2, 512, 2, 128, 64),
    (1, 768, 3, 256, 128),
    (5, 384, 1, 128, 16),
    (2, 320, 3, 64, 32),       # five pages of 64
    # 512-token pages (the largest page of the pages' ablation grid): two
    # TMA loads per tile, two decode units per page
    (2, 1024, 3, 512, 16),
    (1, 1536, 2, 512, 32),
    (2, 1024, 1, 512, 64),
    (1, 1024, 2, 512, 128),
]


@pytest.mark.parametrize("B,L,H,P,C", CASES)
def test_encode_decode_match_oracle(lynx_lib, oracle_mod, cuda_dev, B, L, H, P, C):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(B, L, H, 128, seed=B * 1000 + L + P + C, device=cuda_dev,
                        n_outlier=max(2, H * 128 // 100))
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
    torch.cuda.synchronize()
    x = bits_of(kv)
    oa, orr, om = oracle_mod.encode(x, P, C, ALPHA, threads=THREADS)
    assert_same(anc, oa, "anchor")
    assert_same(res, orr, "residual")
    assert_same(meta, om, "meta")
    for mode in ("full", "anchor"):
        r_or = orr if mode == "full" else None
        ref = oracle_mod.decode(oa, r_or, om, L, P, C, ALPHA, threads=THREADS)
        if mode == "full":
            f32 = lynx_lib.lynx_decode_full(anc, res, meta, L, P, C, ALPHA, torch.float32)
            b16 = lynx_lib.lynx_decode_full(anc, res, meta, L, P, C, ALPHA, torch.bfloat16)
        else:
            f32 = lynx_lib.lynx_decode_anchor(anc, meta, L, P, C, ALPHA, torch.float32)
            b16 = lynx_lib.lynx_decode_anchor(anc, meta, L, P, C, ALPHA, torch.bfloat16)
        torch.cuda.synchronize()
        assert_same(f32, ref, f"decode {mode} fp32")
        assert np.array_equal(bits_of(b16), oracle_mod.f32_to_bf16_bits(ref)), f"{mode} bf16"
    assert lynx_lib.lynx_wait_timeouts() == 0


def _special_kv(device):
    """Degenerate pages: constant, zeros of both signs, one spike per chunk,
    subnormal-sized values, two-valued, huge range, one negative ramp."""
    P, H = 128, 2
    blocks = []
    g = torch.Generator().manual_seed(7)
    base = torch.randn((P, 128), generator=g)
    blocks.append(torch.full((P, 128), 3.25))
    z = torch.zeros((P, 128))
    z[::2] = -0.0
    blocks.append(z)
    spike = base.clone() * 0.01
    spike[5::32, :] = 1000.0
    blocks.append(spike)
    blocks.append(base * 1e-38)
    two = torch.where(base > 0, torch.tensor(1.5), torch.tensor(-2.0))
    blocks.append(two)
    blocks.append(base * torch.logspace(-20, 20, 128).unsqueeze(0))
    blocks.append(-torch.arange(P * 128, dtype=torch.float32).view(P, 128))
    blocks.append(base.round())
    kv = torch.stack(blocks).view(4, 2, P, 128).permute(0, 2, 1, 3).contiguous()
    return kv.to(torch.bfloat16).to(device)   # [B=4][L=128][H=2][128]


def test_special_pages_match_oracle(lynx_lib, oracle_mod, cuda_dev):
    kv = _special_kv(cuda_dev)
    B, L, H, _ = kv.shape
    for P, C in ((128, 32), (128, 16), (128, 128)):
        anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
        torch.cuda.synchronize()
        oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, ALPHA)
        assert_same(anc, oa, f"anchor P={P} C={C}")
        assert_same(res, orr, f"residual P={P} C={C}")
        assert_same(meta, om, f"meta P={P} C={C}")
        ref = oracle_mod.decode(oa, orr, om, L, P, C, ALPHA)
        f32 = lynx_lib.lynx_decode_full(anc, res, meta, L, P, C, ALPHA, torch.float32)
        torch.cuda.synchronize()
        assert_same(f32, ref, "decode full special")


def test_empty_tensor_is_a_no_op(lynx_lib, cuda_dev):
    kv = torch.empty((0, 256, 2, 128), dtype=torch.bfloat16, device=cuda_dev)
    anc, res, meta = lynx_lib.lynx_encode(kv, 128, 32, ALPHA)
    assert anc.numel() == 0
    out = lynx_lib.lynx_decode_full(anc, res, meta, 256, 128, 32, ALPHA)
    assert out.numel() == 0


# Full-size configurations, checked on seeded samples of page blocks.
FULL = [
    ("llama3_8b_16k", 64, 16384, 8, 128, 32, 96),
    ("qwen_32b_16k", 128, 16384, 8, 128, 32, 96),
    ("qwen3_235b_128k", 188, 131072, 4, 256, 64, 64),
]


@pytest.mark.parametrize("name,B,L,H,P,C,nsamp", FULL)
def test_full_size_sampled_blocks(lynx_lib, oracle_mod, cuda_dev, name, B, L, H, P, C, nsamp):
    from split_stream_kv_gb300 import synth
    free, _ = torch.cuda.mem_get_info(cuda_dev)
    need = B * L * H * 128 * (2 + 1 + 2) + (B * L * H * 128 * 4) // C
    if free < need * 1.1:
        pytest.skip(f"{name} needs {need / 2**30:.1f} GiB")
    kv = synth.kv_cache(B, L, H, 128, seed=11, device=cuda_dev)
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
    NB = L // P
    rng = np.random.default_rng(123)
    blks = np.unique(np.concatenate([[0, B * NB * H - 1], rng.integers(0, B * NB * H, nsamp)]))
    hh = torch.as_tensor(blks % H, device=cuda_dev)
    pp = torch.as_tensor((blks // H) % NB, device=cuda_dev)
    bb = torch.as_tensor(blks // (H * NB), device=cuda_dev)
    full = lynx_lib.lynx_decode_full(anc, res, meta, L, P, C, ALPHA, torch.bfloat16)
    part = lynx_lib.lynx_decode_anchor(anc, meta, L, P, C, ALPHA, torch.bfloat16)
    torch.cuda.synchronize()
    tok = pp[:, None] * P + torch.arange(P, device=cuda_dev)[None, :]
    tiles = kv[bb[:, None], tok, hh[:, None]]                 # [n][P][128]
    ga, gr, gm = anc[bb, pp, hh].cpu().numpy(), res[bb, pp, hh].cpu().numpy(), \
        meta[bb, pp, hh].cpu().numpy()
    gf = bits_of(full[bb[:, None], tok, hh[:, None]])
    gp = bits_of(part[bb[:, None], tok, hh[:, None]])
    tb = bits_of(tiles)
    for i in range(len(blks)):
        oa, orr, om = oracle_mod.encode_block(tb[i], C, ALPHA)
        assert ga[i].tobytes() == oa.tobytes(), f"{name} block {blks[i]} anchor"
        assert gr[i].tobytes() == orr.tobytes(), f"{name} block {blks[i]} residual"
        assert gm[i].tobytes() == om.tobytes(), f"{name} block {blks[i]} meta"
        rf = oracle_mod.decode_block(oa, orr, om, C, ALPHA)
        rp = oracle_mod.decode_block(oa, None, om, C, ALPHA)
        assert np.array_equal(gf[i], oracle_mod.f32_to_bf16_bits(rf)), f"{name} full {blks[i]}"
        assert np.array_equal(gp[i], oracle_mod.f32_to_bf16_bits(rp)), f"{name} anc {blks[i]}"
    assert lynx_lib.lynx_wait_timeouts() == 0
