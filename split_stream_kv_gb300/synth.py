"""Seeded synthetic inputs: KV caches with the statistics the pages describe,
and decode queries.

This module draws random numbers only; it holds none of the codec's or the
attention's arithmetic, so the CUDA path and the CPU oracle can both be fed
from it.  (The oracle always receives the very tensor the GPU received, copied
back to the host, so no generator parity between devices is needed.)

KV statistics (from "Lynx: Progressive Speculative KV Cache Transfer for
Disaggregated LLM Inference", Prerequisites section 4 and Mechanism 1
Stage 1): centred KV values are Laplacian-like, and a few channels hold values
about 100x larger than the rest, at the same channel indices in every layer.
Recipe, per tensor kv[B][L][H][D] with B = 2 * layers (b = 2*layer + 0 for K,
+1 for V):

    x[b, t, h, d] = bf16_rn( s[b, h, d] * o[b % 2, h, d] * Laplace(0, 1) )
    s[b, h, d]    = exp(0.5 * N(0, 1))              per (layer, K/V, head, ch)
    o[k, h, d]    = outlier_scale on n_outlier (h, d) channels of tensor type
                    k (K or V, drawn independently), 1 elsewhere

Queries are N(0, 1) rounded to bf16.
"""
from __future__ import annotations

import torch


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def outlier_channels(H: int, D: int, n_outlier: int, seed: int):
    """Outlier (head, channel) indices for K and for V: two lists of flat
    indices h*D + d, the same for every layer."""
    g = _gen("cpu", seed * 1000003 + 17)
    k_idx = torch.randperm(H * D, generator=g)[:n_outlier]
    v_idx = torch.randperm(H * D, generator=g)[:n_outlier]
    return k_idx, v_idx


def default_outliers(H: int, D: int) -> int:
    """round(1% of H*D) outlier channels per tensor type (at least 1)."""
    return max(1, int(round(0.01 * H * D)))


@torch.no_grad()
def kv_cache(B: int, L: int, H: int, D: int, *, n_outlier: int | None = None,
             outlier_scale: float = 100.0, seed: int = 0, device="cpu",
             out: torch.Tensor | None = None) -> torch.Tensor:
    """BF16 KV tensor [B][L][H][D]; generated one b-slice at a time so that
    large caches need only a slice of float32 scratch."""
    if n_outlier is None:
        n_outlier = default_outliers(H, D)
    if out is None:
        out = torch.empty((B, L, H, D), dtype=torch.bfloat16, device=device)
    device = out.device
    gs = _gen("cpu", seed * 7919 + 3)
    scale = torch.exp(0.5 * torch.randn((B, H * D), generator=gs))
    k_idx, v_idx = outlier_channels(H, D, n_outlier, seed)
    o = torch.ones((2, H * D))
    o[0, k_idx] = outlier_scale
    o[1, v_idx] = outlier_scale
    for b in range(B):
        g = _gen(device, seed * 1000 + b + 1)
        u = torch.rand((L, H * D), generator=g, device=device, dtype=torch.float32)
        u = u.clamp_(min=2.0 ** -24, max=1.0 - 2.0 ** -24) - 0.5
        lap = -torch.sign(u) * torch.log1p(-2.0 * u.abs())
        col = (scale[b] * o[b % 2]).to(device)
        out[b].copy_((lap * col).view(L, H, D).to(torch.bfloat16))
    return out


@torch.no_grad()
def queries(batch: int, T: int, H_q: int, D: int, *, seed: int = 0,
            device="cpu") -> torch.Tensor:
    """BF16 decode queries [batch][T][H_q][D], N(0, 1)."""
    g = _gen(device, seed * 31 + 5)
    q = torch.randn((batch, T, H_q, D), generator=g, device=device)
    return q.to(torch.bfloat16)
