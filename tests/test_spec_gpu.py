"""Speculative verification and correction (Eq. 10-11) through the C ABI,
bit-exact against the oracle: the accepted prefix length and the next token
of every sequence."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(batch, T, V, temp, seed, same=False):
    """Target and draft distributions that agree more or less (temp scales the
    draft's perturbation), drafts drawn from q, seeded uniforms."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((batch, T + 1, V)).astype(np.float32) * 3.0
    p = np.exp(logits - logits.max(axis=-1, keepdims=True))
    p = (p / p.sum(axis=-1, keepdims=True)).astype(np.float32)
    if same:
        q = p[:, :T].copy()
    else:
        ql = logits[:, :T] + temp * rng.standard_normal((batch, T, V)).astype(np.float32)
        q = np.exp(ql - ql.max(axis=-1, keepdims=True))
        q = (q / q.sum(axis=-1, keepdims=True)).astype(np.float32)
    s = np.empty((batch, T), np.int32)
    for b in range(batch):
        for t in range(T):
            qq = q[b, t].astype(np.float64)
            s[b, t] = rng.choice(V, p=qq / qq.sum())
    u = rng.random((batch, T), dtype=np.float32)
    r = rng.integers(0, 2 ** 32, size=batch, dtype=np.uint64).astype(np.uint32)
    return p, q, s, u, r


def _check(lynx_lib, oracle_mod, dev, p, q, s, u, r):
    kt, tt = lynx_lib.lynx_spec_verify(
        torch.from_numpy(p).to(dev), torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev),
        torch.from_numpy(u).to(dev), torch.from_numpy(r.view(np.int32)).to(dev))
    torch.cuda.synchronize()
    ko, to = oracle_mod.spec_verify(p, q, s, u, r)
    assert np.array_equal(kt.cpu().numpy(), ko), (kt.cpu().numpy(), ko)
    assert np.array_equal(tt.cpu().numpy(), to), (tt.cpu().numpy(), to)
    return ko


@pytest.mark.parametrize("batch,T,V,temp", [(16, 8, 1000, 0.3), (8, 8, 128003, 0.05),
                                            (4, 64, 5000, 0.02), (32, 1, 77, 1.0)])
def test_spec_verify_matches_oracle(lynx_lib, oracle_mod, cuda_dev, batch, T, V, temp):
    ko = _check(lynx_lib, oracle_mod, cuda_dev, *_inputs(batch, T, V, temp, seed=V + T))
    print("accepted", ko)


def test_spec_verify_full_acceptance_draws_the_bonus_token(lynx_lib, oracle_mod, cuda_dev):
    """q = p on every position: the whole draft is kept and the next token is
    drawn from p_{T+1}."""
    p, q, s, u, r = _inputs(8, 5, 3000, 0.0, seed=1, same=True)
    ko = _check(lynx_lib, oracle_mod, cuda_dev, p, q, s, u, r)
    assert np.all(ko == 5)
    assert lynx_lib.lynx_device_errors() & 4 == 0


@pytest.mark.parametrize("batch,T,V", [(20, 3, 131072), (2, 2, 131073), (3, 4, 200003)])
def test_spec_verify_segment_length_boundaries(lynx_lib, oracle_mod, cuda_dev, batch, T, V):
    """Segments of exactly 1024 tokens (V = 131072: every lane's tokens read in
    one batch of loads), of 1025 and of 1563 (read as a stream)."""
    _check(lynx_lib, oracle_mod, cuda_dev, *_inputs(batch, T, V, 0.05, seed=V % 97))


def test_spec_verify_zero_residual_draws_from_p(lynx_lib, oracle_mod, cuda_dev):
    """q = p and u = 1 at position 3: that draft token is rejected (u q < p
    fails), yet max(0, p - q) is 0 everywhere, so the next token is drawn from
    p at position 3."""
    p, q, s, u, r = _inputs(6, 4, 3001, 0.0, seed=2, same=True)
    u[:, 2] = 1.0
    ko = _check(lynx_lib, oracle_mod, cuda_dev, p, q, s, u, r)
    assert np.all(ko == 2)


def test_spec_verify_unnormalised_and_tiny_weights(lynx_lib, oracle_mod, cuda_dev):
    """Weights that are not distributions: p and q up to 100 (a warp meeting a
    weight of 8 or more sums with the integer-only form of floor(w 2^40); the
    totals stay far below 2^64), and rows sprinkled with subnormal and zero
    entries.  Tokens as the oracle's."""
    rng = np.random.default_rng(17)
    batch, T, V = 6, 4, 70001
    p = (rng.random((batch, T + 1, V)) ** 4 * 100.0).astype(np.float32)
    q = (rng.random((batch, T, V)) ** 4 * 100.0).astype(np.float32)
    tiny = rng.random((batch, T + 1, V)) < 0.2
    p[tiny] = np.float32(1e-40)
    p[:, :, ::97] = 0.0
    p[2] *= np.float32(1e-6)                       # one sequence entirely below 8
    s = rng.integers(0, V, size=(batch, T)).astype(np.int32)
    u = rng.random((batch, T), dtype=np.float32)
    r = rng.integers(0, 2 ** 32, size=batch, dtype=np.uint64).astype(np.uint32)
    _check(lynx_lib, oracle_mod, cuda_dev, p, q, s, u, r)
