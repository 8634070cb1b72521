"""Comparison points on the GPU, through the C ABI, against the oracle:
the linear INT-B baseline of Eq. 4 and the other Anchor/Residual bit splits
("Lynx: Progressive Speculative KV Cache Transfer for Disaggregated LLM
Inference", technical review: Prerequisites Eq. 4; Concrete Improvement
Suggestions, items 4-5).  Codes, metadata and float32 decodes bit-exact;
BF16 decodes equal the oracle's float32 rounded to nearest even."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def same_bytes(gpu, ref, what):
    g = gpu.cpu().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    if g.tobytes() != ref.tobytes():
        gv, rv = g.reshape(-1).view(np.uint8), ref.reshape(-1).view(np.uint8)
        bad = np.nonzero(gv != rv)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[:8]}")


def special_rows(device):
    """Constant, mixed-sign zeros, one outlier, tiny, huge, two-valued rows."""
    g = torch.Generator().manual_seed(2)
    base = torch.randn((8, 128), generator=g)
    rows = [torch.full((128,), -1.75), torch.where(torch.arange(128) % 3 == 0, -0.0, 0.0),
            torch.cat([base[0, :127] * 0.01, torch.tensor([100.0])]), base[1] * 1e-30,
            base[2] * 1e30, torch.where(base[3] > 0, 2.0, -3.0), base[4].round(), base[5]]
    return torch.stack(rows).to(torch.bfloat16).to(device)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("shape", [(2, 512, 3), (1, 333, 2), (3, 128, 8)])
def test_int_baseline_matches_oracle(lynx_lib, oracle_mod, cuda_dev, bits, shape):
    from split_stream_kv_gb300 import synth
    B, L, H = shape
    kv = synth.kv_cache(B, L, H, 128, seed=B + L + H + bits, device=cuda_dev, n_outlier=2)
    codes, meta = lynx_lib.lynx_int_encode(kv, bits)
    f32 = lynx_lib.lynx_int_decode(codes, meta, bits, torch.float32)
    b16 = lynx_lib.lynx_int_decode(codes, meta, bits, torch.bfloat16)
    torch.cuda.synchronize()
    oc, om = oracle_mod.int_encode(bits_of(kv), bits)
    same_bytes(codes, oc, "codes")
    same_bytes(meta, om, "meta")
    ref = oracle_mod.int_decode(oc, om, bits)
    same_bytes(f32, ref, "decode fp32")
    assert np.array_equal(bits_of(b16), oracle_mod.f32_to_bf16_bits(ref))


@pytest.mark.parametrize("bits", [8, 4])
def test_int_baseline_special_rows(lynx_lib, oracle_mod, cuda_dev, bits):
    kv = special_rows(cuda_dev)
    codes, meta = lynx_lib.lynx_int_encode(kv, bits)
    f32 = lynx_lib.lynx_int_decode(codes, meta, bits, torch.float32)
    torch.cuda.synchronize()
    oc, om = oracle_mod.int_encode(bits_of(kv), bits)
    same_bytes(codes, oc, "codes")
    same_bytes(meta, om, "meta")
    same_bytes(f32, oracle_mod.int_decode(oc, om, bits), "decode")


def test_int_baseline_at_scale_on_samples(lynx_lib, oracle_mod, cuda_dev):
    """The Llama-3-8B-shaped codec tensor (64 x 16384 tokens x 8 heads): seeded
    rows against the oracle."""
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(64, 16384, 8, 128, seed=11, device=cuda_dev)
    flat = kv.view(-1, 128)
    rng = np.random.default_rng(1)
    idx = torch.from_numpy(rng.choice(flat.shape[0], size=4096, replace=False)).to(cuda_dev)
    xs = bits_of(flat[idx])
    for bits in (8, 4):
        codes, meta = lynx_lib.lynx_int_encode(kv, bits)
        torch.cuda.synchronize()
        oc, om = oracle_mod.int_encode(xs, bits)
        same_bytes(codes.view(-1, codes.shape[-1])[idx], oc, f"INT{bits} codes")
        same_bytes(meta.view(-1, 2)[idx], om, f"INT{bits} meta")
        del codes, meta


CASES = [(2, 512, 2, 128, 32), (1, 512, 3, 256, 64), (3, 256, 1, 64, 16), (2, 384, 2, 128, 128),
         (1, 1024, 2, 512, 32), (2, 1024, 1, 512, 16)]


@pytest.mark.parametrize("k", [3, 4, 5, 6])
@pytest.mark.parametrize("rows", [1, 63, 100, 64 * 3 + 17, 64 * 40])
def test_bit_splits_ragged_rows(lynx_lib, oracle_mod, cuda_dev, k, rows):
    """Raw 4+4 streams of any row count: the kernel stages 64 rows (256 quads)
    at a time, so counts that are not a multiple of 64 end in a partial tile."""
    g = torch.Generator(device="cpu").manual_seed(1000 * k + rows)
    anc = torch.randint(0, 256, (rows, 64), generator=g, dtype=torch.uint8)
    res = torch.randint(0, 256, (rows, 64), generator=g, dtype=torch.uint8)
    ak, rk = lynx_lib.lynx_split_bits(anc.to(cuda_dev), res.to(cuda_dev), k)
    a4, r4 = lynx_lib.lynx_join_bits(ak, rk, k)
    torch.cuda.synchronize()
    ok_, okr = oracle_mod.split_bits(anc.numpy(), res.numpy(), k)
    same_bytes(ak, ok_, "anchor_k")
    same_bytes(rk, okr, "residual_k")
    assert torch.equal(a4.cpu(), anc) and torch.equal(r4.cpu(), res)


@pytest.mark.parametrize("k", [3, 4, 5, 6])
@pytest.mark.parametrize("B,L,H,P,C", CASES)
def test_bit_splits_match_oracle(lynx_lib, oracle_mod, cuda_dev, k, B, L, H, P, C):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(B, L, H, 128, seed=7 * k + L + P, device=cuda_dev, n_outlier=2)
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
    ak, rk = lynx_lib.lynx_split_bits(anc, res, k)
    a4, r4 = lynx_lib.lynx_join_bits(ak, rk, k)
    f32 = lynx_lib.lynx_decode_anchor_bits(ak, meta, L, P, C, ALPHA, k, torch.float32)
    b16 = lynx_lib.lynx_decode_anchor_bits(ak, meta, L, P, C, ALPHA, k, torch.bfloat16)
    torch.cuda.synchronize()
    oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, ALPHA)
    ok_, okr = oracle_mod.split_bits(oa, orr, k)
    same_bytes(ak, ok_, "anchor_k")
    same_bytes(rk, okr, "residual_k")
    assert torch.equal(a4, anc) and torch.equal(r4, res)        # join inverts split
    ref = oracle_mod.decode_anchor_bits(ok_, om, L, P, C, ALPHA, k)
    same_bytes(f32, ref, "decode anchor k fp32")
    assert np.array_equal(bits_of(b16), oracle_mod.f32_to_bf16_bits(ref))
    if k == 4:       # the 4-bit split decodes like the 4+4 Anchor decoder
        plain = lynx_lib.lynx_decode_anchor(anc, meta, L, P, C, ALPHA, torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(plain, f32)


def test_vnmse_harness_matches_the_oracle(lynx_lib, oracle_mod, cuda_dev):
    """The benchmark's accuracy table (GPU decodes, float64 attention) agrees
    with the oracle's float64 attention over the oracle's decodes."""
    import bench
    from split_stream_kv_gb300 import synth
    B, L, Hkv, Hq, T = 2, 1024, 2, 8, 4
    K = synth.kv_cache(B, L, Hkv, 128, seed=21, device=cuda_dev, n_outlier=2)
    V = synth.kv_cache(B, L, Hkv, 128, seed=22, device=cuda_dev, n_outlier=2)
    q = synth.queries(B, T, Hq, 128, seed=23, device=cuda_dev)
    table = bench.accuracy_table(K, V, q, P=128, C=32, alpha=ALPHA, sweep=False)
    qf = q.float().cpu().numpy()

    def bf(x):
        return oracle_mod.bf16_bits_to_f32(oracle_mod.f32_to_bf16_bits(x))

    kb, vb = bits_of(K), bits_of(V)
    ref = oracle_mod.attention_rows(qf, oracle_mod.bf16_bits_to_f32(kb),
                                    oracle_mod.bf16_bits_to_f32(vb))
    want = {}
    for bits in (8, 4):
        kc, km = oracle_mod.int_encode(kb, bits)
        vc, vm = oracle_mod.int_encode(vb, bits)
        o = oracle_mod.attention_rows(qf, bf(oracle_mod.int_decode(kc, km, bits)),
                                      bf(oracle_mod.int_decode(vc, vm, bits)))
        want[f"int{bits}"] = oracle_mod.vnmse(o, ref)
    ka, kr, kmeta = oracle_mod.encode(kb, 128, 32, ALPHA)
    va, vr, vmeta = oracle_mod.encode(vb, 128, 32, ALPHA)
    o = oracle_mod.attention_rows(qf, bf(oracle_mod.decode(ka, kr, kmeta, L, 128, 32, ALPHA)),
                                  bf(oracle_mod.decode(va, vr, vmeta, L, 128, 32, ALPHA)))
    want["lynx_full"] = oracle_mod.vnmse(o, ref)
    for k in (3, 4, 5, 6):
        kk, _ = oracle_mod.split_bits(ka, kr, k)
        vk, _ = oracle_mod.split_bits(va, vr, k)
        o = oracle_mod.attention_rows(
            qf, bf(oracle_mod.decode_anchor_bits(kk, kmeta, L, 128, 32, ALPHA, k)),
            bf(oracle_mod.decode_anchor_bits(vk, vmeta, L, 128, 32, ALPHA, k)))
        want[f"lynx_anchor_{k}bit"] = oracle_mod.vnmse(o, ref)
    a1k = oracle_mod.a1_encode(kb, 128, 100.0)
    a1v = oracle_mod.a1_encode(vb, 128, 100.0)
    o = oracle_mod.attention_rows(qf, bf(oracle_mod.a1_decode(*a1k, L, 128, 100.0)),
                                  bf(oracle_mod.a1_decode(*a1v, L, 128, 100.0)))
    want["a1_full"] = oracle_mod.vnmse(o, ref)
    o = oracle_mod.attention_rows(qf, bf(oracle_mod.a1_decode(a1k[0], None, a1k[2], L, 128, 100.0)),
                                  bf(oracle_mod.a1_decode(a1v[0], None, a1v[2], L, 128, 100.0)))
    want["a1_anchor"] = oracle_mod.vnmse(o, ref)
    for name, w in want.items():
        got = table[name]["vnmse"]
        assert abs(got - w) <= 1e-3 * w + 1e-9, (name, got, w)
    # the pages' two headline comparisons (Table 3): the full Lynx code beats
    # INT8 and its 4-bit Anchor beats INT4
    assert want["lynx_full"] < want["int8"]
    assert want["lynx_anchor_4bit"] < want["int4"]
    print({n: f"{v:.3g}" for n, v in want.items()})


A1_CASES = [(2, 512, 2, 128), (1, 512, 3, 256), (3, 256, 1, 64), (2, 1024, 2, 512)]


@pytest.mark.parametrize("B,L,H,P", A1_CASES)
@pytest.mark.parametrize("alpha", [100.0, 255.0, 1.0, 0.5])
def test_a1_variant_matches_oracle(lynx_lib, oracle_mod, cuda_dev, B, L, H, P, alpha):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(B, L, H, 128, seed=B * 3 + L + P, device=cuda_dev, n_outlier=2)
    kv[0, :P, 0, 5] = 0          # a zero channel in one page block
    anc, res, meta = lynx_lib.lynx_a1_encode(kv, P, alpha)
    torch.cuda.synchronize()
    oa, orr, om = oracle_mod.a1_encode(bits_of(kv), P, alpha)
    same_bytes(anc, oa, "a1 anchor")
    same_bytes(res, orr, "a1 residual")
    same_bytes(meta, om, "a1 meta")
    for r_gpu, r_or, what in ((res, orr, "full"), (None, None, "anchor")):
        ref = oracle_mod.a1_decode(oa, r_or, om, L, P, alpha)
        f32 = lynx_lib.lynx_a1_decode(anc, r_gpu, meta, L, P, alpha, torch.float32)
        b16 = lynx_lib.lynx_a1_decode(anc, r_gpu, meta, L, P, alpha, torch.bfloat16)
        torch.cuda.synchronize()
        same_bytes(f32, ref, f"a1 decode {what}")
        assert np.array_equal(bits_of(b16), oracle_mod.f32_to_bf16_bits(ref)), what


def test_a1_variant_special_values(lynx_lib, oracle_mod, cuda_dev):
    """Infinities (a page maximum of inf makes every scale 0), a NaN (coded
    0, left out of the maxima), signed zeros, an all-zero channel, the
    largest finite BF16 and a subnormal: codes and metadata as the oracle's."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn((1, 256, 2, 128), generator=g)
    x[0, 3, 0, 5] = float("inf")
    x[0, 40, 1, 9] = float("-inf")
    x[0, 77, 0, 17] = float("nan")
    x[0, 100, 1, 33] = -0.0
    x[0, :, 0, 60] = 0.0
    x[0, 200, 1, 70] = 3.3895e38
    x[0, 5, 1, 90] = 1e-40
    kv = x.to(torch.bfloat16).to(cuda_dev)
    for P in (64, 128, 256):
        anc, res, meta = lynx_lib.lynx_a1_encode(kv, P, 100.0)
        torch.cuda.synchronize()
        oa, orr, om = oracle_mod.a1_encode(bits_of(kv), P, 100.0)
        same_bytes(anc, oa, f"a1 anchor P={P}")
        same_bytes(res, orr, f"a1 residual P={P}")
        same_bytes(meta, om, f"a1 meta P={P}")
