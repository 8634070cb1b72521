"""Split-stream transfer on the GPU ("Lynx: Progressive Speculative KV Cache
Transfer for Disaggregated LLM Inference", technical review, Mechanism 2 and
Figure 4; Implementation Notes), through the C ABI.

Receiver: the streams the oracle encoded are copied from pinned host memory;
once every Anchor has landed the output holds, group by group, either the
oracle's Anchor-only decode or (for groups already upgraded) its full decode,
and at the end exactly the full decode.  Sender: encoding group by group and
copying to host gives the oracle's streams bit for bit.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def pinned_like(a: np.ndarray):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


def device_streams(lynx, B, L, H, P, C, dev):
    ca, cr, cm = lynx.stream_shapes(B, L, H, 128, P, C)
    return (torch.empty(ca, dtype=torch.uint8, device=dev),
            torch.empty(cr, dtype=torch.uint8, device=dev),
            torch.empty(cm, dtype=torch.float32, device=dev))


def page_groups(B, L, H, P, G):
    """Token-row ranges of the flattened [B*L] axis covered by each group."""
    pages = B * (L // P)
    return [(g * P, min(g + G, pages) * P) for g in range(0, pages, G)]


CASES = [(3, 512, 2, 128, 32, 2), (2, 1024, 3, 256, 64, 3), (1, 768, 1, 64, 16, 1),
         (2, 512, 2, 128, 128, 100)]


@pytest.mark.parametrize("B,L,H,P,C,G", CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_receive_anchor_phase_then_full(lynx_lib, oracle_mod, cuda_dev, B, L, H, P, C, G,
                                        out_dtype):
    from split_stream_kv_gb300 import synth
    errors_before = lynx_lib.lynx_device_errors()   # sticky bits other tests set on purpose
    kv = synth.kv_cache(B, L, H, 128, seed=B * 7 + L + G, device=cuda_dev, n_outlier=2)
    oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, ALPHA)
    ref_full = oracle_mod.decode(oa, orr, om, L, P, C, ALPHA)
    ref_anc = oracle_mod.decode(oa, None, om, L, P, C, ALPHA)
    host = (pinned_like(oa), pinned_like(orr), pinned_like(om))
    dev = device_streams(lynx_lib, B, L, H, P, C, cuda_dev)
    out = torch.full((B, L, H, 128), float("nan"), dtype=out_dtype, device=cuda_dev)
    copy_s = torch.cuda.Stream(cuda_dev)
    hi = torch.cuda.Stream(cuda_dev, priority=-1)
    lo = torch.cuda.Stream(cuda_dev, priority=0)
    a_ready, f_ready = torch.cuda.Event(), torch.cuda.Event()
    torch.cuda.synchronize()
    # hold the low-priority queue (a bounded sleep) so that the Anchor phase
    # can be observed before any upgrade
    with torch.cuda.stream(lo):
        torch.cuda._sleep(200_000_000)
    lynx_lib.lynx_split_receive(host, dev, L, P, C, ALPHA, G, out=out, copy_stream=copy_s,
                                hi_stream=hi, lo_stream=lo, anchor_ready=a_ready,
                                full_ready=f_ready)
    with torch.cuda.stream(hi):
        a_ready.wait(hi)
        snap = out.clone()
    hi.synchronize()
    f_ready.synchronize()
    torch.cuda.synchronize()

    def as_ref(x):
        return (oracle_mod.f32_to_bf16_bits(x) if out_dtype == torch.bfloat16
                else x.view(np.uint32))

    def as_got(t):
        return bits_of(t) if out_dtype == torch.bfloat16 else t.cpu().numpy().view(np.uint32)

    rf, ra = as_ref(ref_full).reshape(B * L, -1), as_ref(ref_anc).reshape(B * L, -1)
    s = as_got(snap).reshape(B * L, -1)
    n_anchor = 0
    for t0, t1 in page_groups(B, L, H, P, G):
        if np.array_equal(s[t0:t1], ra[t0:t1]):
            n_anchor += 1
        else:
            assert np.array_equal(s[t0:t1], rf[t0:t1]), f"group rows {t0}..{t1}: neither phase"
    print(f"groups in the Anchor phase at anchor_ready: {n_anchor}")
    assert np.array_equal(as_got(out).reshape(B * L, -1), rf)
    for d, h in zip(dev, host):
        assert torch.equal(d.cpu(), h)
    assert lynx_lib.lynx_device_errors() == errors_before
    assert errors_before & 1 == 0


def test_receive_without_output_copies_the_streams(lynx_lib, cuda_dev):
    B, L, H, P, C = 4, 1024, 2, 128, 32
    g = torch.Generator().manual_seed(3)
    ca, cr, cm = lynx_lib.stream_shapes(B, L, H, 128, P, C)
    host = (torch.randint(0, 256, ca, dtype=torch.uint8, generator=g).pin_memory(),
            torch.randint(0, 256, cr, dtype=torch.uint8, generator=g).pin_memory(),
            torch.randn(cm, generator=g).pin_memory())
    dev = device_streams(lynx_lib, B, L, H, P, C, cuda_dev)
    a_ready, f_ready = torch.cuda.Event(), torch.cuda.Event()
    lynx_lib.lynx_split_receive(host, dev, L, P, C, ALPHA, 5, anchor_ready=a_ready,
                                full_ready=f_ready)
    a_ready.synchronize()
    assert torch.equal(dev[0].cpu(), host[0]) and torch.equal(dev[2].cpu(), host[2])
    f_ready.synchronize()
    assert torch.equal(dev[1].cpu(), host[1])


@pytest.mark.parametrize("B,L,H,P,C,G", CASES)
def test_send_gives_the_oracle_streams(lynx_lib, oracle_mod, cuda_dev, B, L, H, P, C, G):
    from split_stream_kv_gb300 import synth
    kv = synth.kv_cache(B, L, H, 128, seed=B * 5 + L + G, device=cuda_dev, n_outlier=2)
    oa, orr, om = oracle_mod.encode(bits_of(kv), P, C, ALPHA)
    dev = device_streams(lynx_lib, B, L, H, P, C, cuda_dev)
    host = tuple(torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in dev)
    hi, copy_s = torch.cuda.Stream(cuda_dev, priority=-1), torch.cuda.Stream(cuda_dev)
    a_sent, all_sent = torch.cuda.Event(), torch.cuda.Event()
    torch.cuda.synchronize()
    lynx_lib.lynx_split_send(kv, P, C, ALPHA, dev, host, G, hi_stream=hi, copy_stream=copy_s,
                             anchor_sent=a_sent, all_sent=all_sent)
    a_sent.synchronize()
    assert host[0].numpy().tobytes() == oa.tobytes()
    assert host[2].numpy().tobytes() == om.tobytes()
    all_sent.synchronize()
    assert host[1].numpy().tobytes() == orr.tobytes()


def test_send_then_receive_at_scale(lynx_lib, oracle_mod, cuda_dev):
    """A Llama-3-8B-shaped slice (8 tensors x 16384 tokens x 8 heads): sender,
    host, receiver; the receiver's output equals the one-shot full decode,
    and seeded page blocks equal the oracle's decode."""
    from split_stream_kv_gb300 import synth
    B, L, H, P, C, G = 8, 16384, 8, 128, 32, 96
    errors_before = lynx_lib.lynx_device_errors()
    kv = synth.kv_cache(B, L, H, 128, seed=17, device=cuda_dev)
    dev = device_streams(lynx_lib, B, L, H, P, C, cuda_dev)
    host = tuple(torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in dev)
    lynx_lib.lynx_split_send(kv, P, C, ALPHA, dev, host, G)
    torch.cuda.synchronize()
    rx = device_streams(lynx_lib, B, L, H, P, C, cuda_dev)
    out = torch.empty_like(kv)
    f_ready = torch.cuda.Event()
    lynx_lib.lynx_split_receive(host, rx, L, P, C, ALPHA, G, out=out,
                                hi_stream=torch.cuda.Stream(cuda_dev, priority=-1),
                                lo_stream=torch.cuda.Stream(cuda_dev), full_ready=f_ready)
    f_ready.synchronize()
    torch.cuda.synchronize()
    one_shot = lynx_lib.lynx_decode_full(*dev, L, P, C, ALPHA, torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out, one_shot)
    rng = np.random.default_rng(5)
    NB = L // P
    xb = bits_of(kv)
    for flat in rng.choice(B * NB, size=12, replace=False):
        b, p = divmod(int(flat), NB)
        blk = xb[b:b + 1, p * P:(p + 1) * P]
        oa, orr, om = oracle_mod.encode(blk, P, C, ALPHA)
        ref = oracle_mod.decode(oa, orr, om, P, P, C, ALPHA)
        got = bits_of(out[b:b + 1, p * P:(p + 1) * P])
        assert np.array_equal(got, oracle_mod.f32_to_bf16_bits(ref)), (b, p)
    assert lynx_lib.lynx_device_errors() == errors_before
    assert errors_before & 1 == 0
