"""Guards on the CUDA kernels (the race-detection plan of the build, with
compute-sanitizer unavailable): every output buffer sits between canary
regions that must come back untouched, every kernel run twice on the same
inputs gives bitwise-equal outputs, and a bounded wait on a barrier that
nothing completes gives up, reports it, and leaves the context usable."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALPHA = 255.0
GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` placed inside a byte buffer whose GUARD
    bytes before and after hold PATTERN (offset keeps 16-byte alignment)."""

    def __init__(self, shape, dtype, device):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def intact(self):
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[-GUARD:].cpu().numpy()
        return (head == PATTERN).all() and (tail == PATTERN).all()


def twice(run, outs):
    """Run `run(outs)` into two guarded copies; check canaries and equality."""
    dev = outs[0][2]
    a = [Guarded(s, d, dev) for s, d, _ in outs]
    b = [Guarded(s, d, dev) for s, d, _ in outs]
    run([g.t for g in a])
    run([g.t for g in b])
    torch.cuda.synchronize()
    for i, (ga, gb) in enumerate(zip(a, b)):
        assert ga.intact() and gb.intact(), f"output {i}: a canary was overwritten"
        assert torch.equal(ga.t.view(torch.uint8), gb.t.view(torch.uint8)), \
            f"output {i}: two runs differ"
    return [g.t for g in a]


@pytest.fixture(scope="module")
def kv(cuda_dev):
    from split_stream_kv_gb300 import synth
    return synth.kv_cache(2, 512, 2, 128, seed=3, device=cuda_dev, n_outlier=2)


def test_codec_guards_and_determinism(lynx_lib, cuda_dev, kv):
    B, L, H, _ = kv.shape
    P, C = 128, 32
    ca, cr, cm = lynx_lib.stream_shapes(B, L, H, 128, P, C)
    enc = twice(lambda o: lynx_lib.lynx_encode(kv, P, C, ALPHA, o[0], o[1], o[2]),
                [(ca, torch.uint8, cuda_dev), (cr, torch.uint8, cuda_dev),
                 (cm, torch.float32, cuda_dev)])
    for dt in (torch.bfloat16, torch.float32):
        twice(lambda o: lynx_lib.lynx_decode_full(*enc, L, P, C, ALPHA, out=o[0]),
              [((B, L, H, 128), dt, cuda_dev)])
        twice(lambda o: lynx_lib.lynx_decode_anchor(enc[0], enc[2], L, P, C, ALPHA, out=o[0]),
              [((B, L, H, 128), dt, cuda_dev)])


def test_attention_guards_and_determinism(lynx_lib, cuda_dev):
    from split_stream_kv_gb300 import synth
    batch, L, Hkv, Hq, P, C = 2, 2048, 2, 8, 128, 32
    kva = synth.kv_cache(2 * batch, L, Hkv, 128, seed=9, device=cuda_dev, n_outlier=2)
    ks = lynx_lib.lynx_encode(kva[0::2].contiguous(), P, C, ALPHA)
    vs = lynx_lib.lynx_encode(kva[1::2].contiguous(), P, C, ALPHA)
    for T, mode in ((1, lynx_lib.LYNX_ANCHOR), (8, lynx_lib.LYNX_FULL)):
        q = synth.queries(batch, T, Hq, 128, seed=T, device=cuda_dev)
        ws_n = lynx_lib.lynx_attn_workspace_bytes(batch, T, Hq, L, Hkv, 128, P)
        kk = ks if mode == lynx_lib.LYNX_FULL else (ks[0], None, ks[2])
        vv = vs if mode == lynx_lib.LYNX_FULL else (vs[0], None, vs[2])
        twice(lambda o: lynx_lib.lynx_attn_decode(q, kk, vv, L, P, C, ALPHA, mode, out=o[0],
                                                  workspace=o[1]),
              [((batch, T, Hq, 128), torch.float32, cuda_dev), ((ws_n,), torch.uint8, cuda_dev)])
    q = synth.queries(batch, 4, Hq, 128, seed=4, device=cuda_dev)
    kt = synth.kv_cache(batch, 4, Hkv, 128, seed=5, device=cuda_dev)
    vt = synth.kv_cache(batch, 4, Hkv, 128, seed=6, device=cuda_dev)
    ws_n = lynx_lib.lynx_attn_workspace_bytes(batch, 4, Hq, L, Hkv, 128, P)
    twice(lambda o: lynx_lib.lynx_attn_decode(q, ks, vs, L, P, C, ALPHA, lynx_lib.LYNX_FULL,
                                              k_tail=kt, v_tail=vt, out=o[0], workspace=o[1]),
          [((batch, 4, Hq, 128), torch.float32, cuda_dev), ((ws_n,), torch.uint8, cuda_dev)])


def test_variant_guards_and_determinism(lynx_lib, cuda_dev, kv):
    B, L, H, _ = kv.shape
    P, C = 128, 32
    for bits in (8, 4):
        codes, meta = twice(lambda o: lynx_lib.lynx_int_encode(kv, bits, o[0], o[1]),
                            [((B, L, H, 128 * bits // 8), torch.uint8, cuda_dev),
                             ((B, L, H, 2), torch.float32, cuda_dev)])
        twice(lambda o: lynx_lib.lynx_int_decode(codes, meta, bits, out=o[0]),
              [((B, L, H, 128), torch.bfloat16, cuda_dev)])
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
    shp = anc.shape[:-1]
    for k in (3, 6):
        ak, rk = twice(lambda o: lynx_lib.lynx_split_bits(anc, res, k, o[0], o[1]),
                       [(shp + (16 * k,), torch.uint8, cuda_dev),
                        (shp + (16 * (8 - k),), torch.uint8, cuda_dev)])
        twice(lambda o: lynx_lib.lynx_join_bits(ak, rk, k, o[0], o[1]),
              [(shp + (64,), torch.uint8, cuda_dev), (shp + (64,), torch.uint8, cuda_dev)])
        twice(lambda o: lynx_lib.lynx_decode_anchor_bits(ak, meta, L, P, C, ALPHA, k, out=o[0]),
              [((B, L, H, 128), torch.float32, cuda_dev)])
    a1 = lynx_lib.lynx_a1_encode(kv, P)
    twice(lambda o: lynx_lib.lynx_a1_decode(*a1, L, P, out=o[0]),
          [((B, L, H, 128), torch.bfloat16, cuda_dev)])


def test_split_receive_guards(lynx_lib, cuda_dev, kv):
    B, L, H, _ = kv.shape
    P, C = 128, 32
    anc, res, meta = lynx_lib.lynx_encode(kv, P, C, ALPHA)
    host = tuple(t.cpu().pin_memory() for t in (anc, res, meta))

    def run(o):
        lynx_lib.lynx_split_receive(host, (o[0], o[1], o[2]), L, P, C, ALPHA, 3, out=o[3])

    twice(run, [(anc.shape, torch.uint8, cuda_dev), (res.shape, torch.uint8, cuda_dev),
                (meta.shape, torch.float32, cuda_dev), ((B, L, H, 128), torch.bfloat16, cuda_dev)])


def test_bounded_wait_gives_up_and_reports(lynx_lib, cuda_dev, kv):
    # nothing arrives: the wait must give up after its limit (1 ms), report 2,
    # and the context must stay usable
    assert lynx_lib.lynx_wait_selftest(1_000_000, False, cuda_dev) == 2
    assert lynx_lib.lynx_wait_selftest(1_000_000, True, cuda_dev) == 1
    # the verification pass's wait: the first gives up after 1 ms and raises
    # the abort word, the second (2 s limit) then returns at once
    assert lynx_lib.lynx_wait_selftest(1_000_000, 2, cuda_dev) == 3
    # the self-test keeps its own flag word: the library's timeout bit stays clear
    assert (lynx_lib.lynx_device_errors() & 1) == 0
    assert lynx_lib.lynx_wait_timeouts() == 0
    anc, res, meta = lynx_lib.lynx_encode(kv, 128, 32, ALPHA)
    torch.cuda.synchronize()
    assert anc.numel() > 0
