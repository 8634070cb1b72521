"""Host-side checks of the split-stream transfer that need no GPU: the
schedule obeys the pages' rules ("Lynx: Progressive Speculative KV Cache
Transfer for Disaggregated LLM Inference", technical review, Mechanism 2 and
Figure 4; Implementation Notes), and the request header matches the format
written out independently in the oracle (struct layout + zlib's CRC-32)."""
import ctypes

import pytest

ANCHOR, META, RESIDUAL = 1, 2, 3
ENCODE, DECODE_ANCHOR, UPGRADE = 0, 4, 5
Q_COPY, Q_HI, Q_LO = 0, 1, 2

# (B, L, H, page, C, pages_per_group): ragged last group, one group, one page
# per group, a group larger than the request
DIMS = [
    (2, 512, 2, 128, 32, 3),
    (3, 1024, 1, 256, 64, 2),
    (1, 256, 4, 64, 16, 1),
    (2, 384, 3, 128, 128, 100),
    (64, 16384, 8, 128, 32, 256),
]


def per_page(H, page, C, D=128):
    return H * page * D // 2, H * (2 + 2 * (page // C)) * D * 4


def check_coverage(ops, kind, per, total_pages):
    cs = [o for o in ops if o["kind"] == kind]
    off = 0
    pages = 0
    for g, o in enumerate(cs):
        assert o["group"] == g
        assert o["page0"] == pages
        assert o["offset"] == off == o["page0"] * per
        assert o["bytes"] == o["n_pages"] * per > 0
        off += o["bytes"]
        pages += o["n_pages"]
    assert pages == total_pages
    return cs


@pytest.mark.parametrize("B,L,H,P,C,G", DIMS)
def test_receive_schedule_follows_the_drain_rule(lynx_lib, B, L, H, P, C, G):
    ops = lynx_lib.lynx_split_plan(B, L, H, 128, P, C, G, send=False, with_decode=True)
    pages = B * (L // P)
    groups = -(-pages // G)
    a_pp, m_pp = per_page(H, P, C)
    for kind, per in ((ANCHOR, a_pp), (META, m_pp), (RESIDUAL, a_pp)):
        cs = check_coverage(ops, kind, per, pages)
        assert len(cs) == groups
        assert all(o["queue"] == Q_COPY for o in cs)
        if groups > 1:
            assert cs[-1]["n_pages"] == pages - (groups - 1) * G   # ragged last group
    copy_kinds = [o["kind"] for o in ops if o["queue"] == Q_COPY]
    first_res = copy_kinds.index(RESIDUAL)
    # every Anchor and meta copy precedes the first Residual copy
    assert set(copy_kinds[:first_res]) == {ANCHOR, META}
    assert set(copy_kinds[first_res:]) == {RESIDUAL}
    # group g's Anchor precedes its meta on the queue
    for g in range(groups):
        ia = next(i for i, o in enumerate(ops) if o["kind"] == ANCHOR and o["group"] == g)
        im = next(i for i, o in enumerate(ops) if o["kind"] == META and o["group"] == g)
        assert ia < im
    index = {(o["kind"], o["group"]): i for i, o in enumerate(ops)}
    last = {}
    for i, o in enumerate(ops):
        last[o["kind"]] = i
        for k, g in o["waits"]:
            j = index[(k, g)] if g >= 0 else max(jj for (kk, _), jj in index.items() if kk == k)
            assert j < i, "a wait names a later operation"
    decs = [o for o in ops if o["kind"] == DECODE_ANCHOR]
    ups = [o for o in ops if o["kind"] == UPGRADE]
    assert [o["group"] for o in decs] == list(range(groups))
    assert [o["group"] for o in ups] == list(range(groups))
    for o in decs:
        assert o["queue"] == Q_HI and (META, o["group"]) in o["waits"]
    for o in ups:
        assert o["queue"] == Q_LO and (RESIDUAL, o["group"]) in o["waits"]
    # the upgrades start after every Anchor group is decoded (the first one
    # waits for all of them; the rest follow it on the same queue)
    assert (DECODE_ANCHOR, -1) in ups[0]["waits"]
    for o in decs + ups:
        same = [c for c in ops if c["kind"] == ANCHOR and c["group"] == o["group"]][0]
        assert (o["page0"], o["n_pages"]) == (same["page0"], same["n_pages"])


@pytest.mark.parametrize("B,L,H,P,C,G", DIMS)
def test_receive_schedule_without_decode_is_copies_only(lynx_lib, B, L, H, P, C, G):
    ops = lynx_lib.lynx_split_plan(B, L, H, 128, P, C, G, send=False, with_decode=False)
    assert {o["kind"] for o in ops} == {ANCHOR, META, RESIDUAL}
    assert all(o["queue"] == Q_COPY and not o["waits"] for o in ops)


@pytest.mark.parametrize("B,L,H,P,C,G", DIMS)
def test_send_schedule_overlaps_encode_and_copies(lynx_lib, B, L, H, P, C, G):
    ops = lynx_lib.lynx_split_plan(B, L, H, 128, P, C, G, send=True)
    pages = B * (L // P)
    groups = -(-pages // G)
    a_pp, m_pp = per_page(H, P, C)
    for kind, per in ((ANCHOR, a_pp), (META, m_pp), (RESIDUAL, a_pp)):
        check_coverage(ops, kind, per, pages)
    enc = [o for o in ops if o["kind"] == ENCODE]
    assert [o["group"] for o in enc] == list(range(groups))
    assert all(o["queue"] == Q_HI for o in enc)
    for o in ops:
        if o["kind"] == ANCHOR:
            assert (ENCODE, o["group"]) in o["waits"]
    # encode g+1 is issued before the copy of group g can have finished, and
    # the copies of group g are issued before encode g+2 (ping-pong)
    kinds = [(o["kind"], o["group"]) for o in ops]
    for g in range(groups - 1):
        assert kinds.index((ENCODE, g + 1)) > kinds.index((ANCHOR, g))
        assert kinds.index((META, g)) < kinds.index((ENCODE, g + 1))
    copy_kinds = [o["kind"] for o in ops if o["queue"] == Q_COPY]
    first_res = copy_kinds.index(RESIDUAL)
    assert set(copy_kinds[:first_res]) == {ANCHOR, META}
    assert set(copy_kinds[first_res:]) == {RESIDUAL}


def test_plan_rejects_bad_arguments(lynx_lib):
    lib = lynx_lib.lib()
    n = ctypes.c_int64(-1)
    assert lib.lynx_split_plan(2, 512, 2, 128, 128, 32, 0, 0, 1, None, 0, ctypes.byref(n)) == -1
    assert lib.lynx_split_plan(2, 512, 2, 128, 96, 32, 1, 0, 1, None, 0, ctypes.byref(n)) == -3
    assert lib.lynx_split_plan(2, 500, 2, 128, 128, 32, 1, 0, 1, None, 0, ctypes.byref(n)) == -2
    buf = (lynx_lib.SplitOp * 4)()
    rc = lib.lynx_split_plan(2, 512, 2, 128, 128, 32, 3, 0, 1, buf, 4, ctypes.byref(n))
    assert rc == -5 and n.value == 15      # 3 groups x (anchor, meta, decode, residual, upgrade)
    rc = lib.lynx_split_plan(0, 512, 2, 128, 128, 32, 3, 0, 1, None, 0, ctypes.byref(n))
    assert rc == 0 and n.value == 0


OK = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: every call below fails first
BAD = ctypes.c_void_p(0x10008)


def test_receive_and_send_reject_before_enqueueing(lynx_lib):
    lib = lynx_lib.lib()

    def recv(ha=OK, out=None, ppg=2, alpha=255.0, dtype=0, page=128):
        return lib.lynx_split_receive(ha, OK, OK, OK, OK, OK, 2, 512, 2, 128, page, 32, alpha,
                                      ppg, out, dtype, None, None, None, None, None)

    assert recv(ppg=0) == -1
    assert recv(ha=None) == -1
    assert recv(ha=BAD) == -1
    assert recv(out=BAD) == -1
    assert recv(out=OK, dtype=7) == -1
    assert recv(alpha=0.0) == -1
    assert recv(page=96) == -3

    def send(kv=OK, ppg=2, alpha=255.0):
        return lib.lynx_split_send(kv, 2, 512, 2, 128, 128, 32, alpha, OK, OK, OK, OK, OK, OK,
                                   ppg, None, None, None, None)

    assert send(ppg=0) == -1
    assert send(kv=None) == -1
    assert send(kv=BAD) == -1
    assert send(alpha=float("nan")) == -1


HDR = [(2, 512, 2, 128, 32, 255.0, True), (64, 16384, 8, 128, 32, 255.0, True),
       (188, 131072, 4, 256, 64, 100.0, False), (1, 256, 1, 64, 16, 1.0, True)]


@pytest.mark.parametrize("B,L,H,P,C,alpha,res", HDR)
def test_header_matches_the_written_out_format(lynx_lib, oracle_mod, B, L, H, P, C, alpha, res):
    h = lynx_lib.lynx_header_init(B, L, H, 128, P, C, alpha, res)
    assert h == oracle_mod.request_header(B, L, H, P, C, alpha, res)
    parsed = lynx_lib.lynx_header_check(h)
    a, r, m = oracle_mod.stream_bytes(B, L, H, P, C)
    assert (parsed.anchor_bytes, parsed.meta_bytes) == (a, m)
    assert parsed.residual_bytes == (r if res else 0)
    # the Anchor phase (codes + metadata) is one contiguous byte range
    assert parsed.meta_offset == parsed.anchor_offset + parsed.anchor_bytes == 128 + a
    assert parsed.total_bytes == 128 + a + m + parsed.residual_bytes


def test_header_rejects_every_corruption(lynx_lib, oracle_mod):
    h = bytearray(lynx_lib.lynx_header_init(2, 512, 2, 128, 128, 32, 255.0))
    for i in range(len(h)):
        for bit in (0, 7):
            bad = bytearray(h)
            bad[i] ^= 1 << bit
            with pytest.raises(lynx_lib.LynxError):
                lynx_lib.lynx_header_check(bytes(bad))
    # well-formed CRC but inconsistent contents
    a, r, m = oracle_mod.stream_bytes(2, 512, 2, 128, 32)
    for hdr in (oracle_mod.request_header(2, 512, 2, 128, 32, 255.0, sizes=(a, r, m + 512)),
                oracle_mod.request_header(2, 512, 2, 128, 32, 255.0, version=2),
                oracle_mod.request_header(2, 500, 2, 128, 32, 255.0),
                oracle_mod.request_header(2, 512, 2, 128, 32, -1.0)):
        with pytest.raises(lynx_lib.LynxError):
            lynx_lib.lynx_header_check(hdr)
