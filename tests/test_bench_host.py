"""Host-side pieces of bench.py that feed the roofline: the algorithmic bytes
of each row, the DRAM-traffic records read from profiles/traffic.json, the
e2e pipeline's slicing and the CPU leg's rate arithmetic."""
import json
import re

import pytest

import bench

ROWS = ("encode", "decode_anchor", "decode_full", "attn_draft", "attn_verify")


def test_algorithmic_bytes_of_the_headline_workload():
    """The largest single-GPU configuration (Qwen3-235B-A22B-shaped KV at
    128K: B = 188, L = 131072, H = 4, page 256, C 64) moves per element
    encode 2 + 0.5 + 0.5 + meta, Anchor decode 0.5 + meta + 2, full decode
    1 + meta + 2 with meta = 8/256 + 8/64 = 0.15625 B; 12,616,466,432
    elements = 23.5 GiB of BF16 (the pages' Eq. 3 example).  Attention reads
    0.5 (draft) or 1 (verify) + meta (8/128 + 8/32) per K or V element of
    536,870,912."""
    alg = bench.algorithmic_bytes()
    n = bench.codec_elems()
    assert n == 188 * 131072 * 4 * 128 == 12616466432
    assert 2 * n == 25232932864                    # 23.50 GiB
    assert alg["encode"] == 3.15625 * n
    assert alg["decode_anchor"] == 2.65625 * n
    assert alg["decode_full"] == alg["encode"]
    assert bench.attn_kv_elems() == 1 << 29
    assert alg["attn_draft"] == 0.8125 * (1 << 29) == 436207616
    assert alg["attn_verify"] == 1.3125 * (1 << 29) == 704643072


def test_other_configurations_bytes():
    """Llama-3-8B at 16K: 2^30 elements at 3.3125 B (page 128, C 32); the
    Qwen-32B setting doubles the layers; the tiny case is 65,536 elements at
    page 256, C 32 (3.28125 B)."""
    c2 = bench.codec_bytes(bench.CODEC_CONFIGS["llama3-8b-16k"])
    assert c2["encode"] == 3.3125 * (1 << 30) == 3556769792
    c3 = bench.codec_bytes(bench.CODEC_CONFIGS["qwen-32b-16k"])
    assert c3["encode"] == 2 * c2["encode"]
    c1 = bench.CODEC_CONFIGS["tiny"]
    assert bench.codec_elems(c1) == 65536
    assert bench.codec_bytes(c1)["encode"] == 3.28125 * 65536


def test_e2e_slices_divide_the_batch():
    assert bench.slices_of(64) == 8
    assert bench.slices_of(188) == 4
    assert bench.slices_of(2) == 2
    assert bench.slices_of(7) == 7
    assert bench.slices_of(11) == 1


def test_step_rate_reweights_to_the_step_mix():
    """Equal codec and attention rates give that rate for the whole step; an
    attention part twice as slow per byte weighs in by its share of bytes."""
    r = bench.step_rate(1.0, 10e9, 1.0, 10e9)
    assert abs(r - 10.0) < 1e-9
    be = bench.bf16_equiv_bytes()
    wc = be["encode"] + be["decode_anchor"] + be["decode_full"]
    wa = be["attn_draft"] + be["attn_verify"]
    r = bench.step_rate(1.0, 10e9, 2.0, 10e9)
    assert abs(r - (wc + wa) / (wc / 10e9 + wa / 5e9) / 1e9) < 1e-9


def _records():
    with open(bench.TRAFFIC) as f:
        return json.load(f)["rows"]


def test_every_row_has_a_traffic_record():
    rec = _records()
    assert set(rec) == set(ROWS)
    for row, r in rec.items():
        assert re.fullmatch(r"[0-9a-f]{16}", r["sources"]), row
        assert r["units"] > 0 and r["dram_bytes"] > 0, row
        assert r["config"], row


@pytest.mark.parametrize("row", ROWS)
def test_recorded_traffic_is_near_the_algorithmic_bytes(row):
    """Where the record matches the current sources and configuration, the
    measured DRAM bytes of a launch lie within 10 % of what the row must move
    (more would mean re-reads; much less, a mis-scaled record)."""
    t = bench.recorded_traffic(row, bench.units_per_launch(row))
    if t is None:
        pytest.skip("sources or configuration changed since the capture: no traffic reported")
    alg = bench.algorithmic_bytes()[row]
    assert 0.9 * alg <= t <= 1.1 * alg, (row, t, alg)


def test_recorded_traffic_ignores_a_stale_record(monkeypatch):
    monkeypatch.setattr(bench, "sources_hash", lambda row: "0" * 16)
    for row in ROWS:
        assert bench.recorded_traffic(row, bench.units_per_launch(row)) is None


def test_recorded_traffic_scales_by_units(monkeypatch):
    rec = {"encode": {"sources": "a" * 16, "config": bench.CODEC["name"], "units": 100,
                      "dram_bytes": 330}}
    monkeypatch.setattr(bench, "traffic_records", lambda: rec)
    monkeypatch.setattr(bench, "sources_hash", lambda row: "a" * 16)
    assert bench.recorded_traffic("encode", 1000) == 3300
    rec["encode"]["config"] = "llama3-8b-16k"
    assert bench.recorded_traffic("encode", 1000) is None
