"""Host-side pieces of bench.py that feed the roofline: the algorithmic bytes
of each row and the DRAM-traffic records read from profiles/traffic.md."""
import re

import pytest

import bench

ROWS = ("encode", "decode_anchor", "decode_full", "attn_draft", "attn_verify")


def test_algorithmic_bytes_of_the_bench_workload():
    """Per element at page 128, C 32 (metadata 8/128 + 8/32 = 0.3125 B):
    encode 2 + 0.5 + 0.5 + meta, Anchor decode 0.5 + meta + 2, full decode
    1 + meta + 2; attention reads 0.5 (draft) or 1 (verify) + meta per K or V
    element.  1,073,741,824 codec elements; 536,870,912 K+V elements."""
    alg = bench.algorithmic_bytes()
    assert bench.codec_elems() == 1 << 30
    assert bench.attn_kv_elems() == 1 << 29
    assert alg["encode"] == 3.3125 * (1 << 30) == 3556769792
    assert alg["decode_anchor"] == 2.8125 * (1 << 30) == 3019898880
    assert alg["decode_full"] == alg["encode"]
    assert alg["attn_draft"] == 0.8125 * (1 << 29) == 436207616
    assert alg["attn_verify"] == 1.3125 * (1 << 29) == 704643072


def _records():
    rec = {}
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.md")) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] in ROWS:
                rec[cells[0]] = cells[1:4]
    return rec


def test_every_row_has_a_traffic_record():
    rec = _records()
    assert set(rec) == set(ROWS)
    for row, (sha, units, nbytes) in rec.items():
        assert re.fullmatch(r"[0-9a-f]{16}", sha), row
        assert float(units) > 0 and float(nbytes) > 0, row


@pytest.mark.parametrize("row", ROWS)
def test_recorded_traffic_is_near_the_algorithmic_bytes(row):
    """Where the record matches the current sources, the measured DRAM bytes
    of a launch lie within 10 % of what the row must move (more would mean
    re-reads; much less, a mis-scaled record)."""
    t = bench.recorded_traffic(row, bench.units_per_launch(row))
    if t is None:
        pytest.skip("sources changed since the capture: the bench reports no traffic")
    alg = bench.algorithmic_bytes()[row]
    assert 0.9 * alg <= t <= 1.1 * alg, (row, t, alg)


def test_recorded_traffic_ignores_a_stale_record(monkeypatch):
    monkeypatch.setattr(bench, "sources_hash", lambda row: "0" * 16)
    for row in ROWS:
        assert bench.recorded_traffic(row, bench.units_per_launch(row)) is None
