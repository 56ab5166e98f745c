"""Host logic of bench.py that needs no GPU: the DRAM rate beside the
roofline, and the traffic records keyed to the kernels' current sources."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_dram_rate():
    # 13.65 GB in 4.86 ms against a 6,789.6 GB/s peak
    r = bench.dram_rate(13.65e9, 4.86, 6789.6)
    assert r["dram_gbs"] == pytest.approx(13.65e9 / 4.86e-3 / 1e9)
    assert r["dram_frac"] == pytest.approx(r["dram_gbs"] / 6789.6)
    assert 0.40 < r["dram_frac"] < 0.42
    assert bench.dram_rate(None, 4.86, 6789.6) == {}
    assert bench.dram_rate(1e9, 0.0, 6789.6) == {}


def test_traffic_records_match_the_current_sources():
    """Every committed DRAM-traffic record names the hash of its kernel family's
    sources; a record taken on other sources is not reported (null)."""
    with open(bench.TRAFFIC_FILE) as f:
        t = json.load(f)
    for wl, d in t.items():
        if wl.startswith("_"):
            continue
        for k, e in d.items():
            assert e["dram_bytes_per_launch"] > 0
            assert bench.traffic_for(k, wl) == (e["dram_bytes_per_launch"]
                                                if e["source_hash"] == bench.source_hash(k) else None)
    assert bench.traffic_for("gt_bwd_dkdv", "no_such_workload") is None
