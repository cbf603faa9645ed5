"""bench.py's host-side helpers on CPU: the roofline entries and the DRAM
traffic record.

A roofline entry divides a kernel family's algorithmic bytes by its time;
for the merge loop's families the profiled time is scaled so that all
families add up to the timed train leg.  The traffic record is used only
while the kernel's source file still has the recorded hash.
"""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_roofline_entry_arithmetic():
    stats = {"merge_tail": {"launches": 10, "bytes": 2.0e6, "ms": 4.0}}
    e = bench.kernel_roofline(stats, "merge_tail", 5000.0, "measured", {}, scale=0.5)
    # 2 MB over 4 ms * 0.5 = 2 ms -> 1 GB/s
    assert e["achieved"] == pytest.approx(1.0)
    assert e["frac"] == pytest.approx(1.0 / 5000.0, abs=1e-4)
    assert e["avg_launch_ms"] == pytest.approx(0.2)
    assert e["profiled_avg_launch_ms"] == pytest.approx(0.4)
    assert e["algorithmic_bytes_per_launch"] == pytest.approx(2.0e5)
    assert e["traffic"] is None
    assert bench.kernel_roofline({}, "merge_tail", 5000.0, "measured", {}) is None
    assert bench.kernel_roofline({"x": {"launches": 0, "bytes": 1.0, "ms": 1.0}}, "x", 1.0, "m", {}) is None


def test_roofline_traffic_scales_with_the_launch():
    stats = {"pair_count": {"launches": 2, "bytes": 4.0e9, "ms": 1.0}}
    rec = {"pair_count": {"dram_bytes": 1.1e9, "algorithmic_bytes": 1.0e9, "scale": True}}
    e = bench.kernel_roofline(stats, "pair_count", 6791.0, "measured", rec)
    assert e["traffic"] == pytest.approx(2.2e9)   # 1.1 x the 2 GB of one launch
    rec["pair_count"]["scale"] = False
    assert bench.kernel_roofline(stats, "pair_count", 6791.0, "measured", rec)["traffic"] == pytest.approx(1.1e9)


def test_traffic_record_follows_the_source_hash():
    """Every committed record is either live (its source hash matches) or
    dropped; the live ones name files of this repository."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)["kernels"]
    live = bench.traffic_record()
    for name, r in rec.items():
        src = os.path.join(ROOT, r["source"])
        assert os.path.exists(src), r["source"]
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        assert (name in live) == (h == r["source_sha256"])
        assert r["dram_bytes"] > 0 and r["algorithmic_bytes"] > 0


def test_throughput_and_peaks():
    assert bench.throughput(1000, 500.0) == pytest.approx(2000.0)
    assert bench.throughput(1000, 0.0) == 0.0
    peak, kind = bench.peaks()
    assert peak > 0 and kind in ("measured", "fallback")
