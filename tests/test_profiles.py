"""The committed DRAM-traffic evidence matches the kernels it was taken from:
every entry of profiles/traffic.json still hashes to its kernel's source, and
names a summary that exists.  (The bench reports an entry's traffic only
while its hash matches, so a stale entry would silently drop the figure.)"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _entries():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        data = json.load(fh)
    return {k: v for k, v in data.items() if k != "about"}


def test_traffic_entries_match_current_sources():
    entries = _entries()
    assert entries
    for name, e in entries.items():
        assert bench._source_hash(e["sources"], e.get("span")) == e["sha256"], (
            f"{name}: the kernel changed since its traffic was captured")
        assert e["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, e["summary"])), name


def test_dominant_kernel_has_traffic():
    # the bench's roofline object reads this entry for the headline kernel
    assert "fused_add_rmsnorm reg 16384x8192" in _entries()
