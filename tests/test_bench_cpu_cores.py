"""bench.py's all-cores oracle timing on CPU: one spawned process per core,
each running the unchanged oracle on its share, reported as one throughput."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_all_cores_oracle_timing():
    wl = bench.QwzFP16()
    d = bench.time_cpu_all_cores(wl, 1 << 20)
    assert "error" not in d, d
    assert d["cores"] == len(os.sched_getaffinity(0)) and d["kind"] == "oracle"
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["seconds"] > 0
