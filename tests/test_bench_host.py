"""bench.py's host-side bookkeeping: the algorithmic byte formulas agree with
the oracle's sizes, and DRAM traffic from the committed ncu summaries is only
reported for the kernel sources it was taken on."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle as O  # noqa: E402


@pytest.mark.parametrize("fmt", [O.INT2, O.INT4, O.INT6, O.INT8, O.E4M3])
def test_packed_bytes_match_the_oracle(fmt):
    for G in (32, 64, 128, 256, 512, 1024):
        for n in (1, G - 1, G, 3 * G + 5, 8192 * 8192):
            assert bench.packed_bytes(fmt, n, G) == O.codes_bytes(fmt, n) + 4 * O.num_blocks(n, G)


def test_traffic_is_keyed_by_the_kernel_sources(monkeypatch):
    d = {"source_sets": {"codec": "c" * 16, "gemm": "g" * 16},
         "workloads": {"llama70b": {"quantize": 123}, "llama70b_gemm": {"gemm_dequant": 456}}}
    monkeypatch.setattr(bench.json, "load", lambda f: d)
    monkeypatch.setattr(bench, "csrc_sha", lambda sset: {"codec": "c" * 16, "gemm": "g" * 16}[sset])
    assert bench.lookup_traffic("llama70b", "quantize") == 123
    assert bench.lookup_traffic("llama70b_gemm", "gemm_dequant") == 456
    # a change in the GEMM's sources leaves the codec captures valid, and the reverse
    monkeypatch.setattr(bench, "csrc_sha", lambda sset: {"codec": "c" * 16, "gemm": "x" * 16}[sset])
    assert bench.lookup_traffic("llama70b", "quantize") == 123
    assert bench.lookup_traffic("llama70b_gemm", "gemm_dequant") is None
    monkeypatch.setattr(bench, "csrc_sha", lambda sset: "0" * 16)
    assert bench.lookup_traffic("llama70b", "quantize") is None


def test_source_sets_split_the_gemm_files():
    assert bench.source_set("gemm_dequant") == "gemm" and bench.source_set("quantize") == "codec"
    assert bench.csrc_sha("codec") != bench.csrc_sha("gemm")
