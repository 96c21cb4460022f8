"""The ncu summaries under profiles/ stay reproducible: every command they
quote runs committed files only, every ncu command keeps the GPU's clocks
(--clock-control none) and repeats a plain run quoted before it (the plain run
exits 0 first), every bench.py command line is one bench.py accepts today, and
the traffic table names launch lists and workloads that exist."""
import glob
import json
import os
import shlex
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def commands(path):
    """The commands of the fenced blocks of one summary, continuation lines
    joined, in order."""
    out, block, cur = [], False, ""
    with open(path) as f:
        for line in f:
            if line.startswith("```"):
                block = not block
                continue
            if not block:
                continue
            line = line.strip()
            if line.endswith("\\"):
                cur += line[:-1] + " "
                continue
            cur += line
            if cur.strip():
                out.append(cur.strip())
            cur = ""
    return out


def bench_argv(cmd):
    """The bench.py arguments of a command ("python bench.py ..." alone or at
    the end of an ncu command), or None."""
    words = shlex.split(cmd)
    for i in range(len(words) - 1):
        if words[i] == "python" and words[i + 1] == "bench.py":
            return words[i + 2:]
    return None


def test_every_summary_quotes_its_commands():
    assert SUMMARIES
    for path in SUMMARIES:
        cmds = commands(path)
        assert any(c.startswith("ncu ") for c in cmds), os.path.basename(path)


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_commands_are_reproducible(path):
    plain = []
    for cmd in commands(path):
        assert "_work" not in cmd and "/root" not in cmd, cmd
        argv = bench_argv(cmd)
        assert argv is not None, f"a command that is not bench.py or ncu on it: {cmd}"
        bench.parse_args(argv)  # exits (SystemExit) on an option bench.py refuses
        if cmd.startswith("ncu "):
            words = shlex.split(cmd)
            assert "--clock-control" in words, cmd
            assert words[words.index("--clock-control") + 1] == "none", cmd
            assert argv in plain, f"ncu on a command with no plain run before it: {cmd}"
            if "--set" in words or "--section" in words:  # many passes: one kernel, few launches
                assert "-k" in words and int(words[words.index("-c") + 1]) <= 3, cmd
        else:
            plain.append(argv)


def test_bench_refuses_options_of_another_workload():
    with pytest.raises(SystemExit):
        bench.parse_args(["--pair", "4:128"])  # the default workload is not gm_sweep
    with pytest.raises(SystemExit):
        bench.parse_args(["--workload", "gm_sweep", "--pair", "3:128"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--workload", "gm_sweep", "--pair", "4:100"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--workload", "gm_sweep", "--pair", "four"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--schedule-steps", "36"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    a = bench.parse_args(["--workload", "gm_sweep", "--pair", "8:1024", "--configs", "none"])
    assert a.pair == "8:1024" and a.configs == "none"
    assert bench.parse_args(["--impl", "reference", "--warmup", "0"]).warmup == 0


def test_traffic_table_names_existing_lists_and_workloads():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    assert set(d["source_sets"]) == {"codec", "gemm"}
    for name in d["source"].replace(",", " ").split():
        if name.endswith(".md"):
            assert os.path.exists(os.path.join(ROOT, "profiles", name)), name
    for wl, fams in d["workloads"].items():
        assert wl in bench.WORKLOADS, wl
        assert fams and all(isinstance(v, int) and v > 0 for v in fams.values()), wl
