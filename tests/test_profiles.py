"""The committed ncu summaries under profiles/ (CPU only): every summary
names the command that made it, every ncu command in one leaves the GPU
clocks alone and captures a bounded number of launches, and the kernel
summaries carry the fields the benchmark reads (kernel, workload, source
hash, DRAM bytes per launch) in the form it parses them."""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def fields(path):
    out = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                out[k.strip()] = v.strip().strip("`")
    return out


def test_there_are_summaries():
    assert SUMMARIES


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_ncu_commands_are_bounded_and_leave_clocks_alone(path):
    text = open(path).read()
    assert "python bench.py" in text, "a summary names the committed command that made it"
    for cmd in re.findall(r"^ncu .*$", text, flags=re.M):
        assert "--clock-control none" in cmd, cmd
        assert re.search(r"(^| )-c \d+", cmd), cmd  # a bounded number of launches
        assert "-k " in cmd or "--metrics gpu__time_duration.sum" in cmd, cmd  # one kernel, or the one-pass launch list


@pytest.mark.parametrize("path", [p for p in SUMMARIES if fields(p).get("kernel")], ids=os.path.basename)
def test_kernel_summaries_parse_as_the_benchmark_reads_them(path):
    import bench
    f = fields(path)
    assert f["kernel"] in bench.KERNEL_SOURCES
    assert os.path.basename(path).startswith(f["kernel"] + "_")
    assert re.fullmatch(r"[0-9a-f]{16}", f["source_sha256"])
    assert int(float(f["dram_bytes_per_launch"])) > 0
    # the same (kernel, workload) is summarised once, so the lookup is unambiguous
    same = [p for p in SUMMARIES if (fields(p).get("kernel"), fields(p).get("workload")) == (f["kernel"], f["workload"])]
    assert same == [path]


def test_traffic_lookup_follows_the_source_hash(monkeypatch):
    """profiled_traffic returns a summary's bytes only while its hash is the
    current source's."""
    import bench
    rows = [fields(p) for p in SUMMARIES if fields(p).get("kernel") in bench.KERNEL_SOURCES]
    assert rows
    f = rows[0]
    monkeypatch.setattr(bench, "source_sha", lambda kernel: f["source_sha256"])
    assert bench.profiled_traffic(f["kernel"], f["workload"]) == int(float(f["dram_bytes_per_launch"]))
    monkeypatch.setattr(bench, "source_sha", lambda kernel: "0" * 16)
    assert bench.profiled_traffic(f["kernel"], f["workload"]) is None
