"""The committed profiler evidence keeps to the capture rules: every ncu
command leaves the GPU clocks alone, full-size DRAM records use one-pass
metrics only, and every record names a workload bench.py can run."""
import glob
import json
import os
import re

import pytest

from moe_grouped_gemm_side_gb300 import workloads as wl

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
ONE_PASS = {"dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum"}


def _ncu_commands():
    """Every ncu command in the profile summaries, continuation lines joined."""
    out = []
    for path in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        lines = open(path).read().splitlines()
        i = 0
        while i < len(lines):
            line = lines[i].strip()
            if line.startswith("ncu "):
                cmd = line
                while cmd.endswith("\\") and i + 1 < len(lines):
                    i += 1
                    cmd = cmd[:-1] + " " + lines[i].strip()
                out.append((os.path.basename(path), cmd))
            i += 1
    return out


def test_profiles_hold_only_text_summaries():
    for path in glob.glob(os.path.join(PROFILES, "*")):
        assert os.path.splitext(path)[1] in (".md", ".txt", ".json"), path
        assert os.path.getsize(path) < 64 * 1024, path


def test_every_ncu_command_leaves_the_clocks_alone():
    cmds = _ncu_commands()
    assert len(cmds) >= 10
    for name, cmd in cmds:
        assert "--clock-control none" in cmd, (name, cmd)


def test_every_ncu_command_is_limited_to_one_kernel_and_few_launches():
    """A launch list (device time alone, one pass) may cover many launches;
    any other capture names one kernel and takes at most three launches."""
    for name, cmd in _ncu_commands():
        m = re.search(r"--metrics (\S+)", cmd)
        if m and m.group(1) == "gpu__time_duration.sum":
            continue
        assert re.search(r"-k '?regex:\S+", cmd), (name, cmd)
        m = re.search(r"-c (\d+)", cmd)
        assert m and int(m.group(1)) <= 3, (name, cmd)


def test_dram_traffic_records():
    recs = json.load(open(os.path.join(PROFILES, "dram_traffic.json")))
    assert recs
    for w, r in recs.items():
        assert w in wl.WORKLOADS, w
        cmd = r["command"]
        assert "--clock-control none" in cmd, w
        metrics = set(re.search(r"--metrics (\S+)", cmd).group(1).split(","))
        assert metrics <= ONE_PASS, (w, metrics)
        assert f"--workload {w}" in cmd, w
        assert len(r["launch_read_bytes"]) == len(r["launch_write_bytes"]) == r["launches"]
        assert r["read_bytes"] == sum(r["launch_read_bytes"])
        assert r["write_bytes"] == sum(r["launch_write_bytes"])
        assert r["bytes_per_step"] == r["read_bytes"] + r["write_bytes"]
        assert re.fullmatch(r"[0-9a-f]{64}", r["sources_sha256"]), w
