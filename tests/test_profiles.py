"""The ncu summaries under profiles/ must be reproducible from committed files:
every quoted command runs a script of the repository (never a working file),
with arguments bench.py accepts and a workload it knows, and every ncu command
leaves the GPU clocks alone (--clock-control none). The recorded kernel traffic
points at a committed capture."""
import glob
import json
import os
import re
import shlex
import sys
from unittest import mock

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _commands(text):
    """Indented command blocks (backslash continuations joined)."""
    out, cur = [], ""
    for line in text.splitlines():
        if not line.startswith("    "):
            if cur:
                out.append(cur)
                cur = ""
            continue
        cur += line.strip().rstrip("\\") + " "
        if not line.rstrip().endswith("\\"):
            out.append(cur)
            cur = ""
    if cur:
        out.append(cur)
    return [c.strip() for c in out if c.strip()]


def test_profiles_present():
    assert PROFILES, "no ncu summaries under profiles/"


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_commands_run_committed_files(path):
    text = open(path).read()
    assert "_work/" not in text, "a profile names a working file"
    cmds = _commands(text)
    assert cmds, "a profile must give the command that made it"
    import bench
    for c in cmds:
        if c.startswith("ncu "):
            assert "--clock-control none" in c, f"ncu without --clock-control none: {c}"
        m = re.search(r"\bpython3? (\S+\.py)(.*)$", c)
        if not m:
            continue
        script, args = m.group(1), m.group(2)
        assert not script.startswith("_work"), script
        assert os.path.exists(os.path.join(ROOT, script)), f"{script} is not in the repository"
        if script == "bench.py":
            argv = [a for a in shlex.split(args.replace("<workload>", "rope_qkv_4096"))]
            with mock.patch.object(sys, "argv", ["bench.py", *argv]):
                a = bench.parse()
            if a.only is not None:
                assert a.only in bench.SUITE_WORKLOADS, a.only


def test_recorded_traffic_points_at_a_capture():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    for kernel, d in rec.items():
        assert os.path.exists(os.path.join(ROOT, d["capture"])), kernel
        assert d["dram_bytes_per_launch"] == pytest.approx(d["dram_read_bytes"] + d["dram_write_bytes"])
        assert re.fullmatch(r"[0-9a-f]{16}", d["src_hash"])
