"""The committed ncu summaries under profiles/: every ncu command they give
keeps the GPU's clocks as they are (--clock-control none); a full capture
names one kernel (-k) and at most three launches (-c); every summary the
benchmark reads carries its machine-read traffic and source-digest lines;
and no summary refers to scratch files or to paths of one machine.  A
summary whose digest no longer matches the kernel's sources is reported
(its traffic then reads as null in the benchmark line), not failed."""
import glob
import os
import re
import warnings

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MDS = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _ncu_commands(text):
    """ncu command lines, joined across backslash continuations."""
    cmds, cur = [], None
    for line in text.splitlines():
        s = line.strip()
        if cur is not None:
            cur += " " + s.rstrip("\\").strip()
            if not s.endswith("\\"):
                cmds.append(cur)
                cur = None
        elif re.match(r"^(\S+\s+[&|]+\s+)?ncu\s", s) or s.startswith("ncu "):
            cur = s.rstrip("\\").strip()
            if not s.endswith("\\"):
                cmds.append(cur)
                cur = None
    return cmds


def test_there_are_profiles():
    assert MDS, "no ncu summaries committed"


@pytest.mark.parametrize("md", MDS, ids=[os.path.basename(m) for m in MDS])
def test_ncu_commands_keep_clocks_and_stay_small(md):
    text = open(md).read()
    for cmd in _ncu_commands(text):
        assert "--clock-control none" in cmd, f"{os.path.basename(md)}: {cmd}"
        if "--set full" in cmd or "--section" in cmd:
            assert re.search(r"\s-k\s", cmd), f"full capture without -k: {cmd}"
            m = re.search(r"\s-c\s+(\d+)", cmd)
            assert m and int(m.group(1)) <= 3, f"full capture of more than 3 launches: {cmd}"


@pytest.mark.parametrize("md", MDS, ids=[os.path.basename(m) for m in MDS])
def test_no_scratch_or_machine_paths(md):
    text = open(md).read()
    assert "_work/" not in text
    assert "/root/" not in text


@pytest.mark.parametrize("workload", list(bench.PROFILES))
def test_benchmark_summaries_carry_machine_read_lines(workload):
    md, files = bench.PROFILES[workload]
    text = open(os.path.join(ROOT, "profiles", md)).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    assert m and int(m.group(1)) > 0, md
    assert s, md
    if s.group(1) != bench.source_digest(files):
        warnings.warn(f"{md}: kernel sources changed since the capture; its traffic reads as null")
