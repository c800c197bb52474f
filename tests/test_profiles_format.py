"""The ncu summaries under profiles/ are short text named for an operation and
a workload that exist (besides the compiler's resource summary of every
kernel), each giving its kernel, the source hash it was taken
on and the DRAM bytes per launch the bench line reads, and the full commands
that made it: commands that run committed files only, with every ncu call
leaving the GPU clocks alone (--clock-control none)."""
import glob
import os
import re

import pytest

from numerically_stable_online_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))
OPS = set(wl.OPS) | {"attention"}
NAMES = set(wl.WORKLOADS) | set(wl.ATTN_WORKLOADS)


def test_profiles_exist_for_the_bench_workload():
    names = {os.path.basename(f) for f in FILES}
    assert f"softmax_{wl.BENCH_WORKLOAD}.md" in names
    assert "attention_attn_bf16_4x32x4096x128.md" in names


NCU_FILES = [f for f in FILES if not os.path.basename(f).startswith("resources_")]
RESOURCE_FILES = [f for f in FILES if os.path.basename(f).startswith("resources_")]


@pytest.mark.parametrize("path", RESOURCE_FILES, ids=[os.path.basename(f) for f in RESOURCE_FILES])
def test_resource_summary(path):
    """The ptxas summary: the compile commands of committed sources with -Xptxas -v."""
    text = open(path).read()
    assert os.path.getsize(path) < 16 * 1024
    cmds = [line.strip() for line in text.splitlines() if line.startswith("    nvcc ")]
    assert cmds
    for c in cmds:
        assert "-Xptxas -v" in c and "arch=compute_103a,code=sm_103a" in c, c
        src = c.split(" -c ")[1].split()[0]
        assert os.path.exists(os.path.join(ROOT, src)), src


@pytest.mark.parametrize("path", NCU_FILES, ids=[os.path.basename(f) for f in NCU_FILES])
def test_profile_summary(path):
    base = os.path.basename(path)
    assert base.endswith((".md", ".txt")), "text summaries only"
    assert os.path.getsize(path) < 16 * 1024, "a short summary"
    stem = base.rsplit(".", 1)[0]
    op = next((o for o in sorted(OPS, key=len, reverse=True) if stem.startswith(o + "_")), None)
    assert op is not None and stem[len(op) + 1:] in NAMES, f"{base}: not <op>_<workload>"
    text = open(path).read()
    assert re.search(r"^kernel: \S+", text, re.M)
    assert re.search(r"^source_hash: [0-9a-f]{16}$", text, re.M)
    assert re.search(r"^dram_bytes_per_launch: [0-9]+$", text, re.M)
    cmds = [line.strip() for line in text.splitlines() if line.startswith("    ")]
    ncu = [c for c in cmds if c.startswith("ncu ")]
    assert ncu, "the ncu commands are given"
    for c in ncu:
        assert "--clock-control none" in c, c
    for c in cmds:
        if c.startswith(("python ", "ncu ")):
            assert "_work" not in c and os.path.dirname(ROOT) + os.sep not in c, c
            assert "bench.py" in c, c
