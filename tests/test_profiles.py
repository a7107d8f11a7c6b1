"""The committed ncu summaries under profiles/ describe the kernel sources as
they are now.  Each summary names the source hash (bench.py's
source_hash: SHA-256 over the kernel's .cu, the PTX helpers, the parameter
structs and the host code that orders its work units) it was taken on; an
edit of those sources without a new capture fails here.  Every ncu command
a summary records leaves the GPU clocks alone (--clock-control none), and
the two traffic summaries give bench.py a DRAM figure for its roofline."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROF = os.path.join(ROOT, "profiles")
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SUMMARIES = sorted(f for f in os.listdir(PROF) if f.endswith(".md"))


def _read(name):
    with open(os.path.join(PROF, name)) as f:
        return f.read()


def _hashes(name, text):
    """kernel -> source hash named by the summary."""
    if name.startswith("step_launches"):
        m = re.search(r"backward source_sha256_16 ([0-9a-f]{16}), forward\s+([0-9a-f]{16})", text)
        assert m, f"{name}: no backward/forward source hashes"
        return {"attn_bwd_kernel": m.group(1), "attn_fwd_kernel": m.group(2)}
    kernel = next(k for k in bench.KERNEL_SOURCES if name.startswith(k))
    found = set(re.findall(r"source_sha256_16:?\s+([0-9a-f]{16})", text))
    assert len(found) == 1, f"{name}: expected one source hash, found {found}"
    return {kernel: found.pop()}


def _ncu_commands(text):
    """The ncu command lines of the summary's code blocks, with backslash
    continuations joined."""
    cmds, blocks = [], re.findall(r"```(.*?)```", text, flags=re.S)
    for block in blocks:
        joined = re.sub(r"\\\n\s*", " ", block)
        cmds += [ln.strip() for ln in joined.splitlines() if ln.strip().startswith("ncu ")]
    return cmds


def test_every_kernel_has_summaries():
    names = " ".join(SUMMARIES)
    for kernel in bench.KERNEL_SOURCES:
        assert f"{kernel}_llama7b_32k_full.md" in names
        assert f"{kernel}_llama7b_128k_traffic.md" in names
    assert "step_launches_llama7b_128k.md" in names


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_was_taken_on_the_current_sources(name):
    for kernel, h in _hashes(name, _read(name)).items():
        assert h == bench.source_hash(kernel), (
            f"{name} describes {kernel} at {h}; the sources are now at "
            f"{bench.source_hash(kernel)}: capture it again")


@pytest.mark.parametrize("name", SUMMARIES)
def test_recorded_ncu_commands_leave_clocks_alone(name):
    cmds = _ncu_commands(_read(name))
    assert cmds, f"{name}: no ncu command recorded"
    for c in cmds:
        if c.startswith("ncu -i "):
            continue  # reading a saved report runs nothing on a GPU
        assert "--clock-control none" in c, f"{name}: {c}"


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SOURCES))
def test_traffic_summary_feeds_the_roofline(kernel):
    t = bench.kernel_traffic(f"{kernel}_llama7b_128k_traffic.md", kernel)
    assert isinstance(t, int) and t > 0
