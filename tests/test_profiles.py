"""The committed profile summaries are self-consistent: each names the full
command that produced it (an ncu run with clocks left alone, over a bench.py
case that exists, or the verbose library build for the ptxas resource
summary), and each traffic record belongs to a summary. CPU only."""
import json
import os
import re

import pytest

import qmm_synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _commands(text):
    blocks = re.findall(r"```\n(.*?)```", text, re.S)
    return [l.strip() for b in blocks for l in b.splitlines()
            if l.strip().startswith(("ncu ", "python "))]


def _case_exists(name):
    if name.endswith("_backward_input"):
        return name[:-len("_backward_input")] in qmm_synth.WORKLOADS
    if name.startswith("q4_k_prefill"):
        return re.fullmatch(r"q4_k_prefill(_N\d+)?(_gemv)?", name) is not None
    m = re.fullmatch(r"(\w+?)_(swiglu|geglu)_pair(_N\d+)?", name)
    if m:
        return (m.group(1) + "_gemv") in qmm_synth.WORKLOADS
    m = re.fullmatch(r"(\w+_experts)_pos\d+(_gemv|_grouped)?", name)
    if m:
        return m.group(1) in qmm_synth.EXPERT_WORKLOADS
    return name in qmm_synth.WORKLOADS or name in qmm_synth.AFFINE_WORKLOADS


def test_there_are_summaries():
    assert SUMMARIES


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_gives_its_command(name):
    text = open(os.path.join(PROFILES, name)).read()
    cmds = _commands(text)
    assert cmds, f"{name}: no command"
    for c in cmds:
        if not c.startswith("ncu "):
            # a build-log summary: it rebuilds from the committed sources
            assert "build_lib.build(" in c and "verbose=True" in c, c
            continue
        assert "--clock-control none" in c, c
        assert " python bench.py" in c, c
        m = re.search(r"--case (\S+)", c)
        if m:
            assert _case_exists(m.group(1)), c
        if "--set full" in c or "--section" in c:
            # a multi-pass capture: one kernel, a few launches
            assert re.search(r"-k regex:\S+", c) and re.search(r"-c [1-3]\b", c), c
    assert len(text.encode()) < 16 * 1024  # a short summary, not raw output


def test_traffic_records_belong_to_summaries():
    with open(os.path.join(PROFILES, "traffic.json")) as f:
        rec = json.load(f)
    for key, r in rec.items():
        assert os.path.exists(os.path.join(PROFILES, key + ".md")), key
        assert re.fullmatch(r"[0-9a-f]{16}", r["source_hash"]), key
        assert r["dram_bytes_per_launch"] > 0 and r["workload"]


def test_only_text_under_profiles():
    for f in os.listdir(PROFILES):
        assert f.endswith((".md", ".txt", ".json")), f
