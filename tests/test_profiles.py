"""The committed ncu summaries: each names its kernel, its sources, its
workload and the command that made it, and every ncu command in them leaves
the GPU clocks alone. (Whether a summary still matches the sources is
decided at run time by the bench, from the recorded source hash.)"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def fields(text):
    out = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            out.setdefault(k.strip(), v.strip().strip("`"))
    return out


def ncu_commands(text):
    """Every ncu invocation in the text, with its continuation lines joined."""
    joined = re.sub(r"\\\n\s*", " ", text)
    return [m.group(0) for m in re.finditer(r"(?m)^\s*ncu (?!-i ).*$", joined)]


def test_there_are_summaries():
    assert "gla_fwd_full.md" in SUMMARIES and "bench_launch_list.md" in SUMMARIES


@pytest.mark.parametrize("name", SUMMARIES)
def test_every_ncu_command_leaves_the_clocks_alone(name):
    text = open(os.path.join(PROFILES, name)).read()
    cmds = ncu_commands(text)
    assert cmds, f"{name}: no ncu command recorded"
    for c in cmds:
        assert "--clock-control none" in c, f"{name}: {c}"


@pytest.mark.parametrize("name", [n for n in SUMMARIES if n != "bench_launch_list.md"])
def test_kernel_summary_fields(name):
    f = fields(open(os.path.join(PROFILES, name)).read())
    for key in ("kernel", "source_files", "source_sha256_16", "workload", "traffic_bytes_per_launch",
                "algorithmic_bytes_per_launch"):
        assert key in f, f"{name}: no {key}"
    for src in f["source_files"].split(","):
        assert os.path.exists(os.path.join(ROOT, src.strip())), f"{name}: {src.strip()} is missing"
    assert re.fullmatch(r"[0-9a-f]{16}", f["source_sha256_16"]), name
    assert float(f["traffic_bytes_per_launch"]) > 0
    assert int(f["algorithmic_bytes_per_launch"].split()[0]) > 0
