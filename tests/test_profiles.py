"""The ncu summaries under profiles/ stay runnable: every bench.py command
they quote parses with bench.py's own options, every profile that
profiles/traffic.txt names exists, and every traffic entry's kernel family is
one bench.py knows."""
import os
import re
import shlex

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _bench_commands(text):
    """bench.py argument lists of the fenced commands (continuation lines
    joined)."""
    cmds = []
    for block in re.findall(r"```\n(.*?)```", text, re.S):
        joined = block.replace("\\\n", " ")
        for line in joined.splitlines():
            words = shlex.split(line)
            if "bench.py" in words:
                cmds.append(words[words.index("bench.py") + 1:])
    return cmds


@pytest.mark.parametrize("name", _summaries())
def test_summary_commands_parse(name):
    text = open(os.path.join(PROFILES, name)).read()
    cmds = _bench_commands(text)
    assert cmds, "%s quotes no bench.py command" % name
    parser = bench.make_parser()
    for args in cmds:
        ns = parser.parse_args(args)
        assert ns.warmup >= 3, (name, args)
    # the capture itself is made without clock control
    for block in re.findall(r"```\n(.*?)```", text, re.S):
        if "ncu " in block:
            assert "--clock-control none" in block, name


def test_traffic_entries_point_at_profiles():
    lines = open(os.path.join(PROFILES, "traffic.txt")).read().splitlines()
    entries = [ln.split() for ln in lines if ln and not ln.startswith("#")]
    assert entries
    for key, nbytes, digest in entries:
        assert int(nbytes) > 0 and len(digest) == 16
        assert bench.kernel_source_digest(key) != "unknown", key
    for ln in lines:
        for ref in re.findall(r"profiles/([\w.]+\.md)", ln):
            assert os.path.exists(os.path.join(PROFILES, ref)), ref
