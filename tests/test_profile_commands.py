"""The commands recorded in profiles/ still run against the current code: every
`python bench.py ...` and `python -m quantized_moe_noaux_b300.profile_run ...` line parses
with the tools' own argument parsers, and the workloads and layers it names exist. Nothing
is executed (CPU)."""

import glob
import os
import re
import shlex
import sys

import pytest

import bench
from quantized_moe_noaux_b300 import profile_run
from synth import LAYERS, WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands():
    found = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for line in text.splitlines():
            for m in re.finditer(r"python (bench\.py|-m quantized_moe_noaux_b300\.profile_run)((?: +--?[\w-]+(?: +[\w.]+)?)*)", line):
                found.append((os.path.basename(path), m.group(1), shlex.split(m.group(2))))
    return found


COMMANDS = _commands()


def test_profiles_record_commands():
    assert len({name for name, _, _ in COMMANDS}) >= 5, COMMANDS


@pytest.mark.parametrize("name,tool,argv", COMMANDS, ids=[f"{n}:{i}" for i, (n, _, _) in enumerate(COMMANDS)])
def test_recorded_command_parses(name, tool, argv, monkeypatch):
    if tool == "bench.py":
        monkeypatch.setattr(sys, "argv", ["bench.py"] + argv)
        args = bench.parse()
        assert args.workload in WORKLOADS, (name, args.workload)
    else:
        args = profile_run.parser().parse_args(argv)
        assert args.layer in LAYERS, (name, args.layer)
