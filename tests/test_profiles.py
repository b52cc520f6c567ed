"""The committed ncu summaries: each names the command that made it, and that
command runs committed files only; the traffic table carries, per workload,
the kernel, the source hash it was taken on and bytes per launch."""
from __future__ import annotations

import glob
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def test_every_summary_names_its_command():
    files = sorted(glob.glob(os.path.join(PROFILES, "*.md")))
    assert files
    for f in files:
        text = open(f).read()
        assert re.search(r"^(ncu |python )", text, re.M), f"{f}: no command line"
        assert "_work" not in text and "/root/" not in text, f"{f}: names an uncommitted or machine path"
        for script in re.findall(r"python\s+(\S+\.py)", text):
            assert os.path.exists(os.path.join(ROOT, script)), f"{f}: {script} is not in the repository"


def test_traffic_table():
    t = json.load(open(os.path.join(PROFILES, "ncu_traffic.json")))
    workloads = {k: v for k, v in t.items() if not k.startswith("_")}
    assert workloads
    for name, v in workloads.items():
        assert re.fullmatch(r"[0-9a-f]{16}", v["source_hash"]), name
        assert v["dram_bytes_per_launch"] > 0 and v["kernel"], name
    # the bench reports a workload's traffic only while the sources match
    cur = bench.kernel_source_hash()
    for name, v in workloads.items():
        assert (bench.ncu_traffic(name) is not None) == (v["source_hash"] == cur), name


def test_source_hash_ignores_comments_only():
    import bench

    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x // y /* z */"; char q = \'"\'; int b;\n'
    assert bench.strip_comments(src) == 'int a = 1;\n const char* s = "x // y /* z */"; char q = \'"\'; int b;'
    # a comment growing by a line is no change either
    assert bench.strip_comments(src.replace("// note", "// note\n// more")) == bench.strip_comments(src)
    # an edit to code is a change, an edit to a comment is not
    assert bench.strip_comments(src.replace("note", "other note")) == bench.strip_comments(src)
    assert bench.strip_comments(src.replace("int b", "int c")) != bench.strip_comments(src)
