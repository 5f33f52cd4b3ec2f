"""The documents stay true to the tree (no GPU): every source, test or fixture
file that README.md or a profile summary names exists, and every
command in a profile summary runs committed files with options and workloads
that bench.py accepts."""
import glob
import os
import re
import shlex

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEARCH = ["", "ring_allreduce_rank_gb300", "tests", "tests/golden", "include", "oracle", "profiles"]
DOCS = ["DESIGN.md", "README.md"] + sorted(os.path.relpath(p, ROOT) for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _named_files(text):
    # file names in backticks; JSON keys such as roofline.traffic are not files
    toks = set(re.findall(r"`([A-Za-z0-9_./-]+\.(?:cu|cuh|h|py|c|md|json|traffic))`", text))
    return sorted(t for t in toks if not t.startswith("roofline."))


@pytest.mark.parametrize("doc", DOCS)
def test_named_files_exist(doc):
    text = open(os.path.join(ROOT, doc)).read()
    missing = [t for t in _named_files(text)
               if not any(os.path.exists(os.path.join(ROOT, d, t)) for d in SEARCH)]
    assert not missing, "%s names files that do not exist: %s" % (doc, missing)


def _bench_commands(text):
    """`python bench.py ...` invocations in a summary (continuation lines joined)."""
    text = text.replace("\\\n", " ")
    return [m.group(0) for m in re.finditer(r"python bench\.py[^\n>&|]*", text)]


def _bench_parser():
    import bench
    src = open(os.path.join(ROOT, "bench.py")).read()
    flags = set(re.findall(r'add_argument\("(--[a-z0-9-]+)"', src))
    return flags, set(bench.ROWS) | {"allreduce"}


@pytest.mark.parametrize("doc", [d for d in DOCS if d.startswith("profiles")])
def test_profile_commands_use_real_options(doc):
    text = open(os.path.join(ROOT, doc)).read()
    cmds = _bench_commands(text)
    assert cmds, "%s gives no bench.py command" % doc
    flags, workloads = _bench_parser()
    for cmd in cmds:
        args = shlex.split(cmd)[2:]
        for i, a in enumerate(args):
            if a.startswith("--"):
                assert a in flags, "%s: unknown option %s" % (doc, a)
            if a == "--workload":
                assert args[i + 1] in workloads, "%s: unknown workload %s" % (doc, args[i + 1])
    # the ncu line profiles the same command that first ran without it
    assert "--clock-control none" in text or "ncu" not in text
