"""Overlap and NULL-pointer validation of thirteen entry points over thousands
of random pointer layouts (no GPU): the cases run in a child process that sees
no device (tests/validation_fuzz.py), where every call the library accepts can
only fail its launch."""
import os
import subprocess
import sys

import pytest


@pytest.fixture(scope="module", autouse=True)
def _built():
    from ring_allreduce_rank_gb300 import build
    build.build()


def test_overlap_rules_match_the_header_contract():
    here = os.path.dirname(os.path.abspath(__file__))
    env = {k: v for k, v in os.environ.items() if not k.startswith("CCL_")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.join(here, "validation_fuzz.py")], env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-3000:]
    assert "validation fuzz ok" in res.stdout
