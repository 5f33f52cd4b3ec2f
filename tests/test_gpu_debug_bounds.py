"""Memory safety without compute-sanitizer: the GPU parity tests run again
against the bounds-checking debug build (libccl_debug.so, CCL_DEBUG_BOUNDS).
There every global load and store of every kernel is checked against the byte
ranges of the calling collective's own buffers (workspace and counters
included); an access outside them is counted and skipped, never performed.
The parity tests must still pass and no access may fall outside.  A control
run registers only the first half of every range and must see the checker
count the other half's accesses."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RUNNER = os.path.join(ROOT, "tests", "debug_bounds_run.py")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# every GPU test file that exercises the collectives at small sizes; not the
# full-size files (the debug check scans the range table on every access),
# not CUDA-graph capture (the range table is uploaded with a copy per call),
# not the C example (it links the release library)
FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_small_chunks.py", "tests/test_gpu_orders.py",
         "tests/test_gpu_compressed.py", "tests/test_gpu_host.py", "tests/test_gpu_checks.py",
         "tests/test_gpu_premul.py", "tests/test_gpu_topk.py", "tests/test_zz_no_alloc.py"]


@pytest.fixture(scope="module")
def debug_lib():
    from ring_allreduce_rank_gb300 import build
    return build.build(debug_bounds=True)


def _run(lib, args, extra_env=None):
    env = dict(os.environ, CCL_LIBRARY=lib, **(extra_env or {}))
    res = subprocess.run([sys.executable, RUNNER, "-q", "-x", "-p", "no:cacheprovider", *args], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=3000)
    line = [l for l in res.stdout.splitlines() if l.startswith("DEBUG_FAULTS")]
    return res, (int(line[-1].split()[1]) if line else None)


def test_every_kernel_access_stays_inside_the_calls_buffers(debug_lib):
    res, faults = _run(debug_lib, ["-m", "gpu and not slow", "-k", "not 1024 and not graph_capture", *FILES])
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    assert faults == 0, res.stdout[-2000:]


def test_the_checker_counts_accesses_outside_the_registered_ranges(debug_lib):
    res, faults = _run(debug_lib, ["-m", "gpu", "tests/test_gpu_parity.py::test_allreduce_count_zero_and_single_rank",
                                   "tests/test_gpu_checks.py::test_check_identical_counts_planted_differences"],
                       {"CCL_DEBUG_SHRINK": "1"})
    assert faults is not None and faults > 0, res.stdout[-2000:] + res.stderr[-2000:]
