"""Child process of tests/test_gpu_debug_bounds.py: runs GPU test files in
this process against the library named by CCL_LIBRARY (the bounds-checking
debug build), then prints how many kernel accesses fell outside the calls'
own buffers.  Usage: python debug_bounds_run.py <pytest arguments>"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

if __name__ == "__main__":
    rc = pytest.main(sys.argv[1:])
    import ring_allreduce_rank_gb300 as ccl
    faults, first = ccl.ccl_debug_faults()
    print("DEBUG_FAULTS %d first 0x%x" % (faults, first))
    sys.exit(int(rc))
