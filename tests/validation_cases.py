"""Argument-validation cases for libccl.so, run by test_abi_host.py in a child
process with CUDA_VISIBLE_DEVICES="" (the pointers below are fake and are
never dereferenced: each call must be rejected before any launch)."""
import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import ring_allreduce_rank_gb300 as ccl  # noqa: E402


def _pp(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


FAKE = 0x7f0000000000  # never dereferenced: every call below fails validation first


def invalid_arguments(L):
    s = _pp([FAKE, FAKE + 4096])
    r = _pp([FAKE + 8192, FAKE + 12288])
    ok = ctypes.c_void_p(0)
    assert L.ccl_allreduce(s, r, 0, 16, 0, 0, 0, ok) == 1          # nranks < 1
    assert L.ccl_allreduce(s, r, 2000, 16, 0, 0, 0, ok) == 1       # nranks > max
    assert L.ccl_allreduce(s, r, 2, 16, 7, 0, 0, ok) == 1          # dtype
    assert L.ccl_allreduce(s, r, 2, 16, 0, 9, 0, ok) == 1          # op
    assert L.ccl_allreduce(s, r, 2, 16, 0, 0, 5, ok) == 1          # mode
    assert L.ccl_allreduce(None, r, 2, 16, 0, 0, 0, ok) == 1       # null array
    assert L.ccl_allreduce(_pp([FAKE, None]), r, 2, 16, 0, 0, 0, ok) == 1  # null rank pointer
    assert L.ccl_allreduce(s, r, 2, 1 << 62, 0, 0, 0, ok) == 1     # bytes overflow
    assert L.ccl_broadcast(s, r, 2, 2, 16, 0, 0, ok) == 1          # root out of range
    assert L.ccl_broadcast(s, r, 2, -1, 16, 0, 0, ok) == 1
    assert L.ccl_allreduce(s, r, 2, 0, 0, 0, 0, ok) == 0           # count 0: no-op


def overlaps(L):
    ok = ctypes.c_void_p(0)
    # two ranks' outputs overlap
    assert L.ccl_allreduce(_pp([FAKE, FAKE + 4096]), _pp([FAKE + 8192, FAKE + 8192 + 32]), 2, 16, 0, 0, 0, ok) == 3
    # an input partially overlaps another rank's output
    assert L.ccl_allreduce(_pp([FAKE + 8192 + 16, FAKE + 4096]), _pp([FAKE + 8192, FAKE + 12288]), 2, 16, 0, 0, 0,
                           ok) == 3
    # in place but shifted by one element
    assert L.ccl_allreduce(_pp([FAKE + 4, FAKE + 4096]), _pp([FAKE, FAKE + 4096]), 2, 16, 0, 0, 0, ok) == 3
    # all-to-all in place is not allowed
    assert L.ccl_alltoall(_pp([FAKE, FAKE + 4096]), _pp([FAKE, FAKE + 4096]), 2, 8, 0, 0, ok) == 3
    # reduce-scatter output inside the input but not at the chunk's offset
    assert L.ccl_reduce_scatter(_pp([FAKE, FAKE + 4096]), _pp([FAKE, FAKE + 4096 + 16]), 2, 16, 0, 0, 0, ok) == 3
    # bucket tensors overlapping each other
    nums = (ctypes.c_size_t * 2)(16, 16)
    assert L.ccl_bucket_allreduce(_pp([FAKE, FAKE + 32]), nums, 2, 1, 0, 0, 0, 0, ok) == 3


def host_allreduce(L):
    """ccl_allreduce_host: work buffer checks and overlaps, before any launch."""
    ok = ctypes.c_void_p(0)
    s, r = _pp([FAKE, FAKE + 4096]), _pp([FAKE + 8192, FAKE + 12288])
    W = FAKE + (1 << 30)
    need = 3 * 2 * 256 * 4  # three stages of 256 fp32 elements per rank
    f = L.ccl_allreduce_host
    assert f(s, r, 2, 16, 0, 0, None, need, ok) == 1              # no work buffer
    assert f(s, r, 2, 16, 0, 0, ctypes.c_void_p(W + 8), need, ok) == 1  # misaligned
    assert f(s, r, 2, 16, 0, 0, ctypes.c_void_p(W), need - 1, ok) == 1  # too small for one unit
    assert f(s, r, 2, 16, 7, 0, ctypes.c_void_p(W), need, ok) == 1      # dtype
    assert f(s, r, 0, 16, 0, 0, ctypes.c_void_p(W), need, ok) == 1      # nranks
    assert f(s, r, 2, 1 << 62, 0, 0, ctypes.c_void_p(W), need, ok) == 1  # bytes overflow
    # the work buffer overlaps an output, or an input
    assert f(s, r, 2, 16, 0, 0, ctypes.c_void_p(FAKE + 12288), need, ok) == 3
    assert f(s, r, 2, 16, 0, 0, ctypes.c_void_p(FAKE), need, ok) == 3
    # two outputs overlap
    assert f(s, _pp([FAKE + 8192, FAKE + 8192 + 32]), 2, 16, 0, 0, ctypes.c_void_p(W), need, ok) == 3
    assert f(s, r, 2, 0, 0, 0, None, 0, ok) == 0                   # count 0: no-op, nothing checked further


def traced_rejections(L):
    """Rejected calls are traced with their status; nothing is launched."""
    ccl.ccl_trace_clear()
    ccl.ccl_set_trace(True)
    s = _pp([FAKE, FAKE + 4096])
    assert L.ccl_allreduce(s, s, 0, 16, 0, 0, 0, ctypes.c_void_p(0)) == 1
    assert L.ccl_broadcast(s, s, 2, 5, 16, 1, 0, ctypes.c_void_p(0)) == 1
    recs = ccl.ccl_trace_read()
    assert [r["collective"] for r in recs] == ["allreduce", "broadcast"]
    assert [r["status"] for r in recs] == [1, 1] and all(r["launches"] == 0 for r in recs)
    assert recs[0]["count"] == 16 and recs[1]["dtype"] == 1
    ccl.ccl_set_trace(False)
    assert L.ccl_allreduce(s, s, 0, 16, 0, 0, 0, ctypes.c_void_p(0)) == 1
    assert len(ccl.ccl_trace_read()) == 2


if __name__ == "__main__":
    assert os.environ.get("CUDA_VISIBLE_DEVICES") == "", "run with CUDA_VISIBLE_DEVICES=''"
    L = ccl.lib()
    invalid_arguments(L)
    overlaps(L)
    host_allreduce(L)
    traced_rejections(L)
    print("validation cases ok")
