"""ccl_reduce_scatter_step_static: the step-by-step ReduceScatter whose working
space is a fixed array in device memory, for callers that cannot let the
library call cudaMalloc (a framework's caching pool already holds the GPU's
memory, or an allocation's implicit device synchronisation would stall other
streams).

Called through the C ABI and checked bit for bit (the collectives' tolerance)
against the existing ccl_reduce_scatter on two calls in a row.  The second call
is smaller, so stale data from the first is still in the shared array.  This
file is collected last and runs the same alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 * 1024 * 1024  # CCL_STATIC_SCRATCH_BYTES in include/ccl.h


def _entry():
    L = ccl.lib()
    fn = L.ccl_reduce_scatter_step_static
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, pp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _run_both(fn, x, dtype, op):
    N, K = x.shape
    if dtype == torch.bfloat16:
        send = [torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).cuda() for r in x]
    else:
        send = [torch.from_numpy(r).cuda() for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    got = [torch.full((ln[r],), 7, dtype=dtype, device="cuda") for r in range(N)]
    ref_step = [torch.empty(ln[r], dtype=dtype, device="cuda") for r in range(N)]
    ref_fused = [torch.empty(ln[r], dtype=dtype, device="cuda") for r in range(N)]
    stream = torch.cuda.current_stream()
    opc = ccl.ccl.OPS[op]
    dtc = 1 if dtype == torch.bfloat16 else 0
    rc = fn(_ptrs(send), _ptrs(got), N, K, dtc, opc, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, ccl.ccl_status_string(rc)
    ccl.ccl_reduce_scatter(send, ref_step, op=op, mode="step")
    ccl.ccl_reduce_scatter(send, ref_fused, op=op, mode="fused")
    torch.cuda.synchronize()
    for r in range(N):
        np.testing.assert_array_equal(_bits(got[r]), _bits(ref_step[r]))
        np.testing.assert_array_equal(_bits(got[r]), _bits(ref_fused[r]))


def test_static_scratch_reduce_scatter_two_calls_match_existing_entry():
    assert torch.cuda.is_available()
    fn = _entry()
    # first call: N=8 bf16 AVG, 1 Mi elements per rank (16 MiB of working space)
    _run_both(fn, W.normal_bf16(8, 1 << 20, std=1e-3, seed_base=0), torch.bfloat16, "avg")
    # second call in a row: smaller, different dtype, op and rank count (ragged)
    _run_both(fn, W.mixed_fp32(5, 100_003, seed_base=9), torch.float32, "sum")


def test_static_scratch_rejects_sizes_beyond_the_array():
    fn = _entry()
    N = 8
    K = STATIC_SCRATCH_BYTES // N // 2 + 1  # one bf16 element more than fits per rank
    send = [torch.zeros(K, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    _, ln = ccl.ccl_plan_chunks(K, N)
    out = [torch.zeros(ln[r], dtype=torch.bfloat16, device="cuda") for r in range(N)]
    rc = fn(_ptrs(send), _ptrs(out), N, K, 1, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1  # CCL_ERR_INVALID_ARG, nothing enqueued
    torch.cuda.synchronize()
    assert all(int(o.abs().sum()) == 0 for o in out)
