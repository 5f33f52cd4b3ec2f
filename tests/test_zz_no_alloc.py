"""ccl_reduce_scatter_step_static: the step-by-step ReduceScatter whose working
space is a fixed array in device memory, for callers that cannot let the
library call cudaMalloc (a framework's caching pool already holds the GPU's
memory, or an allocation's implicit device synchronisation would stall other
streams).

Called through the C ABI and checked bit for bit (the collectives' tolerance)
against the CPU oracle's ReduceScatter and against the existing
ccl_reduce_scatter, on two calls in a row: the second call is smaller, so stale
data from the first is still in the shared array.  Also: the in-place form,
one rank, a ragged bf16 pre-multiplied AVG, the size limit, and -- in a fresh
process -- that the set-up call reserves the array and later calls change the
device's free memory by nothing.  This file is collected last and runs the
same alone in a fresh process."""
import ctypes
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 * 1024 * 1024  # CCL_STATIC_SCRATCH_BYTES in include/ccl.h
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _entry():
    fn = ccl.lib().ccl_reduce_scatter_step_static
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, pp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() if t is not None else None for t in ts])


def _call(fn, send, recv, K, dtype, op):
    stream = torch.cuda.current_stream()
    return fn(_ptrs(send), _ptrs(recv), len(send), K, 1 if dtype == torch.bfloat16 else 0, ccl.ccl.OPS[op],
              ctypes.c_void_p(stream.cuda_stream))


def _run_both(fn, x, op):
    """The static entry against the oracle and against ccl_reduce_scatter in
    step and fused mode, out of place."""
    N, K = x.shape
    send = [to_dev(r) for r in x]
    dtype = send[0].dtype
    _, ln = ccl.ccl_plan_chunks(K, N)
    got = [torch.full((ln[r],), 7, dtype=dtype, device="cuda") for r in range(N)]
    ref_step = [torch.empty(ln[r], dtype=dtype, device="cuda") for r in range(N)]
    ref_fused = [torch.empty(ln[r], dtype=dtype, device="cuda") for r in range(N)]
    rc = _call(fn, send, got, K, dtype, op)
    assert rc == 0, ccl.ccl_status_string(rc)
    ccl.ccl_reduce_scatter(send, ref_step, op=op, mode="step")
    ccl.ccl_reduce_scatter(send, ref_fused, op=op, mode="fused")
    torch.cuda.synchronize()
    want = oracle.reduce_scatter(list(x), op)
    for r in range(N):
        g = bits(got[r])
        assert_bits_equal(g, want[r], "static vs oracle, rank %d" % r)
        assert_bits_equal(g, bits(ref_step[r]), "static vs step mode, rank %d" % r)
        assert_bits_equal(g, bits(ref_fused[r]), "static vs fused mode, rank %d" % r)


def test_static_scratch_reduce_scatter_two_calls_match_oracle_and_existing_entry():
    fn = _entry()
    # first call: N=8 bf16 AVG, 1 Mi elements per rank (16 MiB of working space)
    _run_both(fn, W.normal_bf16(8, 1 << 20, std=1e-3, seed_base=0), "avg")
    # second call in a row: smaller, different dtype, op and rank count (ragged)
    _run_both(fn, W.mixed_fp32(5, 100_003, seed_base=9), "sum")


def test_static_scratch_bf16_ragged_avg_premul():
    _run_both(_entry(), W.mixed_bf16(7, 7 * 3001 + 5, seed_base=21), "avg_premul")


@pytest.mark.parametrize("op", ["sum", "avg", "avg_premul", "max"])
def test_static_scratch_one_rank(op):
    """N = 1: the rank's whole buffer is its chunk; AVG and the pre-multiplied
    AVG still divide (or scale) once, which canonicalises NaNs."""
    _run_both(_entry(), W.mixed_fp32(1, 4099, seed_base=33), op)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_static_scratch_in_place(dtype):
    """recv[i] is rank i's own chunk i inside send[i] (the in-place form the
    header allows): the chunk is overwritten with the reduction, bit for bit
    the oracle's, and the rest of each input is untouched."""
    fn = _entry()
    N, K = 6, 6 * 20011 + 4
    x = W.mixed_fp32(N, K, seed_base=41) if dtype == "fp32" else W.mixed_bf16(N, K, seed_base=41)
    off, ln = ccl.ccl_plan_chunks(K, N)
    send = [to_dev(r) for r in x]
    recv = [send[i][off[i]:off[i] + ln[i]] for i in range(N)]
    rc = _call(fn, send, recv, K, send[0].dtype, "sum")
    assert rc == 0, ccl.ccl_status_string(rc)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter(list(x), "sum")
    for i in range(N):
        b = bits(send[i])
        assert_bits_equal(b[off[i]:off[i] + ln[i]], want[i], "in place, chunk %d" % i)
        rest = np.concatenate([b[:off[i]], b[off[i] + ln[i]:]])
        xi = x[i].view(np.uint32) if dtype == "fp32" else x[i]
        assert_bits_equal(rest, np.concatenate([xi[:off[i]], xi[off[i] + ln[i]:]]), "in place, rest of rank %d" % i)


def test_static_scratch_rejects_sizes_beyond_the_array():
    fn = _entry()
    N = 8
    K = STATIC_SCRATCH_BYTES // N // 2 + 1  # one bf16 element more than fits per rank
    send = [torch.zeros(K, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    _, ln = ccl.ccl_plan_chunks(K, N)
    out = [torch.zeros(ln[r], dtype=torch.bfloat16, device="cuda") for r in range(N)]
    assert _call(fn, send, out, K, torch.bfloat16, "sum") == 1  # CCL_ERR_INVALID_ARG, nothing enqueued
    torch.cuda.synchronize()
    assert all(int(o.abs().sum()) == 0 for o in out)
    # the largest call that fits is accepted
    K = STATIC_SCRATCH_BYTES // N // 2
    send = [torch.ones(K, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    _, ln = ccl.ccl_plan_chunks(K, N)
    out = [torch.zeros(ln[r], dtype=torch.bfloat16, device="cuda") for r in range(N)]
    assert _call(fn, send, out, K, torch.bfloat16, "sum") == 0
    torch.cuda.synchronize()
    assert all(bool((o.float() == N).all()) for o in out)


_CHILD = textwrap.dedent(r"""
    import ctypes, json, sys
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    import ring_allreduce_rank_gb300 as ccl
    from ring_allreduce_rank_gb300 import workloads as W

    torch.cuda.set_device(0)
    N, K = 8, 1 << 20
    x = W.normal_bf16(N, K, std=1e-3, seed_base=0)
    send = [torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).cuda() for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    outs = [[torch.empty(ln[r], dtype=torch.bfloat16, device="cuda") for r in range(N)] for _ in range(2)]
    torch.cuda.synchronize()
    fn = ccl.lib().ccl_reduce_scatter_step_static
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, pp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    P = lambda ts: (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    free = [torch.cuda.mem_get_info()[0]]
    rcs = [fn(P(send), P(outs[0]), N, 0, 1, 1, st)]          # set-up call: count = 0
    torch.cuda.synchronize(); free.append(torch.cuda.mem_get_info()[0])
    for o in outs:                                           # two real calls
        rcs.append(fn(P(send), P(o), N, K, 1, 1, st))
        torch.cuda.synchronize(); free.append(torch.cuda.mem_get_info()[0])
    same = all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(*outs))
    print(json.dumps({"free": free, "rcs": rcs, "same": same}))
""")


def test_static_scratch_setup_reserves_the_array_and_calls_allocate_nothing():
    """In a fresh process under CUDA's default (lazy) module loading: the
    count = 0 set-up call is when the 32 MiB array is reserved, and the two
    AllReduce-sized calls after it leave the device's free memory unchanged
    (no cudaMalloc, no workspace, no kernel loading)."""
    env = dict(os.environ)
    env.pop("CUDA_MODULE_LOADING", None)
    res = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0, res.stderr[-3000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["rcs"] == [0, 0, 0], out
    assert out["same"], out
    f0, f1, f2, f3 = out["free"]
    assert f0 - f1 >= STATIC_SCRATCH_BYTES, out  # reserved by the set-up call
    assert f1 == f2 == f3, out                   # nothing allocated by the calls
