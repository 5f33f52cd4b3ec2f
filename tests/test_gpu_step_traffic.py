"""Per-rank traffic of the step-by-step mode on the device (Lesson 3's
self-check: every rank counts the elements it sends, and an AllReduce sends
2(N-1)K/N per rank when N divides K).  The counts the library keeps for its
ring-step launches must equal the oracle's own step simulation, and the
oracle's schedule table for ReduceScatter and AllGather."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import to_dev

pytestmark = pytest.mark.gpu
CASES = [(1, 100), (2, 5), (3, 6), (4, 4096), (5, 1003), (7, 3), (16, 16_777), (33, 1000)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _rs_phase_sent(N, K):
    """Elements rank j sends in the ReduceScatter phase, from the oracle's
    schedule table ([phase][s][rank] = send, recv, source) and partition."""
    _, ln = oracle.partition(K, N)
    tab = np.asarray(oracle.ring_schedule(N))
    return [int(sum(ln[int(tab[0, s, j, 0])] for s in range(N - 1))) for j in range(N)]


@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("N,K", CASES)
def test_step_allreduce_sends_what_the_oracle_sends(N, K, op):
    x = list(W.uniform_fp32(N, K, seed_base=N))
    _, want = oracle.ring_allreduce(x, op)
    bufs = [to_dev(r) for r in x]
    ccl.ccl_step_sent(N, reset=True)
    ccl.ccl_allreduce(bufs, op=op, mode="step")
    torch.cuda.synchronize()
    got = ccl.ccl_step_sent(N)
    assert got == [int(v) for v in want]
    if K % N == 0:
        assert got == [2 * (N - 1) * K // N] * N
    ccl.ccl_allreduce(bufs, op=op, mode="fused")  # fused mode has no ring steps
    assert ccl.ccl_step_sent(N) == [0] * N


@pytest.mark.parametrize("N,K", CASES)
def test_step_reduce_scatter_and_allgather_send_one_phase(N, K):
    x = list(W.uniform_fp32(N, K, seed_base=3 * N))
    send = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    parts = [torch.empty(ln[r], dtype=torch.float32, device="cuda:0") for r in range(N)]
    full = [torch.empty(K, dtype=torch.float32, device="cuda:0") for _ in range(N)]
    want = _rs_phase_sent(N, K)
    ccl.ccl_step_sent(N, reset=True)
    ccl.ccl_reduce_scatter(send, parts, op="sum", mode="step")
    assert ccl.ccl_step_sent(N) == want
    # the AllGather entry point starts from chunk j at rank j, as the
    # ReduceScatter phase does, so rank j sends the same chunks
    ccl.ccl_allgather(parts, full, mode="step")
    torch.cuda.synchronize()
    got = ccl.ccl_step_sent(N)
    assert got == want
    assert sum(got) == (N - 1) * K  # every step moves each chunk once
