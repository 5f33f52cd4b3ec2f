"""Failure detection on the host (no GPU is faulted, trapped or hung): the
oracle's ring with one thread per rank, where the thread owning one rank
leaves before its first send, as a failed rank would.  The pages note that a
rank that exits early hangs every other rank until a timeout (Lesson 3,
pitfalls); here every wait is bounded, so the others give up after the
deadline and the call returns a timeout status instead of hanging."""
import time

import numpy as np
import pytest

from ring_allreduce_rank_gb300 import workloads as W


@pytest.mark.parametrize("N,threads,withhold", [(8, 8, 3), (8, 4, 0), (5, 5, 4), (16, 3, 15), (2, 2, 1)])
def test_a_rank_that_leaves_is_detected_within_the_deadline(oracle_mod, N, threads, withhold):
    x = list(W.normal_fp32(N, 1000, seed_base=N))
    t0 = time.monotonic()
    _, rc = oracle_mod.ring_allreduce_threads_status(x, "sum", threads, withhold=withhold, timeout_ms=200)
    dt = time.monotonic() - t0
    assert rc == oracle_mod.TIMED_OUT
    assert dt < 10.0  # one deadline (0.2 s), then every other wait returns at once


def test_without_a_failure_the_same_call_completes_with_the_ring_bits(oracle_mod):
    x = list(W.mixed_bf16(8, 777, seed_base=2))
    outs, rc = oracle_mod.ring_allreduce_threads_status(x, "avg", 8, withhold=-1, timeout_ms=5000)
    assert rc == 0
    want, _ = oracle_mod.ring_allreduce(x, "avg")
    for r in range(8):
        np.testing.assert_array_equal(outs[r], want[r])


def test_a_failure_needs_someone_to_notice(oracle_mod):
    x = list(W.normal_fp32(4, 10, seed_base=1))
    with pytest.raises(RuntimeError):
        oracle_mod.ring_allreduce_threads_status(x, "sum", 1, withhold=0, timeout_ms=100)
