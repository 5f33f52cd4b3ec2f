"""The bucketer: buckets launched on a communication stream as a synthetic
backward pass marks gradients ready (events on a compute stream) give the
same bits as the oracle's bucket AllReduce, in any marking order, step
after step."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, assert_bits_equal, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)


def _grads(N, numels, seed):
    return [[W.normal_bf16(1, n, seed_base=seed + 97 * r + t)[0] for t, n in enumerate(numels)] for r in range(N)]


@pytest.mark.parametrize("be", [10000, 2500, 60000])
@pytest.mark.parametrize("max_ctas", [0, 3])
@pytest.mark.parametrize("order", ["backward", "forward", "shuffled"])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_bucketer_matches_oracle_over_two_steps(order, op, max_ctas, be):
    """Bucket sizes from many small buckets (a bucket per few thousand
    elements) to few large ones, the bucket-size policies the overlap
    benchmark compares."""
    N = 4
    numels = [5000, 20000, 3, 70001, 4096, 1]
    dev_grads = [[torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in numels] for _ in range(N)]
    bk = ccl.CclBucketer(dev_grads, bucket_bytes=be * 2, op=op, max_ctas=max_ctas)
    nb, _ = bk.status()
    assert nb == (sum(numels) + be - 1) // be
    compute = torch.cuda.Stream()
    comm = torch.cuda.Stream()
    T = len(numels)
    seq = {"backward": list(range(T - 1, -1, -1)), "forward": list(range(T)),
           "shuffled": [3, 0, 5, 1, 4, 2]}[order]
    for step in range(2):
        host = _grads(N, numels, seed=1000 * step)
        pinned = [[torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory() for h in row]
                  for row in host]
        bk.reset()
        events = []
        for t in seq:
            with torch.cuda.stream(compute):
                for r in range(N):  # "backward" produces tensor t on every rank
                    dev_grads[r][t].copy_(pinned[r][t], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(compute)
            events.append(ev)
            bk.mark_ready(t, ev, comm)
        assert bk.status() == (nb, nb)
        comm.synchronize()
        want = oracle.bucket_allreduce(host, be, op)
        for r in range(N):
            for t in range(T):
                assert_bits_equal(bits(dev_grads[r][t]), want[r][t], "step %d rank %d tensor %d" % (step, r, t))
    with pytest.raises(ccl.CclError):
        bk.mark_ready(0, None, comm)
        bk.mark_ready(0, None, comm)
    bk.close()
