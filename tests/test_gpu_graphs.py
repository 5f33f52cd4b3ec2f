"""The fused collectives enqueue kernels only (no host synchronisation, no
allocation), so a sequence of calls can be captured once in a CUDA graph and
replayed.  Replays must give the same bits as the oracle."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)


def test_graph_replay_allreduce_reduce_scatter_allgather():
    N, K = 8, 70003
    x = W.normal_bf16(N, K, std=1e-3, seed_base=4)
    bufs = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    rs = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    ag = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    out = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccl.ccl_reduce_scatter(bufs, rs, op="avg")
        ccl.ccl_allgather(rs, ag)
        ccl.ccl_allreduce(bufs, out, op="avg")
    for _ in range(2):  # replays are idempotent: inputs are not overwritten
        g.replay()
        torch.cuda.synchronize()
        want, _ = oracle.ring_allreduce(list(x), "avg")
        for r in range(N):
            assert_bits_equal(bits(out[r]), want[r], "graph AR rank %d" % r)
            assert_bits_equal(bits(ag[r]), want[r], "graph RS+AG rank %d" % r)


def test_graph_replay_alltoallv_and_buckets():
    N = 4
    counts = np.array([[3, 0, 5, 7], [1, 1, 1, 1], [0, 9, 2, 4], [6, 6, 0, 3]])
    sends_h = [W.random_bits_u16(int(counts[i].sum()), seed=i) for i in range(N)]
    send = [to_dev(s) for s in sends_h]
    recv = [torch.empty(int(counts[:, j].sum()), dtype=torch.bfloat16, device=DEV) for j in range(N)]
    numels = [100, 4096, 3, 20000]
    grads_h = [[W.normal_bf16(1, n, seed_base=10 * r + t)[0] for t, n in enumerate(numels)] for r in range(N)]
    grads = [[to_dev(gh) for gh in row] for row in grads_h]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccl.ccl_alltoallv(send, recv, counts.tolist())
        ccl.ccl_bucket_allreduce(grads, bucket_bytes=2 * 5000, op="max")
    g.replay()
    torch.cuda.synchronize()
    want = oracle.alltoallv(sends_h, counts)
    for j in range(N):
        assert_bits_equal(bits(recv[j]), want[j], "graph A2Av %d" % j)
    wantb = oracle.bucket_allreduce(grads_h, 5000, "max")
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(bits(grads[r][t]), wantb[r][t], "graph bucket r%d t%d" % (r, t))
