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


def test_graph_replay_rooted_collectives_orders_compressed_and_check():
    """Reduce, Gather, Scatter, Broadcast, the other schedules' orders, the
    compressed AllReduce (after one call outside the capture) and the result
    check, all captured in one graph and replayed once."""
    N, K, root = 6, 40_009, 4
    x = list(W.mixed_bf16(N, K, seed_base=21))
    _, ln = ccl.ccl_plan_chunks(K, N)
    send = [to_dev(r) for r in x]
    red = [None] * N
    red[root] = torch.empty(K, dtype=torch.bfloat16, device=DEV)
    parts = [send[r][:ln[r]].clone() for r in range(N)]
    parts_h = [x[r][:ln[r]] for r in range(N)]
    gat = [None] * N
    gat[root] = torch.empty(K, dtype=torch.bfloat16, device=DEV)
    sca = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    bc = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    algo = {a: [to_dev(r) for r in x] for a in ("halving_doubling", "tree", "hierarchical")}
    gq = W.normal_bf16(N, 8192 + 77, std=1e-2, seed_base=31)
    grads = [to_dev(r) for r in gq]
    res = [torch.zeros(gq.shape[1], dtype=torch.float32, device=DEV) for _ in range(N)]
    warm_g = [to_dev(r) for r in gq]
    warm_e = [torch.zeros(gq.shape[1], dtype=torch.float32, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce_compressed(warm_g, warm_e, op="avg", comp="int8_block", block=128)
    mism = torch.zeros(1, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccl.ccl_reduce(send, red, root=root, op="sum")
        ccl.ccl_gather(parts, gat, root=root)
        ccl.ccl_scatter(gat, sca, root=root)
        ccl.ccl_broadcast(send, bc, root=root)
        for a, bufs in algo.items():
            ccl.ccl_allreduce_algo(bufs, op="sum", algo=a, group_size=3 if a == "hierarchical" else 0)
        ccl.ccl_allreduce_compressed(grads, res, op="avg", comp="int8_block", block=128)
        ccl.ccl_check_identical(algo["tree"], mism)
    g.replay()
    torch.cuda.synchronize()
    want_red = oracle.reduce(x, root, "sum")
    assert_bits_equal(bits(red[root]), want_red[root], "graph reduce")
    want_g = oracle.gather(parts_h, K)
    assert_bits_equal(bits(gat[root]), want_g, "graph gather")
    for r in range(N):
        assert_bits_equal(bits(sca[r]), parts_h[r], "graph scatter %d" % r)
        assert_bits_equal(bits(bc[r]), x[root], "graph broadcast %d" % r)
    for a, bufs in algo.items():
        want = oracle.allreduce_algo(x, a, "sum", 3 if a == "hierarchical" else 0)
        for r in (0, N - 1):
            assert_bits_equal(bits(bufs[r]), want[r], "graph %s rank %d" % (a, r))
    wq, we = oracle.allreduce_compressed(list(gq), [np.zeros(gq.shape[1], np.float32)] * N, "avg", "int8_block", 128)
    for r in range(N):
        assert_bits_equal(bits(grads[r]), wq[r], "graph compressed grads %d" % r)
        assert_bits_equal(res[r].cpu().numpy().view(np.uint32), we[r].view(np.uint32), "graph residual %d" % r)
    assert int(mism.item()) == 0


def test_graph_replay_step_mode():
    """Step mode: one launch per ring step, every step after a phase's first
    chained to the one before it (programmatic dependent launch).  The first
    calls, outside the capture, set up the working space; the captured calls
    then enqueue kernels only, and two replays give the oracle's bits."""
    N, K = 8, 70003
    x = W.normal_bf16(N, K, std=1e-3, seed_base=14)
    bufs = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    rs = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    ag = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    out = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]

    def calls():
        ccl.ccl_reduce_scatter(bufs, rs, op="avg", mode="step")
        ccl.ccl_allgather(rs, ag, mode="step")
        ccl.ccl_allreduce(bufs, out, op="avg", mode="step")

    calls()
    torch.cuda.synchronize()
    for t in rs + ag + out:
        t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    want_rs = oracle.reduce_scatter(list(x), "avg")
    for rep in range(2):
        g.replay()
        torch.cuda.synchronize()
        for r in range(N):
            assert_bits_equal(bits(rs[r]), want_rs[r], "graph step RS rank %d, replay %d" % (r, rep))
            assert_bits_equal(bits(ag[r]), want[r], "graph step RS+AG rank %d, replay %d" % (r, rep))
            assert_bits_equal(bits(out[r]), want[r], "graph step AR rank %d, replay %d" % (r, rep))


def test_graph_replay_no_allocation_reduce_scatter():
    """ccl_reduce_scatter_step_static under capture: after its set-up call
    (count = 0) it needs no device memory, so a graph can hold it; two
    replays give the oracle's bits."""
    import ctypes
    fn = ccl.lib().ccl_reduce_scatter_step_static
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, pp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    N, K = 6, 6 * 10007 + 3
    x = W.mixed_fp32(N, K, seed_base=61)
    send = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    recv = [torch.zeros(ln[r], dtype=torch.float32, device=DEV) for r in range(N)]
    P = lambda ts: (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    sum_op = ccl.ccl.OPS["sum"]
    assert fn(P(send), P(recv), N, 0, 0, sum_op, None) == 0  # set-up call
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin()
        rc = fn(P(send), P(recv), N, K, 0, sum_op, ctypes.c_void_p(side.cuda_stream))
        g.capture_end()
    assert rc == 0, ccl.ccl_status_string(rc)
    want = oracle.reduce_scatter(list(x), "sum")
    for rep in range(2):
        g.replay()
        torch.cuda.synchronize()
        for r in range(N):
            assert_bits_equal(bits(recv[r]), want[r], "graph static RS rank %d, replay %d" % (r, rep))


def test_graph_replay_step_mode_copies():
    """Step-mode Broadcast, Gather, Scatter and AllToAll(v) allocate nothing:
    captured after one call outside the capture, and replayed twice, they give
    the oracle's bits."""
    N, K = 5, 5 * 4099 + 2
    x = W.normal_bf16(N, K, std=1e-2, seed_base=71)
    off, ln = ccl.ccl_plan_chunks(K, N)
    full = [to_dev(r) for r in x]
    bc = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    parts_h = [x[r][off[r]:off[r] + ln[r]] for r in range(N)]
    parts = [to_dev(p) for p in parts_h]
    gat = [None] * N
    gat[1] = torch.empty(K, dtype=torch.bfloat16, device=DEV)
    sc_send = [None] * N
    sc_send[2] = full[2]
    sc = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    counts = np.array([[3, 0, 5, 7, 2], [1, 1, 1, 1, 1], [0, 9, 2, 4, 0], [6, 6, 0, 3, 8], [2, 0, 0, 0, 11]])
    sends_h = [W.random_bits_u16(int(counts[i].sum()), seed=80 + i) for i in range(N)]
    sends = [to_dev(s) for s in sends_h]
    recv_v = [torch.empty(int(counts[:, j].sum()), dtype=torch.bfloat16, device=DEV) for j in range(N)]

    def calls():
        ccl.ccl_broadcast(full, bc, root=3, mode="step")
        ccl.ccl_gather(parts, gat, root=1, mode="step")
        ccl.ccl_scatter(sc_send, sc, root=2, mode="step")
        ccl.ccl_alltoallv(sends, recv_v, counts.tolist(), mode="step")

    calls()
    torch.cuda.synchronize()
    for t in bc + sc + recv_v + [gat[1]]:
        t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    want_bc = oracle.broadcast(list(x), 3)
    want_gat = oracle.gather(parts_h, K)
    want_sc = oracle.scatter(x[2], N)
    want_v = oracle.alltoallv(sends_h, counts)
    for rep in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(bits(gat[1]), want_gat, "graph step gather, replay %d" % rep)
        for r in range(N):
            assert_bits_equal(bits(bc[r]), want_bc[r], "graph step broadcast rank %d, replay %d" % (r, rep))
            assert_bits_equal(bits(sc[r]), want_sc[r], "graph step scatter rank %d, replay %d" % (r, rep))
            assert_bits_equal(bits(recv_v[r]), want_v[r], "graph step alltoallv rank %d, replay %d" % (r, rep))
