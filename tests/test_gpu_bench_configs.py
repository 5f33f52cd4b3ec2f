"""The other benchmark rows at full size, in the launch configuration the
benchmark times, checked against the oracle: N=8 bf16 with 64 Mi elements per
rank (the headline's shape).

  orders      AllReduce AVG in halving-doubling, binomial-tree and 2x4
              hierarchical order (sampled closed-form values of each order)
  compressed  INT8 blocks of 128 + error feedback, AVG (the whole result and
              every residual, against the full oracle run)
  premul      AllReduce with the pre-multiplied AVG (sampled closed-form values)
  topk        Top-k AllReduce AVG, k = 1%, with error feedback (the definition
              checked as properties of the whole result, sums at sampled
              positions against the oracle's closed form)
  reduce      Reduce SUM to rank 0 (sampled closed-form values)
  gather      Gather to rank 0, Scatter back, Broadcast from rank 0 (copies,
              compared in full)
  step mode   the headline AllReduce AVG executed step by step (in full)
"""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W
from ring_allreduce_rank_gb300.arena import RankArena

from gpu_util import DEV, assert_bits_equal, bits, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N, K = 8, 64 * 1024 * 1024


@pytest.fixture(scope="module")
def x():
    assert torch.cuda.is_available()
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    yield W.normal_bf16(N, K, std=1e-3, seed_base=0)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _sample(parts, seed):
    """Random indices plus both ends of every chunk of every given partition."""
    g = np.random.Generator(np.random.PCG64(seed))
    idx = set(g.integers(0, K, size=8192).tolist())
    for n in parts:
        off, ln = ccl.ccl_plan_chunks(K, n)
        for c in range(n):
            if ln[c]:
                idx.update([off[c], off[c] + ln[c] - 1])
    return np.array(sorted(idx), dtype=np.int64)


def _arena(rows):
    a = RankArena(N, K, torch.bfloat16, device=DEV)
    a.load([r.view(np.int16) for r in rows])
    return a


@pytest.mark.parametrize("algo,group", [("halving_doubling", 0), ("tree", 0), ("hierarchical", 4)])
def test_orders_full_size(x, algo, group):
    a = _arena(x)
    ccl.ccl_allreduce_algo(a.ranks, op="avg", algo=algo, group_size=4 if algo == "hierarchical" else 0)
    torch.cuda.synchronize()
    idx = _sample([N, 4, 2], seed=len(algo))
    want = oracle.allreduce_algo_at(list(x), algo, idx.astype(np.uint64), "avg", group)
    it = torch.from_numpy(idx).to(DEV)
    for r in (0, 3, N - 1):
        assert_bits_equal(bits(a.ranks[r].index_select(0, it)), want, "%s rank %d" % (algo, r))
    for r in range(1, N):
        assert torch.equal(a.ranks[r].view(torch.int16), a.ranks[0].view(torch.int16)), "%s rank %d" % (algo, r)


def test_compressed_full_size(x):
    grads = [to_dev(r) for r in x]
    res = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce_compressed(grads, res, op="avg", comp="int8_block", block=128)
    torch.cuda.synchronize()
    got_g = [bits(g) for g in grads]
    got_e = [r.cpu().numpy().view(np.uint32) for r in res]
    del grads, res
    torch.cuda.empty_cache()
    want_g, want_e = oracle.allreduce_compressed(list(x), [np.zeros(K, np.float32) for _ in range(N)], "avg",
                                                 "int8_block", 128)
    for r in range(N):
        assert_bits_equal(got_g[r], want_g[r], "compressed grads rank %d" % r)
        assert_bits_equal(got_e[r], want_e[r].view(np.uint32), "compressed residual rank %d" % r)


def test_premul_full_size(x):
    a = _arena(x)
    ccl.ccl_allreduce(a.ranks, op="avg_premul")
    torch.cuda.synchronize()
    idx = _sample([N], seed=6)
    want = oracle.ring_allreduce_at(list(x), idx.astype(np.uint64), "avg_premul")
    it = torch.from_numpy(idx).to(DEV)
    for r in range(N):
        assert_bits_equal(bits(a.ranks[r].index_select(0, it)), want, "premul rank %d" % r)


def test_topk_full_size(x):
    """Per rank, the sent set S must be exactly the definition's: every value
    of S has a magnitude at least that of every value outside it, S holds at
    least k values, and without the values tied at its smallest magnitude it
    would hold fewer than k.  The result at sampled positions is then the
    oracle's fp32 ring-order AVG of the sent values, rounded to bf16."""
    k = K // 100
    g = [to_dev(r) for r in x]
    u = [gr.float() for gr in g]  # u = g + e with e = 0
    e = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce_topk(g, e, k, op="avg")
    torch.cuda.synchronize()
    sent = []
    for r in range(N):
        m = (e[r] == 0) & (u[r] != 0)  # sent values leave no residual (finite inputs)
        mag = u[r].abs()
        lo = mag[m].min()
        assert int(m.sum()) >= k
        assert bool((mag[~m] <= lo).all())
        assert int((m & (mag > lo)).sum()) < k
        assert int(((mag == lo) & ~m).sum()) == 0  # every tie at the threshold is sent
        assert torch.equal(e[r][~m], u[r][~m])
        sent.append(torch.where(m, u[r], torch.zeros_like(u[r])))
    idx = _sample([N], seed=8)
    it = torch.from_numpy(idx).to(DEV)
    vals = [s.index_select(0, it).cpu().numpy() for s in sent]
    want = oracle.ring_allreduce_gathered(vals, K, idx.astype(np.uint64), "avg")
    want = W.to_bf16_bits(want)
    for r in range(N):
        assert_bits_equal(bits(g[r].index_select(0, it)), want, "topk rank %d" % r)


def test_reduce_full_size(x):
    send = [to_dev(r) for r in x]
    recv = [None] * N
    recv[0] = torch.empty(K, dtype=torch.bfloat16, device=DEV)
    ccl.ccl_reduce(send, recv, root=0, op="sum")
    torch.cuda.synchronize()
    idx = _sample([N], seed=5)
    want = oracle.ring_allreduce_at(list(x), idx.astype(np.uint64), "sum")
    assert_bits_equal(bits(recv[0].index_select(0, torch.from_numpy(idx).to(DEV))), want, "reduce root")
    for r in range(N):  # the inputs are untouched
        assert torch.equal(send[r].view(torch.int16).cpu(), torch.from_numpy(x[r].view(np.int16)))


def test_gather_scatter_broadcast_full_size(x):
    off, ln = ccl.ccl_plan_chunks(K, N)
    parts = [to_dev(x[r][:ln[r]]) for r in range(N)]
    full = [None] * N
    full[0] = torch.empty(K, dtype=torch.bfloat16, device=DEV)
    ccl.ccl_gather(parts, full, root=0)
    back = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    ccl.ccl_scatter(full, back, root=0)
    torch.cuda.synchronize()
    want = np.concatenate([x[r][:ln[r]] for r in range(N)])
    assert_bits_equal(bits(full[0]), want, "gather")
    for r in range(N):
        assert torch.equal(back[r].view(torch.int16), parts[r].view(torch.int16)), "scatter rank %d" % r
    del parts, full, back
    a = _arena(x)
    ccl.ccl_broadcast(a.ranks, a.ranks, root=0)
    torch.cuda.synchronize()
    src = to_dev(x[0])
    for r in range(N):
        assert torch.equal(a.ranks[r].view(torch.int16), src.view(torch.int16)), "broadcast rank %d" % r


def test_step_mode_full_size(x):
    a = _arena(x)
    ccl.ccl_allreduce(a.ranks, op="avg", mode="step")
    torch.cuda.synchronize()
    got = a.rows_bits()
    del a
    torch.cuda.empty_cache()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(got[r].view(np.uint16), want[r], "step mode rank %d" % r)
