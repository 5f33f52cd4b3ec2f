"""The pure-Python ring (oracle/ring_py.py) against the C oracle and the pages
(no GPU): AllReduce, ReduceScatter and the compressed AllReduce with error
feedback.  Two independent statements of the same schedule, in two languages,
must agree bit for bit -- results and the elements each rank sends -- on small
inputs that mix signed zeros, subnormals, infinities and NaNs into values of
widely varying magnitude, for every operator and both buffer types; and the
Python ring must reproduce the pages' printed AllReduce examples."""
import json
import os

import numpy as np
import pytest

from oracle import ring_py
from ring_allreduce_rank_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _bits(a):
    a = np.asarray(a)
    return a if a.dtype == np.uint16 else a.view(np.uint32)


@pytest.mark.parametrize("case", [c for c in json.load(open(GOLD))["cases"] if c["collective"] == "allreduce"],
                         ids=lambda c: c["name"])
def test_printed_allreduce_examples(case):
    ins = [np.asarray(r, dtype=np.float32) for r in case["inputs"]]
    out, sent = ring_py.ring_allreduce(ins, case["op"])
    for r, want in enumerate(case["expected"]):
        np.testing.assert_array_equal(out[r], np.asarray(want, dtype=np.float32))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min", "prod", "avg_premul"])
@pytest.mark.parametrize("N,K", [(1, 5), (2, 9), (3, 1), (3, 17), (4, 40), (5, 4), (7, 23), (8, 64)])
def test_agrees_with_the_c_oracle(oracle_mod, dtype, op, N, K):
    seed = 1000 + 37 * N + K
    x = list(W.mixed_bf16(N, K, seed_base=seed) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=seed))
    want, want_sent = oracle_mod.ring_allreduce(x, op)
    got, got_sent = ring_py.ring_allreduce(x, op)
    for r in range(N):
        np.testing.assert_array_equal(_bits(got[r]), _bits(want[r]), err_msg="rank %d" % r)
    assert got_sent == [int(v) for v in want_sent]


def test_bf16_rounding_agrees_with_the_c_oracle_on_deciding_patterns(oracle_mod):
    g = np.random.default_rng(5)
    hi = g.integers(0, 1 << 16, size=4096, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    pats = (hi[:, None] << 16 | lows[None, :]).ravel()
    want = [oracle_mod.round_bf16(int(p)) for p in pats]
    got = [ring_py.bf16_from_f32(int(p)) for p in pats]
    assert got == want


def test_printed_reduce_scatter_example():
    case = [c for c in json.load(open(GOLD))["cases"] if c["collective"] == "reduce_scatter"][0]
    ins = [np.asarray(r, dtype=np.float32) for r in case["inputs"]]
    out = ring_py.reduce_scatter(ins, case["op"])
    for r, want in enumerate(case["expected"]):
        np.testing.assert_array_equal(out[r], np.asarray(want, dtype=np.float32))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min", "prod", "avg_premul"])
@pytest.mark.parametrize("N,K", [(1, 5), (3, 17), (4, 3), (6, 50)])
def test_reduce_scatter_agrees_with_the_c_oracle(oracle_mod, dtype, op, N, K):
    seed = 2000 + 13 * N + K
    x = list(W.mixed_bf16(N, K, seed_base=seed) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=seed))
    want = oracle_mod.reduce_scatter(x, op)
    got = ring_py.reduce_scatter(x, op)
    for r in range(N):
        np.testing.assert_array_equal(_bits(got[r]), _bits(want[r]), err_msg="rank %d" % r)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("comp,block,k", [("int8_block", 128, 0), ("int8_block", 7, 0), ("threshold", 0, 0),
                                          ("topk", 0, 1), ("topk", 0, 13), ("topk", 0, 0), ("topk", 0, 10_000)])
@pytest.mark.parametrize("N,K", [(1, 40), (3, 300), (5, 129)])
def test_compressed_allreduce_agrees_with_the_c_oracle(oracle_mod, dtype, op, comp, block, k, N, K):
    seed = 3000 + 7 * N + K
    g = list(W.mixed_bf16(N, K, seed_base=seed) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=seed))
    with np.errstate(invalid="ignore"):
        e = list(W.mixed_fp32(N, K, seed_base=seed + 100, special_frac=0.01) * np.float32(1e-3))
    # two steps, the second carrying the first's residuals (error feedback)
    for _ in range(2):
        want_g, want_e = oracle_mod.allreduce_compressed(g, e, op=op, comp=comp, block=block or 128,
                                                         threshold=0.5, k=k)
        got_g, got_e = ring_py.allreduce_compressed(g, e, op=op, comp=comp, block=block or 128,
                                                    threshold=0.5, k=k)
        for r in range(N):
            np.testing.assert_array_equal(_bits(got_g[r]), _bits(want_g[r]), err_msg="grads rank %d" % r)
            np.testing.assert_array_equal(_bits(got_e[r]), _bits(want_e[r]), err_msg="residual rank %d" % r)
        g, e = want_g, want_e


ORDERS = {"halving_doubling": lambda x, op, L: ring_py.allreduce_halving_doubling(x, op),
          "tree": lambda x, op, L: ring_py.allreduce_binomial_tree(x, op),
          "hierarchical": lambda x, op, L: ring_py.allreduce_hierarchical(x, L, op)}


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min", "prod"])
@pytest.mark.parametrize("algo,N,L", [("halving_doubling", 1, 0), ("halving_doubling", 2, 0),
                                      ("halving_doubling", 5, 0), ("halving_doubling", 6, 0),
                                      ("halving_doubling", 8, 0), ("halving_doubling", 11, 0),
                                      ("tree", 3, 0), ("tree", 7, 0), ("tree", 8, 0), ("tree", 13, 0),
                                      ("hierarchical", 6, 3), ("hierarchical", 6, 2), ("hierarchical", 8, 4),
                                      ("hierarchical", 9, 3), ("hierarchical", 4, 1), ("hierarchical", 4, 4)])
@pytest.mark.parametrize("K", [1, 29])
def test_other_orders_agree_with_the_c_oracle(oracle_mod, dtype, op, algo, N, L, K):
    seed = 4000 + 31 * N + K + L
    x = list(W.mixed_bf16(N, K, seed_base=seed) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=seed))
    want = oracle_mod.allreduce_algo(x, algo, op, group=L)
    got = ORDERS[algo](x, op, L)
    for r in range(N):
        np.testing.assert_array_equal(_bits(got[r]), _bits(want[r]), err_msg="%s rank %d" % (algo, r))


@pytest.mark.parametrize("case", json.load(open(os.path.join(os.path.dirname(__file__), "golden", "order_cases.json")))
                         ["cases"], ids=lambda c: c["name"])
def test_other_orders_reproduce_the_hand_derived_cases(case):
    ins = [np.array([int(v, 16) for v in row], dtype=np.uint16 if case["dtype"] == "bf16" else np.uint32)
           for row in case["inputs_bits"]]
    if case["dtype"] == "fp32":
        ins = [a.view(np.float32) for a in ins]
    got = ORDERS[case["algo"]](ins, case["op"], case.get("group", 0))
    want = [int(v, 16) for v in case["expected_bits"]]
    for r in range(len(ins)):
        assert [int(v) for v in _bits(got[r])] == want, "rank %d" % r


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 6), (3, 10), (4, 2), (5, 37)])
def test_other_collectives_agree_with_the_c_oracle(oracle_mod, dtype, N, K):
    seed = 5000 + 3 * N + K
    x = list(W.mixed_bf16(N, K, seed_base=seed) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=seed))
    eq = np.testing.assert_array_equal
    for op in ("sum", "avg", "max", "avg_premul"):
        for root in {0, N - 1}:
            for a, b in zip(ring_py.reduce(x, root, op), oracle_mod.reduce(x, root, op)):
                eq(_bits(a), _bits(b))
    _, ln = ring_py.partition(K, N)
    chunks = [x[r][:ln[r]] for r in range(N)]
    for a, b in zip(ring_py.allgather(chunks, K), oracle_mod.allgather(chunks, K)):
        eq(_bits(a), _bits(b))
    eq(_bits(ring_py.gather(chunks, K)), _bits(oracle_mod.gather(chunks, K)))
    for a, b in zip(ring_py.scatter(x[0], N), oracle_mod.scatter(x[0], N)):
        eq(_bits(a), _bits(b))
    for root in {0, N - 1}:
        for a, b in zip(ring_py.broadcast(x, root), oracle_mod.broadcast(x, root)):
            eq(_bits(a), _bits(b))
    g = np.random.default_rng(seed)
    counts = g.integers(0, 5, size=(N, N))
    sends = [np.asarray(x[i])[:0] if counts[i].sum() == 0 else
             np.resize(np.asarray(x[i]), int(counts[i].sum())) for i in range(N)]
    for a, b in zip(ring_py.alltoallv(sends, counts), oracle_mod.alltoallv(sends, counts)):
        eq(_bits(a), _bits(b))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "avg_premul"])
@pytest.mark.parametrize("B", [1, 7, 64, 1000])
def test_bucket_allreduce_agrees_with_the_c_oracle(oracle_mod, dtype, op, B):
    N, numels = 3, [5, 40, 1, 0, 23]
    gen = W.mixed_bf16 if dtype == "bf16" else W.mixed_fp32
    tensors = [[gen(1, n, seed_base=600 + 10 * r + t)[0] for t, n in enumerate(numels)] for r in range(N)]
    got = ring_py.bucket_allreduce(tensors, B, op)
    want = oracle_mod.bucket_allreduce(tensors, B, op)
    for r in range(N):
        for t in range(len(numels)):
            np.testing.assert_array_equal(_bits(got[r][t]), _bits(want[r][t]), err_msg="rank %d tensor %d" % (r, t))
