"""Pins for the oracle's other schedules (halving-doubling, binomial tree,
two-level hierarchical): hand-derived IEEE cases that separate the orders,
the step simulations against their closed forms, exact brute force on integer
inputs, the degenerate cases that reduce to the ring, and the error bound of
each summation tree."""
import json
import os

import numpy as np
import pytest

from ring_allreduce_rank_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
ALGOS = ["halving_doubling", "tree", "hierarchical"]


def _cases():
    with open(os.path.join(GOLD, "order_cases.json")) as f:
        return json.load(f)["cases"]


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _inputs(dtype, N, K, seed):
    return list(W.mixed_bf16(N, K, seed_base=seed)) if dtype == "bf16" else list(W.mixed_fp32(N, K, seed_base=seed))


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_order_goldens(oracle_mod, case):
    ins = [np.array([int(v, 16) for v in row], dtype=np.uint16) for row in case["inputs_bits"]]
    exp = np.array([int(v, 16) for v in case["expected_bits"]], dtype=np.uint16)
    outs = oracle_mod.allreduce_algo(ins, case["algo"], case["op"], case["group"])
    for o in outs:
        np.testing.assert_array_equal(o, exp)
    cf = oracle_mod.allreduce_algo_at(ins, case["algo"], np.arange(exp.size), case["op"], case["group"])
    np.testing.assert_array_equal(cf, exp)


def _groups(N):
    return [L for L in (1, 2, 3, 4, N) if N % L == 0] or [1]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min"])
@pytest.mark.parametrize("N,K", [(1, 3), (2, 9), (3, 10), (4, 37), (5, 3), (6, 101), (7, 64), (8, 1000), (12, 77),
                                 (16, 257)])
@pytest.mark.parametrize("algo", ALGOS)
def test_step_simulation_equals_closed_form(oracle_mod, algo, N, K, op, dtype):
    x = _inputs(dtype, N, K, seed=N * 31 + K)
    for L in (_groups(N) if algo == "hierarchical" else [0]):
        st = oracle_mod.allreduce_algo(x, algo, op, L)
        cf = oracle_mod.allreduce_algo_at(x, algo, np.arange(K), op, L)
        for r in range(N):
            np.testing.assert_array_equal(_bits(st[r]), _bits(cf))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("N", [3, 4, 6, 8, 9])
def test_integer_inputs_exact(oracle_mod, algo, N):
    x = W.integers_fp32(N, 500, seed=N)
    ref = x.astype(np.float64).sum(axis=0)
    for L in (_groups(N) if algo == "hierarchical" else [0]):
        for o in oracle_mod.allreduce_algo(list(x), algo, "sum", L):
            np.testing.assert_array_equal(o.astype(np.float64), ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N", [2, 3, 4, 6, 8])
def test_degenerate_schedules_reduce_to_the_ring(oracle_mod, N, dtype):
    """One group of N, or N groups of one, is the flat ring; with N = 2 every
    schedule is a single addition."""
    x = _inputs(dtype, N, 333, seed=N)
    ring, _ = oracle_mod.ring_allreduce(x, "sum")
    for L in (1, N):
        h = oracle_mod.allreduce_algo(x, "hierarchical", "sum", L)
        np.testing.assert_array_equal(_bits(h[0]), _bits(ring[0]))
    if N == 2:
        for algo in ("halving_doubling", "tree"):
            np.testing.assert_array_equal(_bits(oracle_mod.allreduce_algo(x, algo, "sum")[0]), _bits(ring[0]))


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_tree_equals_halving_doubling_for_powers_of_two(oracle_mod, N):
    """For N = 2^m the binomial tree and halving-doubling group the same
    leaves in the same order (adjacent pairs, then pairs of pairs)."""
    x = _inputs("bf16", N, 999, seed=N)
    a = oracle_mod.allreduce_algo(x, "tree", "sum")
    b = oracle_mod.allreduce_algo(x, "halving_doubling", "sum")
    np.testing.assert_array_equal(a[0], b[0])


@pytest.mark.parametrize("algo,depth", [("halving_doubling", lambda N: int(np.ceil(np.log2(N))) + 1),
                                        ("tree", lambda N: int(np.ceil(np.log2(N))))])
def test_tree_orders_error_bound(oracle_mod, algo, depth):
    """A summation tree of depth d rounds each contribution at most d times:
    |y - y64| <= d (2^-8 + 2^-24) sum|x| for bf16."""
    N, K = 8, 20000
    x = list(W.normal_bf16(N, K, seed_base=2))
    y = W.bf16_bits_to_f32(oracle_mod.allreduce_algo(x, algo, "sum")[0]).astype(np.float64)
    y64, absum = oracle_mod.sum_f64(x, "sum")
    assert np.all(np.abs(y - y64) <= depth(N) * (2.0 ** -8 + 2.0 ** -24) * absum * (1 + 1e-6) + 1e-300)
