"""GPU parity for AllReduce under the other schedules' summation orders
(halving-doubling, binomial tree, two-level hierarchical) against the
oracle's step-by-step simulations, bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import assert_bits_equal, bits, empty_like_host, to_dev, torch_dtype

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)


def _inputs(dtype, N, K, seed):
    return list(W.mixed_bf16(N, K, seed_base=seed)) if dtype == "bf16" else list(W.mixed_fp32(N, K, seed_base=seed))


def _run(x, algo, op, group, in_place, pad=0):
    send = [to_dev(r, pad_elems=pad) for r in x]
    recv = send if in_place else [empty_like_host(r.size, torch_dtype(x), pad_elems=pad) for r in x]
    ccl.ccl_allreduce_algo(send, recv, op=op, algo=algo, group_size=group)
    torch.cuda.synchronize()
    return [bits(t) for t in recv]


with open(os.path.join(GOLD, "order_cases.json")) as f:
    _CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", _CASES, ids=lambda c: c["name"])
def test_order_goldens_on_gpu(case):
    ins = [np.array([int(v, 16) for v in row], dtype=np.uint16) for row in case["inputs_bits"]]
    exp = np.array([int(v, 16) for v in case["expected_bits"]], dtype=np.uint16)
    for g in _run(ins, case["algo"], case["op"], case["group"], True):
        assert_bits_equal(g, exp, case["name"])


SHAPES = [(1, 7), (2, 4099), (3, 10), (4, 4096), (5, 3), (6, 70001), (7, 333), (8, 70000), (8, 3 * 2048 + 5),
          (12, 9999), (16, 70001), (17, 4097), (32, 5000)]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min"])
@pytest.mark.parametrize("N,K", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("algo", ["halving_doubling", "tree"])
def test_tree_orders_match_oracle(algo, N, K, op, dtype):
    x = _inputs(dtype, N, K, seed=N * 13 + K)
    want = oracle.allreduce_algo(x, algo, op)
    got = _run(x, algo, op, 0, in_place=(K % 2 == 0))
    for r in range(N):
        assert_bits_equal(got[r], want[r], "%s N=%d K=%d rank %d" % (algo, N, K, r))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min"])
@pytest.mark.parametrize("N,L,K", [(4, 2, 4099), (6, 3, 70001), (6, 2, 10), (8, 4, 70000), (8, 2, 3 * 2048 + 5),
                                   (8, 8, 1000), (8, 1, 1000), (12, 4, 9999), (16, 4, 70001), (24, 3, 5000)])
def test_hierarchical_matches_oracle(N, L, K, op, dtype):
    x = _inputs(dtype, N, K, seed=N * 17 + L + K)
    want = oracle.allreduce_algo(x, "hierarchical", op, L)
    got = _run(x, "hierarchical", op, L, in_place=(K % 2 == 1))
    for r in range(N):
        assert_bits_equal(got[r], want[r], "hier N=%d L=%d K=%d rank %d" % (N, L, K, r))


@pytest.mark.parametrize("algo,group", [("halving_doubling", 0), ("tree", 0), ("hierarchical", 2)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_orders_unaligned_buffers(algo, group, dtype):
    N, K = 6, 5003
    x = _inputs(dtype, N, K, seed=99)
    want = oracle.allreduce_algo(x, algo, "sum", group)
    got = _run(x, algo, "sum", group, in_place=False, pad=1)
    for r in range(N):
        assert_bits_equal(got[r], want[r], "%s unaligned rank %d" % (algo, r))
