"""Many ranks, short chunks: more than 16 ranks with at most 64 elements per
chunk take a kernel that stages every rank's copy of a chunk in shared memory
and folds from there.  Its results must be the ring AllReduce's bits, for
every op and type, through AllReduce (in and out of place), ReduceScatter and
Reduce, on both sides of the switch to the long-chunk path."""
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


def _x(dtype, N, K, seed):
    return list(W.mixed_bf16(N, K, seed_base=seed)) if dtype == "bf16" else list(W.mixed_fp32(N, K, seed_base=seed))


def _check_all(x, op, N, K, root):
    want, _ = oracle.ring_allreduce(x, op)
    td = torch.bfloat16 if x[0].dtype == np.uint16 else torch.float32
    # AllReduce out of place, then in place
    send = [to_dev(r) for r in x]
    out = [torch.empty(K, dtype=td, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce(send, out, op=op)
    ccl.ccl_allreduce(send, op=op)
    # ReduceScatter and Reduce from fresh inputs
    src = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    rs = [torch.empty(ln[r], dtype=td, device=DEV) for r in range(N)]
    ccl.ccl_reduce_scatter(src, rs, op=op)
    red = [None] * N
    red[root] = torch.empty(K, dtype=td, device=DEV)
    ccl.ccl_reduce(src, red, root=root, op=op)
    torch.cuda.synchronize()
    off, _ = ccl.ccl_plan_chunks(K, N)
    for r in sorted({0, 1, N // 2, N - 1}):
        assert_bits_equal(bits(out[r]), want[r], "AR out of place rank %d" % r)
        assert_bits_equal(bits(send[r]), want[r], "AR in place rank %d" % r)
        assert_bits_equal(bits(rs[r]), want[0][off[r]:off[r] + ln[r]], "RS rank %d" % r)
    assert_bits_equal(bits(red[root]), want[0], "Reduce root")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min", "prod"])
@pytest.mark.parametrize("N", [17, 64])
@pytest.mark.parametrize("per", [0, 1, 5, 64, 65])
def test_small_chunks_every_op(dtype, op, N, per):
    """per: elements per chunk (0: fewer elements than ranks; 65: just past the
    switch to the long-chunk path), with a ragged remainder."""
    K = max(1, N * per + (N // 3 if per else N // 2))
    _check_all(_x(dtype, N, K, seed=N + per), op, N, K, root=N // 2)


@pytest.mark.parametrize("N,K,dtype,op", [(100, 100 * 7 + 41, "bf16", "sum"), (100, 37, "fp32", "avg"),
                                          (1024, 1024 * 11, "bf16", "avg"), (1024, 3001, "fp32", "sum"),
                                          (1024, 1024 * 11 + 1, "bf16", "max"), (1024, 5, "bf16", "prod")])
def test_small_chunks_up_to_1024_ranks(N, K, dtype, op):
    _check_all(_x(dtype, N, K, seed=K), op, N, K, root=N - 1)
