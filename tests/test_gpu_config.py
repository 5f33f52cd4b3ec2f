"""Library settings on the device: a forced mode (ccl_set_mode_override, or
CCL_MODE in a fresh process) changes how a call runs -- the number of kernels
it launches and the mode its trace record shows -- and never its bits, which
stay the oracle's; the default bucket size (ccl_set_default_bucket_bytes) is
what bucket_bytes = 0 selects."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _restore_settings():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    prior = ccl.ccl_get_config()
    yield
    torch.cuda.synchronize()
    ccl.ccl_set_mode_override(prior["mode_override"])
    ccl.ccl_set_default_bucket_bytes(prior["default_bucket_bytes"])
    ccl.ccl_set_trace(prior["trace"])


def _allreduce(x, op, mode):
    send = [to_dev(r) for r in x]
    before = ccl.ccl_launch_count()
    ccl.ccl_allreduce(send, op=op, mode=mode)
    torch.cuda.synchronize()
    return [bits(t) for t in send], ccl.ccl_launch_count() - before


def _reduce_scatter(x, op, mode):
    N, K = len(x), x[0].size
    send = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    out = [torch.empty(ln[r], dtype=send[0].dtype, device="cuda:0") for r in range(N)]
    before = ccl.ccl_launch_count()
    ccl.ccl_reduce_scatter(send, out, op=op, mode=mode)
    torch.cuda.synchronize()
    return [bits(t) for t in out], ccl.ccl_launch_count() - before


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_forced_mode_changes_the_launches_not_the_bits(dtype):
    N, K = 5, 3 * 4096 + 7
    x = list(W.mixed_bf16(N, K, seed_base=21) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=21))
    want, _ = oracle.ring_allreduce(x, "avg")
    ccl.ccl_set_mode_override(None)
    _, n_fused = _allreduce(x, "avg", "fused")
    _, n_step = _allreduce(x, "avg", "step")
    assert n_fused == 1 and n_step >= 2 * (N - 1)

    ccl.ccl_set_trace(True)
    ccl.ccl_trace_clear()
    ccl.ccl_set_mode_override("step")
    assert ccl.ccl_get_config()["mode_override"] == "step"
    got, n = _allreduce(x, "avg", "fused")
    assert n == n_step
    for r in range(N):
        assert_bits_equal(got[r], want[r], "forced step, rank %d" % r)
    rec = ccl.ccl_trace_read()[-1]
    assert rec["collective"] == "allreduce" and rec["mode"] == 1 and rec["launches"] == n_step

    ccl.ccl_set_mode_override("fused")
    got, n = _allreduce(x, "avg", "step")
    assert n == 1
    for r in range(N):
        assert_bits_equal(got[r], want[r], "forced fused, rank %d" % r)
    assert ccl.ccl_trace_read()[-1]["mode"] == 0

    # ReduceScatter: the forced step mode brings its workspace with it
    want_rs = oracle.reduce_scatter(x, "sum")
    ccl.ccl_set_mode_override("step")
    got, n = _reduce_scatter(x, "sum", "fused")
    assert n > 1
    for r in range(N):
        assert_bits_equal(got[r], want_rs[r], "forced step ReduceScatter, rank %d" % r)

    # an invalid mode argument is still rejected under an override
    with pytest.raises(ccl.CclError) as e:
        ccl.ccl_allreduce([to_dev(r) for r in x], op="sum", mode=7)
    assert e.value.status == 1


def test_default_bucket_size_is_what_zero_selects():
    N, es = 4, 2
    numels = [3000, 70001, 5, 120003, 4096]
    grads_h = [[W.mixed_bf16(1, n, seed_base=100 * r + t)[0] for t, n in enumerate(numels)] for r in range(N)]
    small = 65536  # bytes: 32768 bf16 elements per bucket
    want = oracle.bucket_allreduce(grads_h, small // es, "sum")
    # the setting matters here: one 25 MiB bucket folds these elements in other orders
    other = oracle.bucket_allreduce(grads_h, 25 * W.MiB // es, "sum")
    assert any(not np.array_equal(want[r][t], other[r][t]) for r in range(N) for t in range(len(numels)))

    ccl.ccl_set_default_bucket_bytes(small)
    grads = [[to_dev(g) for g in row] for row in grads_h]
    ccl.ccl_bucket_allreduce(grads, op="sum")  # bucket_bytes = 0
    torch.cuda.synchronize()
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(bits(grads[r][t]), want[r][t], "rank %d tensor %d" % (r, t))
    # the bucketer plans with the same default
    b = ccl.CclBucketer([[to_dev(g) for g in row] for row in grads_h], op="sum")
    try:
        assert b.status()[0] == -(-sum(numels) // (small // es))
    finally:
        b.close()


CHILD = r"""
import sys
sys.path.insert(0, %r)
import numpy as np, torch
import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W
N, K = 8, 8 * 2048 + 3
x = list(W.normal_bf16(N, K, std=1e-3, seed_base=3))
send = [torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).cuda() for r in x]
before = ccl.ccl_launch_count()
ccl.ccl_allreduce(send, op="avg", mode="fused")
torch.cuda.synchronize()
n = ccl.ccl_launch_count() - before
want, _ = oracle.ring_allreduce(x, "avg")
same = all(np.array_equal(send[r].view(torch.int16).cpu().numpy().view(np.uint16), want[r]) for r in range(N))
print(n, int(same), ccl.ccl_get_config()["mode_override"])
""" % ROOT


@pytest.mark.parametrize("env,fused", [({}, True), ({"CCL_MODE": "step"}, False)])
def test_mode_from_the_environment_in_a_fresh_process(env, fused):
    e = {k: v for k, v in os.environ.items() if not k.startswith("CCL_")}
    e.update(env)
    p = subprocess.run([sys.executable, "-c", CHILD], env=e, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    n, same, override = p.stdout.split()[-3:]
    assert same == "1"
    if fused:
        assert int(n) == 1 and override == "None"
    else:
        assert int(n) >= 2 * (8 - 1) and override == "step"
