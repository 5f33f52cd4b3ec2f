"""GPU parity for the compressed AllReduce with error feedback: the pages'
Table 4 trace, and several consecutive steps of blockwise INT8 and the 1-bit
threshold compressor against the oracle, gradients and residuals bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)


def test_table4_trace_on_gpu():
    with open(os.path.join(GOLD, "error_feedback_table4.json")) as f:
        t = json.load(f)
    g = torch.zeros(1, dtype=torch.float32, device=DEV)
    e = torch.zeros(1, dtype=torch.float32, device=DEV)
    cum = 0.0
    for step, gv in enumerate(t["g"]):
        g.fill_(gv)
        ccl.ccl_allreduce_compressed([g], [e], op="sum", comp="threshold", threshold=t["threshold"])
        torch.cuda.synchronize()
        assert float(g.item()) == t["table4_v"][step]
        assert abs(float(e.item()) - t["table4_e_next"][step]) < 1e-6
        cum += float(g.item())
        assert cum == t["table4_cumulative_v"][step]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("comp,block", [("int8_block", 128), ("int8_block", 64), ("threshold", 0)])
@pytest.mark.parametrize("N,K", [(1, 100), (2, 4099), (3, 128 * 7), (4, 70001), (5, 33), (8, 70000), (8, 65),
                                 (16, 20011)])
def test_compressed_steps_match_oracle(N, K, comp, block, op, dtype):
    std = 0.01
    grads_h = [W.to_bf16_bits(r) for r in W.normal_fp32(N, K, std=std, seed_base=N + K)] if dtype == "bf16" \
        else list(W.normal_fp32(N, K, std=std, seed_base=N + K))
    res_h = [np.zeros(K, np.float32) for _ in range(N)]
    res = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    thr = 0.01
    for step in range(3):
        # a fresh gradient every step; the residual carries over
        if step:
            grads_h = [W.to_bf16_bits(r) for r in W.normal_fp32(N, K, std=std, seed_base=100 * step + N)] \
                if dtype == "bf16" else list(W.normal_fp32(N, K, std=std, seed_base=100 * step + N))
        grads = [to_dev(g) for g in grads_h]
        want_g, res_h = oracle.allreduce_compressed(grads_h, res_h, op, comp, block or 128, thr)
        ccl.ccl_allreduce_compressed(grads, res, op=op, comp=comp, block=block or 128, threshold=thr)
        torch.cuda.synchronize()
        for r in range(N):
            assert_bits_equal(bits(grads[r]), want_g[r], "step %d grads rank %d" % (step, r))
            assert_bits_equal(bits(res[r]), res_h[r], "step %d residual rank %d" % (step, r))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_compressed_special_values_and_unaligned(dtype):
    N, K = 4, 1000
    x = W.mixed_bf16(N, K, seed_base=5) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=5)
    res_h = [np.zeros(K, np.float32) for _ in range(N)]
    want_g, want_e = oracle.allreduce_compressed(list(x), res_h, "sum", "int8_block", 128)
    grads = [to_dev(r, pad_elems=1) for r in x]
    res = [torch.zeros(K + 1, dtype=torch.float32, device=DEV)[1:] for _ in range(N)]
    ccl.ccl_allreduce_compressed(grads, res, op="sum", comp="int8_block", block=128)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(grads[r]), want_g[r], "special grads rank %d" % r)
        assert_bits_equal(bits(res[r]), want_e[r], "special residual rank %d" % r)


def _tie_blocks(dtype, n_blocks, seed):
    """Gradients and residuals whose u = g + e sit exactly on, or within a few
    ulps of, the half-integer ties of u / s (INT8, blocks of 128): the cases
    where rounding u * (1/s) could differ from rounding the exact quotient."""
    g = np.random.Generator(np.random.PCG64(seed))
    grads = np.zeros(n_blocks * 128, np.float32)
    res = np.zeros(n_blocks * 128, np.float32)
    for b in range(n_blocks):
        blk = slice(b * 128, (b + 1) * 128)
        k = g.integers(-126, 126, size=128).astype(np.float32)
        if dtype == "bf16" or b % 2 == 0:
            # max |u| = 127: the scale is exactly 1, k + 1/2 is a tie
            vals = k + np.float32(0.5)
            vals[0] = np.float32(127.0)
            jitter = g.choice(np.array([0.0, 2.0 ** -12, -2.0 ** -12, 2.0 ** -20, -2.0 ** -20, 2.0 ** -16],
                                       np.float32), size=128)
            jitter[0] = 0.0
            grads[blk] = vals
            res[blk] = jitter
        else:
            top = np.float32(g.uniform(20.0, 300.0))
            s = np.float32(top / np.float32(127.0))
            vals = ((k + np.float32(0.5)) * s).astype(np.float32)
            step = g.choice(np.array([-2, -1, 0, 1, 2]), size=128)
            vals = np.nextafter(vals, np.where(step > 0, np.inf, -np.inf).astype(np.float32)) * (step != 0) + \
                vals * (step == 0)
            vals = vals.astype(np.float32)
            vals[0] = top
            grads[blk] = vals
    if dtype == "bf16":
        return W.to_bf16_bits(grads), res
    return grads, res


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N", [1, 3, 8])
def test_compressed_ties_and_near_ties(dtype, N):
    nb = 96
    gs, rs = zip(*[_tie_blocks(dtype, nb, seed=17 * N + r) for r in range(N)])
    want_g, want_e = oracle.allreduce_compressed(list(gs), list(rs), "sum", "int8_block", 128)
    grads = [to_dev(x) for x in gs]
    res = [torch.from_numpy(e.copy()).to(DEV) for e in rs]
    ccl.ccl_allreduce_compressed(grads, res, op="sum", comp="int8_block", block=128)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(grads[r]), want_g[r], "ties grads rank %d" % r)
        assert_bits_equal(bits(res[r]), want_e[r], "ties residual rank %d" % r)
