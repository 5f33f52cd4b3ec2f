"""Pins for the oracle's compressed AllReduce with error feedback: the pages'
Table 3 / Table 4 trace, the telescoping identity of error feedback, the
blockwise INT8 error bound, an exact case, and the compression-ratio closed
form."""
import json
import os

import numpy as np
import pytest

from ring_allreduce_rank_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    with open(os.path.join(GOLD, "error_feedback_table4.json")) as f:
        return json.load(f)


def test_table4_error_feedback_trace(oracle_mod):
    """Collective Communication, Table 4: v_t, e_{t+1} and the running total."""
    t = _table()
    e = [np.zeros(1, np.float32)]
    cum = 0.0
    for step, g in enumerate(t["g"]):
        assert abs(float(e[0][0]) - t["table4_e"][step]) < 1e-6
        assert abs(float(np.float32(g) + e[0][0]) - t["table4_g_plus_e"][step]) < 1e-6
        out, e = oracle_mod.allreduce_compressed([np.array([g], np.float32)], e, "sum", "threshold", 0,
                                                 t["threshold"])
        assert float(out[0][0]) == t["table4_v"][step]
        assert abs(float(e[0][0]) - t["table4_e_next"][step]) < 1e-6
        cum += float(out[0][0])
        assert cum == t["table4_cumulative_v"][step]


def test_table3_without_residual_path_transmits_nothing(oracle_mod):
    """Collective Communication, Table 3: the same compressor with the
    residual dropped every step sends 0 five times."""
    t = _table()
    sent = []
    for g in t["g"]:
        out, _ = oracle_mod.allreduce_compressed([np.array([g], np.float32)], [np.zeros(1, np.float32)], "sum",
                                                 "threshold", 0, t["threshold"])
        sent.append(float(out[0][0]))
    assert sent == t["table3_transmitted"]
    np.testing.assert_allclose(np.cumsum(t["g"]), t["table3_cumulative_true"], atol=1e-12)


def test_int8_block_ratio_closed_form():
    """Blockwise INT8: d bytes of codes plus 4 bytes of scale per block of b,
    ratio 4b/(b+4), printed as 3.88 for b = 128."""
    t = _table()
    b = 128
    assert round(4 * b / (b + 4), 2) == t["int8_block128_ratio"]


@pytest.mark.parametrize("block", [64, 128])
def test_int8_quantization_error_bound(oracle_mod, block):
    """|u - v| <= s/2 per element (s = block max / 127), up to fp32 rounding
    of the scale and product."""
    N, K = 1, 10_000
    g = W.normal_fp32(N, K, std=0.01, seed_base=3)
    e0 = [W.normal_fp32(1, K, std=0.001, seed_base=4)[0]]
    out, e1 = oracle_mod.allreduce_compressed(list(g), e0, "sum", "int8_block", block)
    u = (g[0] + e0[0]).astype(np.float64)
    v = out[0].astype(np.float64)
    for b0 in range(0, K, block):
        sl = slice(b0, b0 + block)
        s = np.abs(u[sl]).max() / 127.0
        q = v[sl] / s
        assert np.all(np.abs(q - np.round(q)) < 1e-3) and np.all(np.abs(q) <= 127.001)
        assert np.all(np.abs(u[sl] - v[sl]) <= 0.5 * s * (1 + 2 ** -20) + 1e-12)
    np.testing.assert_allclose(e1[0], (u - v), atol=1e-9)


def test_error_feedback_telescopes(oracle_mod):
    """sum_t v_t = sum_t g_t + e_1 - e_{T+1} (Collective Communication, the
    telescoping sum under Definition 1.4), up to fp32 rounding."""
    K, T = 4096, 20
    e = [np.zeros(K, np.float32)]
    sv = np.zeros(K)
    sg = np.zeros(K)
    for t in range(T):
        g = W.normal_fp32(1, K, std=0.01, seed_base=100 + t)
        out, e = oracle_mod.allreduce_compressed(list(g), e, "sum", "int8_block", 128)
        sv += out[0]
        sg += g[0]
    assert np.max(np.abs(sv - (sg - e[0]))) < 1e-6


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_exact_when_every_block_spans_127(oracle_mod, dtype, op):
    """Integer inputs whose every block holds a +-127 quantize exactly (s = 1):
    the residual stays 0 and the result is the fp32 ring AllReduce rounded
    to the buffer type."""
    N, K, b = 4, 1000, 128
    g = W.integers_fp32(N, K, seed=9, lo=-100, hi=100)
    g[:, ::b] = 127.0
    if dtype == "bf16":
        grads = [W.to_bf16_bits(r) for r in g]  # integers up to 127 are exact in bf16
    else:
        grads = list(g)
    res = [np.zeros(K, np.float32) for _ in range(N)]
    out, e = oracle_mod.allreduce_compressed(grads, res, op, "int8_block", b)
    ring, _ = oracle_mod.ring_allreduce(list(g), op)
    want = W.to_bf16_bits(ring[0]) if dtype == "bf16" else ring[0]
    for r in range(N):
        np.testing.assert_array_equal(out[r], want)
        assert not np.any(e[r])
