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


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


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


def test_threshold_error_feedback_cycle_constant_gradient(oracle_mod):
    """The error accumulator under a constant gradient (the pages' exercise on
    e_t's steady state, with g = 0.25 so every value is exact in binary).  The
    greedy compressor sends 1 when g + e >= 0.5 (Collective Communication,
    Table 3: only values >= 0.5 are sent), so by hand: u = 0.25, 0.5, -0.25, 0,
    then the cycle repeats -- one 1 every four steps, the long-run average of
    what is sent equals g, and the residual stays in [-0.5, 0.5)."""
    e = [np.zeros(1, np.float32)]
    sent, res = [], []
    for _ in range(12):
        out, e = oracle_mod.allreduce_compressed([np.array([0.25], np.float32)], e, "sum", "threshold", 0, 0.5)
        sent.append(float(out[0][0]))
        res.append(float(e[0][0]))
    assert sent == [0.0, 1.0, 0.0, 0.0] * 3
    assert res == [0.25, -0.5, -0.25, 0.0] * 3
    assert sum(sent) / len(sent) == 0.25


def test_int8_rounds_ties_to_even(oracle_mod):
    """Blockwise INT8 takes q = round(u / s) with ties to even (the IEEE
    default rounding).  With max|u| = 127 the scale is exactly 1, so each
    u = k + 1/2 sits on a tie and v must be numpy's rint(u)."""
    halves = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 10.5, 11.5, -126.5, 125.5], np.float32)
    u = np.zeros(128, np.float32)
    u[0] = 127.0
    u[1:1 + halves.size] = halves
    out, e = oracle_mod.allreduce_compressed([u], [np.zeros(128, np.float32)], "sum", "int8_block", 128, 0.0)
    v = out[0]
    np.testing.assert_array_equal(v[1:1 + halves.size], np.rint(halves))
    np.testing.assert_array_equal(np.signbit(v[1:1 + halves.size]), np.signbit(np.rint(halves)))
    np.testing.assert_array_equal(e[0], u - v)
    assert v[0] == 127.0


def test_int8_nan_in_a_block_poisons_only_that_block(oracle_mod):
    """A NaN anywhere in a block makes that block's scale NaN, so every value
    it sends and every residual it keeps is NaN; the next block is untouched
    (the reading of s = max|u| / 127 when the block holds a NaN)."""
    g = W.normal_fp32(1, 256, seed_base=3)[0]
    g[5] = np.float32("nan")
    out, e = oracle_mod.allreduce_compressed([g], [np.zeros(256, np.float32)], "sum", "int8_block", 128, 0.0)
    assert np.isnan(out[0][:128]).all() and np.isnan(e[0][:128]).all()
    assert not np.isnan(out[0][128:]).any() and not np.isnan(e[0][128:]).any()
    clean, _ = oracle_mod.allreduce_compressed([g[128:].copy()], [np.zeros(128, np.float32)], "sum", "int8_block",
                                               128, 0.0)
    np.testing.assert_array_equal(out[0][128:], clean[0])


# ---------------------------------------------------------------- Top-k sparsification

def test_topk_ratio_closed_form():
    """Top-k with fp32 values and int32 indices sends 8 bytes per kept
    element: ratio 4d / (8 K_top) = d / (2 K_top), printed as 500x (not 1000x)
    for K_top = 0.001 d."""
    t = _table()
    d = 1_000_000
    k = int(round(t["topk_kept_fraction"] * d))
    assert d // k == t["topk_kept_fraction_naive_ratio"]
    assert 4 * d / (8 * k) == t["topk_ratio"]


def _topk_numpy(u, k):
    """TopK(u) = u * 1[|u| >= |u|_(k)] with numpy's sort (every value tied
    with the k-th largest magnitude is kept); k = 0 keeps nothing."""
    a = np.abs(u.astype(np.float64))
    if k == 0:
        return np.zeros_like(u)
    kth = np.sort(a)[::-1][min(k, a.size) - 1]
    return np.where(a >= kth, u, np.float32(0)).astype(np.float32)


def _int_grads(dtype, N, K, seed, lo=-20, hi=20):
    g = W.integers_fp32(N, K, seed=seed, lo=lo, hi=hi)
    grads = [W.to_bf16_bits(r) for r in g] if dtype == "bf16" else list(g)
    return g, grads


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("N,K,k", [(1, 50, 7), (3, 1000, 10), (4, 4096, 41), (5, 333, 333), (2, 100, 1),
                                   (3, 64, 500)])
def test_topk_matches_the_definition_on_integers(oracle_mod, dtype, op, N, K, k):
    """Integer gradients and residuals, with many equal magnitudes so that the
    k-th largest is tied: every sum is exact, so the result must be the
    brute-force sum of numpy's TopK of each rank's u = g + e (AVG: numpy's
    float32 quotient by N), rounded to the gradient type, and each residual
    must be u minus what that rank sent.  At least k values are sent per rank."""
    g, grads = _int_grads(dtype, N, K, seed=N * 1000 + K + k)
    e0 = list(W.integers_fp32(N, K, seed=7 + k, lo=-3, hi=3))
    out, e1 = oracle_mod.allreduce_compressed(grads, e0, op, "topk", k=k)
    u = [g[r] + e0[r] for r in range(N)]
    v = [_topk_numpy(u[r], k) for r in range(N)]
    S = np.sum(np.stack(v).astype(np.float64), axis=0).astype(np.float32)
    want = S / np.float32(N) if op == "avg" else S
    want = W.to_bf16_bits(want) if dtype == "bf16" else want
    for r in range(N):
        np.testing.assert_array_equal(_bits(out[r]), _bits(want))
        np.testing.assert_array_equal(_bits(e1[r]), _bits((u[r] - v[r]).astype(np.float32)))
        assert np.count_nonzero(np.abs(u[r]) >= np.sort(np.abs(u[r]))[::-1][min(k, K) - 1]) >= min(k, K)


def test_topk_keeps_exactly_k_distinct_magnitudes(oracle_mod):
    """Distinct magnitudes: exactly k values leave each rank, the k largest."""
    N, K, k = 3, 5000, 37
    x = W.normal_fp32(N, K, seed_base=21)
    out, e1 = oracle_mod.allreduce_compressed(list(x), [np.zeros(K, np.float32)] * N, "sum", "topk", k=k)
    for r in range(N):
        sent = x[r] - e1[r]
        assert np.count_nonzero(sent) == k
        top = np.argsort(-np.abs(x[r]), kind="stable")[:k]
        np.testing.assert_array_equal(np.sort(np.nonzero(sent)[0]), np.sort(top))


def test_topk_k_zero_sends_nothing_and_k_all_sends_everything(oracle_mod):
    N, K = 4, 999
    g, grads = _int_grads("fp32", N, K, seed=3)
    e0 = [np.zeros(K, np.float32) for _ in range(N)]
    out, e1 = oracle_mod.allreduce_compressed(grads, e0, "sum", "topk", k=0)
    for r in range(N):
        np.testing.assert_array_equal(_bits(out[r]), np.zeros(K, np.uint32))  # +0 everywhere
        np.testing.assert_array_equal(_bits(e1[r]), _bits(g[r]))
    for k in (K, K + 5):
        out, e1 = oracle_mod.allreduce_compressed(grads, e0, "sum", "topk", k=k)
        S = np.sum(g.astype(np.float64), axis=0).astype(np.float32)
        for r in range(N):
            np.testing.assert_array_equal(out[r], S)
            assert not np.any(e1[r])


def test_topk_nan_counts_as_the_largest_magnitude(oracle_mod):
    """A NaN in u is ordered above every number, so with k = 1 it is the one
    value its rank sends: the result is NaN there on every rank, that rank
    keeps every other value as residual, and the residual at the NaN is NaN."""
    N, K = 3, 300
    x = W.normal_fp32(N, K, seed_base=5)
    x[1][17] = np.float32("nan")
    out, e1 = oracle_mod.allreduce_compressed(list(x), [np.zeros(K, np.float32)] * N, "sum", "topk", k=1)
    for r in range(N):
        assert np.isnan(out[r][17])
        assert out[r].view(np.uint32)[17] == 0x7FFFFFFF
    assert np.isnan(e1[1][17])
    rest = np.arange(K) != 17
    np.testing.assert_array_equal(e1[1][rest], x[1][rest])


def test_topk_error_feedback_telescopes_exactly(oracle_mod):
    """sum_t v_t = sum_t g_t + e_1 - e_{T+1} (Collective Communication, the
    telescoping sum under Definition 1.4).  Gradients on a 1/8 grid keep every
    value exact, so the identity holds with equality."""
    K, T, k = 512, 40, 32
    e = [np.zeros(K, np.float32)]
    sv = np.zeros(K)
    sg = np.zeros(K)
    g0 = np.random.Generator(np.random.PCG64(11))
    for t in range(T):
        g = (g0.integers(-16, 17, size=K) / 8.0).astype(np.float32)
        out, e = oracle_mod.allreduce_compressed([g], e, "sum", "topk", k=k)
        sv += out[0]
        sg += g
    np.testing.assert_array_equal(sv, sg - e[0].astype(np.float64))
