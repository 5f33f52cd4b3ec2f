"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Nothing here runs the CUDA library.  Each test names what pins it: a value the
pages print (tests/golden/), a hand-derived IEEE result, a closed form, an
invariant, a library routine for a special case, or brute force on tiny inputs.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

from ring_allreduce_rank_gb300 import workloads as W
from accuracy import error_figures, report

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _fp32(rows):
    return [np.asarray(r, dtype=np.float32) for r in rows]


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


# ---------------------------------------------------------------- worked examples

@pytest.mark.parametrize("case", _load("worked_examples.json")["cases"], ids=lambda c: c["name"])
def test_worked_examples(oracle_mod, case):
    """Values printed by the pages (tests/golden/worked_examples.json)."""
    ins = _fp32(case["inputs"])
    exp = _fp32(case["expected"])
    kind = case["collective"]
    if kind == "allreduce":
        outs, _ = oracle_mod.ring_allreduce(ins, case["op"])
        closed = oracle_mod.ring_allreduce_closed(ins, case["op"])
        for o, c, e in zip(outs, closed, exp):
            np.testing.assert_array_equal(o, e)
            np.testing.assert_array_equal(c, e)
    elif kind == "reduce_scatter":
        outs = oracle_mod.reduce_scatter(ins, case["op"])
        for o, e in zip(outs, exp):
            np.testing.assert_array_equal(o, e)
    elif kind == "broadcast":
        outs = oracle_mod.broadcast(ins, case["root"])
        for o, e in zip(outs, exp):
            np.testing.assert_array_equal(o, e)
    elif kind == "allgather":
        K = exp[0].size
        outs = oracle_mod.allgather(ins, K)
        for o, e in zip(outs, exp):
            np.testing.assert_array_equal(o, e)
    elif kind == "alltoall":
        N = len(ins)
        blk = ins[0].size // N
        counts = np.full((N, N), blk)
        outs = oracle_mod.alltoallv(ins, counts)
        for o, e in zip(outs, exp):
            np.testing.assert_array_equal(o, e)
    elif kind == "reduce":
        outs = oracle_mod.reduce(ins, case["root"], case["op"])
        for o, e in zip(outs, exp):
            np.testing.assert_array_equal(o, e)
    elif kind == "gather":
        out = oracle_mod.gather(ins, exp[0].size)
        np.testing.assert_array_equal(out, exp[0])
    else:
        raise AssertionError(kind)


# ---------------------------------------------------------------- ring schedule

def test_schedule_matches_printed_n4_trace(oracle_mod):
    """AllReduce survey, 'why split into N pieces': the printed N=4 step listing."""
    g = _load("ring_schedule_n4.json")
    tab = oracle_mod.ring_schedule(g["N"])
    np.testing.assert_array_equal(tab[0, :, :, 0], np.array(g["rs_send_chunk"]))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 16, 64])
def test_schedule_invariants(oracle_mod, N):
    """Each step is a permutation of chunks, the receiver gets exactly what its
    left neighbour sends, a rank never receives the chunk it sends in the same
    step, every chunk visits every rank once per phase, and after the first
    phase rank i holds chunk (i+1) mod N (Collectives and sharded matmul,
    'ring ReduceScatter'; AllReduce survey, phase 1)."""
    tab = oracle_mod.ring_schedule(N)
    assert tab.shape == (2, max(N - 1, 0), N, 3)
    for ph in range(2):
        for s in range(N - 1):
            send, recv, src = tab[ph, s, :, 0], tab[ph, s, :, 1], tab[ph, s, :, 2]
            assert sorted(send) == list(range(N))
            assert sorted(recv) == list(range(N))
            for i in range(N):
                assert src[i] == (i - 1) % N
                assert recv[i] == send[src[i]]
                assert recv[i] != send[i] or N == 1
    # contributions: chunk c has visited ranks c, c+1, ... after the RS phase,
    # and the last receiver (the holder) is (c-1) mod N = rank i holds (i+1).
    holder = {}
    for c in range(N):
        visited = [c]  # the chunk starts at rank c (step 0 send)
        for s in range(N - 1):
            for i in range(N):
                if tab[0, s, i, 1] == c:
                    visited.append(i)
        assert sorted(visited) == list(range(N))
        holder[c] = visited[-1]
    for c in range(N):
        if N > 1:
            assert holder[c] == (c - 1) % N


@pytest.mark.parametrize("N", [2, 3, 4, 5, 7])
def test_traffic_count(oracle_mod, N):
    """Lesson 3 reference solution: each rank sends 2(N-1)K/N elements (checked
    there for N = 2, 3, 4, 5, 7)."""
    K = 8 * 16 * N
    x = W.normal_fp32(N, K, seed_base=0)
    _, sent = oracle_mod.ring_allreduce(list(x))
    assert sent == [2 * (N - 1) * K // N] * N


def test_traffic_count_ragged(oracle_mod):
    """Ragged K: a rank sends, over both phases, every chunk except the one it
    last receives in each phase; total = sum over the 2(N-1) step entries."""
    N, K = 5, 23
    _, sent = oracle_mod.ring_allreduce(list(W.normal_fp32(N, K)))
    off, ln = oracle_mod.partition(K, N)
    tab = oracle_mod.ring_schedule(N)
    for i in range(N):
        exp = sum(ln[tab[ph, s, i, 0]] for ph in range(2) for s in range(N - 1))
        assert sent[i] == exp


# ---------------------------------------------------------------- partition

@pytest.mark.parametrize("K,N", [(0, 3), (1, 4), (5, 3), (16, 4), (16777259, 16), (67108864, 8), (7, 7), (3, 8)])
def test_partition(oracle_mod, K, N):
    off, ln = oracle_mod.partition(K, N)
    assert sum(ln) == K
    assert off[0] == 0
    for c in range(1, N):
        assert off[c] == off[c - 1] + ln[c - 1]
    assert max(ln) - min(ln) <= 1
    assert ln == sorted(ln, reverse=True)  # remainder goes to the first chunks


def test_partition_c3_sizes(oracle_mod):
    """16,777,259 over 16 ranks: 11 chunks of 1,048,579 then 5 of 1,048,578."""
    _, ln = oracle_mod.partition(16777259, 16)
    assert ln == [1048579] * 11 + [1048578] * 5


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rne_against_torch_all_top_halves(oracle_mod):
    """Every fp32 sign/exponent/high-mantissa pattern (all 65,536 top halves)
    combined with the low halves that decide rounding (zero, just below half,
    exactly half, just above half, maximum, and a few others), against torch's
    CPU float->bfloat16 conversion (a library round-to-nearest-even).  NaNs are
    excluded here (torch returns its own canonical NaN) and pinned separately."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x3fff, 0x7fff, 0x8000, 0x8001, 0xbfff, 0xffff, 0x1234, 0xc000], dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    f = pats.view(np.float32)
    keep = ~np.isnan(f)
    pats = pats[keep]
    ref = torch.from_numpy(pats.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.round_bf16_array(pats)
    np.testing.assert_array_equal(got, ref)


def test_bf16_rne_against_torch_random(oracle_mod):
    pats = np.random.Generator(np.random.PCG64(7)).integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    pats = pats[~np.isnan(pats.view(np.float32))]
    ref = torch.from_numpy(pats.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle_mod.round_bf16_array(pats), ref)


def test_bf16_nan_rule(oracle_mod):
    """NaN keeps its sign and top payload bits and becomes quiet (the
    library's reading; the pages do not mention NaN)."""
    assert oracle_mod.round_bf16(0x7fffffff) == 0x7fff
    assert oracle_mod.round_bf16(0x7fc00000) == 0x7fc0
    assert oracle_mod.round_bf16(0x7f800001) == 0x7fc0
    assert oracle_mod.round_bf16(0xffa00000) == 0xffe0


# ---------------------------------------------------------------- hand-derived rounding

@pytest.mark.parametrize("case", _load("rounding_cases.json")["cases"], ids=lambda c: c["name"])
def test_rounding_cases(oracle_mod, case):
    dt = np.uint16 if case["dtype"] == "bf16" else np.uint32
    ins = [np.array([int(x, 16) for x in row], dtype=dt) for row in case["inputs_bits"]]
    if case["dtype"] == "fp32":
        ins = [a.view(np.float32) for a in ins]
    exp = np.array([int(x, 16) for x in case["expected_bits"]], dtype=dt)
    outs, _ = oracle_mod.ring_allreduce(ins, case["op"])
    closed = oracle_mod.ring_allreduce_closed(ins, case["op"])
    for o, c in zip(outs, closed):
        np.testing.assert_array_equal(_bits(o), exp)
        np.testing.assert_array_equal(_bits(c), exp)


# ---------------------------------------------------------------- two formulations agree

def _inputs(dtype, N, K, seed):
    if dtype == "bf16":
        return list(W.mixed_bf16(N, K, seed_base=seed))
    return list(W.mixed_fp32(N, K, seed_base=seed))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min", "avg_premul"])
@pytest.mark.parametrize("N,K", [(1, 7), (2, 9), (3, 3), (3, 0), (4, 37), (5, 3), (7, 101), (8, 1000), (16, 517)])
def test_step_simulation_equals_closed_form(oracle_mod, dtype, op, N, K):
    """The step-by-step ring simulation and the closed-form fold are written
    independently; they must agree bit for bit, on every rank, with special
    values (signed zeros, subnormals, inf, NaN) mixed in."""
    x = _inputs(dtype, N, K, seed=N * 1000 + K)
    steps, _ = oracle_mod.ring_allreduce(x, op)
    closed = oracle_mod.ring_allreduce_closed(x, op)
    for r in range(N):
        np.testing.assert_array_equal(_bits(steps[r]), _bits(closed[r]))
        np.testing.assert_array_equal(_bits(steps[r]), _bits(steps[0]))
    if K:
        idx = np.arange(K, dtype=np.uint64)[::3]
        np.testing.assert_array_equal(_bits(oracle_mod.ring_allreduce_at(x, idx, op)), _bits(closed[0])[idx.astype(np.int64)])


# ---------------------------------------------------------------- exact special cases

def test_integer_inputs_exact_c1(oracle_mod):
    """Integer-valued inputs (|x| <= 8, N = 4): every partial sum is exact, so
    the ring result equals the brute-force fp64 sum."""
    x = W.integers_fp32(4, 4096, seed=0)
    outs, _ = oracle_mod.ring_allreduce(list(x))
    ref = x.astype(np.float64).sum(axis=0)
    for o in outs:
        np.testing.assert_array_equal(o.astype(np.float64), ref)
    y64, _ = oracle_mod.sum_f64(list(x))
    np.testing.assert_array_equal(y64, ref)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_n1_identity_and_n2_single_add(oracle_mod, dtype):
    """N = 1: the buffer is unchanged.  N = 2: each element is one IEEE fp32
    addition rounded to the buffer type -- numpy's float32 add, then torch's
    bf16 conversion, are the library routines for that."""
    K = 4099
    x = _inputs(dtype, 2, K, seed=11)
    one, _ = oracle_mod.ring_allreduce([x[0]])
    np.testing.assert_array_equal(_bits(one[0]), _bits(x[0]))
    two, _ = oracle_mod.ring_allreduce(x)
    if dtype == "fp32":
        with np.errstate(invalid="ignore", over="ignore"):
            ref = (x[0] + x[1]).astype(np.float32)
        got = two[0]
    else:
        a, b = W.bf16_bits_to_f32(x[0]), W.bf16_bits_to_f32(x[1])
        ref = W.to_bf16_bits(a + b)
        got = two[0]
    rb = _bits(ref)
    gb = _bits(got)
    fin = ~np.isnan(W.bf16_bits_to_f32(rb) if dtype == "bf16" else ref)
    np.testing.assert_array_equal(gb[fin], rb[fin])
    # NaN results are the canonical quiet NaN
    canon = 0x7fff if dtype == "bf16" else 0x7fffffff
    assert np.all(gb[~fin] == canon)


def test_max_is_order_free_brute_force(oracle_mod):
    """MAX takes no rounding: it equals numpy's maximum over ranks (finite,
    non-zero inputs, where the tie rule for signed zeros cannot matter)."""
    for dtype in ("fp32", "bf16"):
        N, K = 7, 333
        x = W.normal_fp32(N, K, seed_base=3)
        if dtype == "bf16":
            xb = [W.to_bf16_bits(r) for r in x]
            outs, _ = oracle_mod.ring_allreduce(xb, "max")
            ref = W.to_bf16_bits(np.max(np.stack([W.bf16_bits_to_f32(r) for r in xb]), axis=0))
            np.testing.assert_array_equal(outs[0], ref)
        else:
            outs, _ = oracle_mod.ring_allreduce(list(x), "max")
            np.testing.assert_array_equal(outs[0], x.max(axis=0))


def test_min_is_order_free_brute_force(oracle_mod):
    """MIN takes no rounding: it equals numpy's minimum over ranks."""
    N, K = 6, 401
    x = W.normal_fp32(N, K, seed_base=8)
    outs, _ = oracle_mod.ring_allreduce(list(x), "min")
    np.testing.assert_array_equal(outs[0], x.min(axis=0))
    xb = [W.to_bf16_bits(r) for r in x]
    outb, _ = oracle_mod.ring_allreduce(xb, "min")
    ref = W.to_bf16_bits(np.min(np.stack([W.bf16_bits_to_f32(r) for r in xb]), axis=0))
    np.testing.assert_array_equal(outb[0], ref)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min", "avg_premul"])
@pytest.mark.parametrize("N,K,root", [(1, 5, 0), (3, 5, 0), (4, 37, 3), (8, 1000, 5), (5, 3, 2)])
def test_reduce_is_allreduce_at_root_others_unchanged(oracle_mod, dtype, op, N, K, root):
    """AllReduce = Reduce + Broadcast (Lesson 3, core concepts): the root gets
    the AllReduce's bits, every other rank keeps its input."""
    x = _inputs(dtype, N, K, seed=N + K + root)
    red = oracle_mod.reduce(x, root, op)
    ar, _ = oracle_mod.ring_allreduce(x, op)
    bc = oracle_mod.broadcast(red, root)
    for r in range(N):
        np.testing.assert_array_equal(_bits(red[r]), _bits(ar[r] if r == root else x[r]))
        np.testing.assert_array_equal(_bits(bc[r]), _bits(ar[r]))


@pytest.mark.parametrize("N,K", [(1, 4), (3, 15), (4, 13), (8, 1000), (5, 3)])
def test_scatter_inverts_gather(oracle_mod, N, K):
    """Scatter is the inverse of Gather (Lesson 3, core concepts); both are
    the chunk partition read or written in rank order."""
    g = np.random.Generator(np.random.PCG64(K))
    full = g.integers(0, 1 << 16, size=K).astype(np.uint16)
    parts = oracle_mod.scatter(full, N)
    off, ln = oracle_mod.partition(K, N)
    for r in range(N):
        np.testing.assert_array_equal(parts[r], full[off[r]:off[r] + ln[r]])
    np.testing.assert_array_equal(oracle_mod.gather(parts, K), full)


def test_prod_exact_on_powers_of_two(oracle_mod):
    """Products of small powers of two are exact: PROD equals the brute-force product."""
    g = np.random.Generator(np.random.PCG64(5))
    N, K = 6, 200
    e = g.integers(-4, 5, size=(N, K))
    s = g.choice([-1.0, 1.0], size=(N, K))
    x = (s * np.exp2(e)).astype(np.float32)
    outs, _ = oracle_mod.ring_allreduce(list(x), "prod")
    np.testing.assert_array_equal(outs[0], np.prod(x.astype(np.float64), axis=0).astype(np.float32))
    xb = [W.to_bf16_bits(r) for r in x]
    outb, _ = oracle_mod.ring_allreduce(xb, "prod")
    np.testing.assert_array_equal(outb[0], W.to_bf16_bits(np.prod(x.astype(np.float64), axis=0).astype(np.float32)))


@pytest.mark.parametrize("N", [3, 5, 6, 7])
def test_avg_is_the_correctly_rounded_quotient(oracle_mod, N):
    """AVG divides the finished sum once by N.  With integer inputs every ring
    partial sum is exact, so the result must be the IEEE quotient S / N of the
    exact sum, computed here by numpy's float32 division.  For N not a power
    of two that differs from S * (1/N) for many S; the inputs include such S."""
    K = 4000
    x = [np.random.Generator(np.random.PCG64(N * 100 + r)).integers(-300, 300, size=K).astype(np.float32)
         for r in range(N)]
    S = np.sum(np.stack(x).astype(np.float64), axis=0).astype(np.float32)  # exact: |S| < 2^24
    want = S / np.float32(N)
    assert (want != S * (np.float32(1) / np.float32(N))).any()
    outs, _ = oracle_mod.ring_allreduce(x, "avg")
    for r in range(N):
        np.testing.assert_array_equal(outs[r].view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "prod", "avg", "avg_premul"])
@pytest.mark.parametrize("N,L", [(3, 7), (4, 16), (5, 3), (8, 9)])
def test_ring_order_is_rotation_equivariant(oracle_mod, dtype, op, N, L):
    """Chunk c is folded starting at rank c, so relabelling ranks and chunks by
    one step moves the result by one chunk: with x'_r[chunk c] =
    x_{r+1}[chunk c+1], AR(x')[chunk c] = AR(x)[chunk c+1] bit for bit (equal
    chunks of L elements, indices mod N).  An order whose start does not
    follow the chunk index breaks this for rounded, non-associative sums."""
    K = N * L
    x = _inputs(dtype, N, K, seed=N * 31 + L)
    xp = []
    for r in range(N):
        row = np.empty_like(x[r])
        for c in range(N):
            row[c * L:(c + 1) * L] = x[(r + 1) % N][((c + 1) % N) * L:((c + 1) % N + 1) * L]
        xp.append(row)
    y, _ = oracle_mod.ring_allreduce(x, op)
    yp, _ = oracle_mod.ring_allreduce(xp, op)
    for c in range(N):
        d = (c + 1) % N
        np.testing.assert_array_equal(_bits(yp[0][c * L:(c + 1) * L]), _bits(y[0][d * L:(d + 1) * L]))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min", "avg_premul"])
@pytest.mark.parametrize("N,K,threads", [(8, 1000, 8), (8, 1001, 3), (5, 37, 2), (16, 517, 16), (3, 2, 3), (1, 9, 1)])
def test_threaded_ring_equals_single_thread(oracle_mod, dtype, op, N, K, threads):
    """The CPU baseline's multi-core form (ranks on threads, a barrier per
    step) is the same computation: identical bits to the one-thread ring."""
    x = _inputs(dtype, N, K, seed=N * 7 + K)
    a, _ = oracle_mod.ring_allreduce(x, op)
    b = oracle_mod.ring_allreduce_threads(x, op, threads)
    for r in range(N):
        np.testing.assert_array_equal(_bits(b[r]), _bits(a[r]))


def test_avg_power_of_two_is_scaled_sum(oracle_mod):
    """For N = 8, dividing by 8 is an exact exponent shift (barring
    subnormals), so AVG equals the SUM result times 2^-3."""
    N, K = 8, 4096
    x = list(W.normal_bf16(N, K, std=1e-3, seed_base=0))
    s, _ = oracle_mod.ring_allreduce(x, "sum")
    a, _ = oracle_mod.ring_allreduce(x, "avg")
    sf = W.bf16_bits_to_f32(s[0]).astype(np.float64)
    af = W.bf16_bits_to_f32(a[0]).astype(np.float64)
    np.testing.assert_array_equal(af, sf / 8.0)


@pytest.mark.parametrize("dtype,op,N,K,rtol", [("bf16", "avg", 8, 65536, 1e-2), ("bf16", "sum", 16, 20000, 1e-2),
                                                ("bf16", "sum", 64, 65536, 1e-2),
                                                ("fp32", "sum", 16, 20011, 1e-5), ("fp32", "avg", 5, 9999, 1e-5)])
def test_error_bound_against_fp64(oracle_mod, dtype, op, N, K, rtol):
    """Accuracy against the plain definition y = sum_r x_r in fp64.
    Elementwise, recursive summation with a rounding after each of the N-1 hops
    obeys |y - y64| <= (N-1) u sum|x| (u = 2^-8 for bf16, on top of fp32's
    2^-24), plus one rounding for the AVG division.  The stated relative
    tolerance (1e-2 bf16, 1e-5 fp32) holds normwise, ||y - y64|| / ||y64||:
    elementwise relative error is unbounded where the sum cancels."""
    if dtype == "bf16":
        x = list(W.normal_bf16(N, K, std=1e-3, seed_base=1))
        u = 2.0 ** -8 + 2.0 ** -24
    else:
        x = list(W.uniform_fp32(N, K, seed_base=1))
        u = 2.0 ** -24
    outs, _ = oracle_mod.ring_allreduce(x, op)
    y = W.bf16_bits_to_f32(outs[0]) if dtype == "bf16" else outs[0]
    y64, absum = oracle_mod.sum_f64(x, op)
    err = np.abs(y.astype(np.float64) - y64)
    bound = (N - 1 + (1 if op == "avg" else 0)) * u * absum * (1 + 1e-6) + 1e-300
    assert np.all(err <= bound)
    assert np.linalg.norm(err) <= rtol * np.linalg.norm(y64)
    fig = error_figures(y, y64, absum)
    report("oracle %s %s N=%d K=%d" % (dtype, op, N, K), fig)
    assert fig["elementwise"] <= (N - 1 + (1 if op == "avg" else 0)) * u * (1 + 1e-6)


# ---------------------------------------------------------------- pre-multiplied AVG

def _prescaled(x, dtype, N):
    """Each contribution times the float32 reciprocal of N, rounded to the
    buffer type: numpy's float32 division and multiplication (IEEE, round to
    nearest even) and torch's bf16 conversion."""
    inv = np.float32(1) / np.float32(N)
    with np.errstate(invalid="ignore", over="ignore", under="ignore"):
        if dtype == "bf16":
            return [W.to_bf16_bits(W.bf16_bits_to_f32(r) * inv) for r in x]
        return [(np.asarray(r, dtype=np.float32) * inv).astype(np.float32) for r in x]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N", [3, 5, 6, 7, 12])
def test_avg_premul_is_the_sum_of_prescaled_contributions(oracle_mod, dtype, N):
    """NCCL's pre-multiplied AVG (Collective Communication, libraries section)
    scales every contribution by 1/N before the ring sums them and divides
    nothing at the end: the result must be the ring SUM of the contributions
    scaled here independently, special values included.  For N not a power of
    two it must differ from AVG's single division somewhere."""
    K = 3001
    x = _inputs(dtype, N, K, seed=N * 17)
    p, _ = oracle_mod.ring_allreduce(x, "avg_premul")
    s, _ = oracle_mod.ring_allreduce(_prescaled(x, dtype, N), "sum")
    a, _ = oracle_mod.ring_allreduce(x, "avg")
    for r in range(N):
        np.testing.assert_array_equal(_bits(p[r]), _bits(s[r]))
    assert (_bits(p[0]) != _bits(a[0])).any()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_avg_premul_power_of_two_equals_avg(oracle_mod, dtype, N):
    """For N a power of two, 1/N is exact and multiplying by it only shifts
    the exponent; rounding commutes with that shift away from the subnormal
    range, so scaling before the sum and dividing after it give the same bits.
    N = 1 leaves every value unchanged."""
    K = 4099
    x = list(W.normal_bf16(N, K, std=1e-3, seed_base=N)) if dtype == "bf16" else \
        list(W.normal_fp32(N, K, seed_base=N))
    p, _ = oracle_mod.ring_allreduce(x, "avg_premul")
    a, _ = oracle_mod.ring_allreduce(x, "avg")
    for r in range(N):
        np.testing.assert_array_equal(_bits(p[r]), _bits(a[r]))
    if N == 1:
        np.testing.assert_array_equal(_bits(p[0]), _bits(x[0]))


@pytest.mark.parametrize("dtype,N,K", [("bf16", 8, 20000), ("bf16", 6, 20000), ("fp32", 5, 9999),
                                       ("fp32", 16, 5000)])
def test_avg_premul_error_bound_against_fp64(oracle_mod, dtype, N, K):
    """Against the fp64 mean m = sum_r x_r / N: each scaled contribution
    carries the reciprocal's and the product's fp32 roundings (and, for bf16,
    one rounding to bf16); the N-1 hops add one rounding each.  So
    |y - m| <= gamma_(N+1) * sum_r |x_r| / N, with gamma_n = n u / (1 - n u)
    and u the per-rounding unit (2^-8 + 2^-24 for bf16, 2^-24 for fp32)."""
    if dtype == "bf16":
        x = list(W.normal_bf16(N, K, std=1e-3, seed_base=3))
        u = 2.0 ** -8 + 2.0 ** -24
    else:
        x = list(W.uniform_fp32(N, K, seed_base=3))
        u = 2.0 ** -24
    outs, _ = oracle_mod.ring_allreduce(x, "avg_premul")
    y = W.bf16_bits_to_f32(outs[0]) if dtype == "bf16" else outs[0]
    m, absum = oracle_mod.sum_f64(x, "avg_premul")
    n = N + 1
    bound = n * u / (1 - n * u) * absum * (1 + 1e-9) + 1e-300
    assert np.all(np.abs(y.astype(np.float64) - m) <= bound)


# ---------------------------------------------------------------- composition invariants

@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "avg_premul"])
@pytest.mark.parametrize("N,K", [(3, 10), (4, 4), (5, 2), (8, 77), (16, 259)])
def test_allreduce_equals_reducescatter_then_allgather(oracle_mod, dtype, op, N, K):
    """AllReduce = AllGather o ReduceScatter (Collectives and sharded matmul,
    'where 2(N-1)/N comes from'; AllReduce survey, semantics and decomposition),
    bit for bit when ReduceScatter gives rank r chunk r folded from rank r (the
    library's placement reading)."""
    x = _inputs(dtype, N, K, seed=N + 7 * K)
    ar, _ = oracle_mod.ring_allreduce(x, op)
    rs = oracle_mod.reduce_scatter(x, op)
    ag = oracle_mod.allgather(rs, K)
    for r in range(N):
        np.testing.assert_array_equal(_bits(ag[r]), _bits(ar[r]))


@pytest.mark.parametrize("N,K", [(3, 6), (4, 13), (8, 64), (5, 3)])
def test_allgather_is_adjoint_of_reducescatter(oracle_mod, N, K):
    """<AG(x), y> = <x, RS(y)> (Collectives and sharded matmul, FSDP slide: the
    transpose of AllGather is ReduceScatter), on integer-valued fp32 where every
    sum is exact."""
    g = np.random.Generator(np.random.PCG64(N * K))
    off, ln = oracle_mod.partition(K, N)
    xs = [g.integers(-8, 9, size=ln[r]).astype(np.float32) for r in range(N)]
    ys = [g.integers(-8, 9, size=K).astype(np.float32) for _ in range(N)]
    agx = oracle_mod.allgather(xs, K)
    rsy = oracle_mod.reduce_scatter(ys, "sum")
    lhs = sum(float(np.dot(agx[q].astype(np.float64), ys[q].astype(np.float64))) for q in range(N))
    rhs = sum(float(np.dot(xs[r].astype(np.float64), rsy[r].astype(np.float64))) for r in range(N))
    assert lhs == rhs


def test_reduce_scatter_brute_force_integers(oracle_mod):
    """On exact integer inputs, rank r's output is the brute-force sum of chunk r."""
    N, K = 6, 47
    x = W.integers_fp32(N, K, seed=3)
    off, ln = oracle_mod.partition(K, N)
    rs = oracle_mod.reduce_scatter(list(x), "sum")
    tot = x.astype(np.float64).sum(axis=0)
    for r in range(N):
        np.testing.assert_array_equal(rs[r].astype(np.float64), tot[off[r]:off[r] + ln[r]])


@pytest.mark.parametrize("N,root", [(1, 0), (3, 2), (8, 5)])
def test_broadcast_copies_root(oracle_mod, N, root):
    x = list(W.mixed_bf16(N, 33, seed_base=9))
    outs = oracle_mod.broadcast(x, root)
    for o in outs:
        np.testing.assert_array_equal(o, x[root])


@pytest.mark.parametrize("N", [1, 2, 3, 8])
def test_alltoall_involution_and_definition(oracle_mod, N):
    """AllToAll is a block transpose (Collectives and sharded matmul, 'AllToAll':
    rank = row, block = column), so applying it twice is the identity; with
    variable blocks the second application uses the transposed counts."""
    g = np.random.Generator(np.random.PCG64(N))
    counts = g.integers(0, 9, size=(N, N))
    sends = [W.random_bits_u16(int(counts[i].sum()), seed=i) for i in range(N)]
    once = oracle_mod.alltoallv(sends, counts)
    # definition, brute force: recv_j block i == send_i block j
    for j in range(N):
        pos = 0
        for i in range(N):
            s0 = int(counts[i, :j].sum())
            np.testing.assert_array_equal(once[j][pos:pos + counts[i, j]], sends[i][s0:s0 + counts[i, j]])
            pos += counts[i, j]
    twice = oracle_mod.alltoallv(once, counts.T.copy())
    for i in range(N):
        np.testing.assert_array_equal(twice[i], sends[i])


# ---------------------------------------------------------------- buckets

def test_c4_bucket_count(oracle_mod):
    """4 Llama layers, 25 MiB bf16 buckets: 809,533,440 elements per rank fill
    61 buckets of 13,107,200 elements and a last one of 9,994,240."""
    numels = W.llama_layer_numels(4)
    assert sum(numels) == 809_533_440
    be = W.bucket_elems(25 * W.MiB, 2)
    assert be == 13_107_200
    n_full, last = divmod(sum(numels), be)
    assert (n_full, last) == (61, 9_994_240)


@pytest.mark.parametrize("op,N", [("sum", 4), ("avg", 3), ("avg_premul", 3)])
def test_bucket_allreduce_matches_flatten_and_ring(oracle_mod, op, N):
    """Bucket fusion (Collective Communication, 'Bucket fusion'): tensors are
    laid out in reverse registration order, cut into fixed-size buckets, and
    each bucket is an independent ring AllReduce.  The packing is re-done here
    with numpy (concatenate reversed, split) and compared."""
    numels = [5, 17, 3, 40, 1, 26]
    be = 13
    grads = [[W.to_bf16_bits(W.normal_fp32(1, n, seed_base=100 * r + t)[0]) for t, n in enumerate(numels)]
             for r in range(N)]
    got = oracle_mod.bucket_allreduce(grads, be, op)
    streams = [np.concatenate(grads[r][::-1]) for r in range(N)]
    total = streams[0].size
    res = [np.empty_like(s) for s in streams]
    for b0 in range(0, total, be):
        outs, _ = oracle_mod.ring_allreduce([s[b0:b0 + be] for s in streams], op)
        for r in range(N):
            res[r][b0:b0 + be] = outs[r]
    for r in range(N):
        back = np.split(res[r], np.cumsum(numels[::-1])[:-1])[::-1]
        for t in range(len(numels)):
            np.testing.assert_array_equal(got[r][t], back[t])


def test_bucket_allreduce_integer_exact(oracle_mod):
    N = 3
    numels = [7, 30, 2, 11]
    g = np.random.Generator(np.random.PCG64(1))
    grads = [[g.integers(-8, 9, size=n).astype(np.float32) for n in numels] for _ in range(N)]
    got = oracle_mod.bucket_allreduce(grads, 9, "sum")
    for t in range(len(numels)):
        ref = sum(grads[r][t].astype(np.float64) for r in range(N))
        for r in range(N):
            np.testing.assert_array_equal(got[r][t].astype(np.float64), ref)
