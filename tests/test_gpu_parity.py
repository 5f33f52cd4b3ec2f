"""GPU parity: every collective through the C ABI against the CPU oracle, bit
for bit, on seeded inputs that span several tiles and a ragged tail, with
signed zeros, subnormals, infinities and NaNs mixed in; plus edge cases
(empty, one rank, fewer elements than ranks, unaligned buffers) and the
composition invariants on the device."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W
from ring_allreduce_rank_gb300.arena import RankArena

from gpu_util import DEV, assert_bits_equal, bits, empty_like_host, to_dev, torch_dtype

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def inputs(dtype, N, K, seed):
    if dtype == "bf16":
        return list(W.mixed_bf16(N, K, seed_base=seed))
    return list(W.mixed_fp32(N, K, seed_base=seed))


def run_allreduce(x, op, mode, in_place=True, pad=0):
    send = [to_dev(r, pad_elems=pad) for r in x]
    if in_place:
        recv = send
    else:
        recv = [empty_like_host(r.size, torch_dtype(x), pad_elems=(pad + 1) % 3) for r in x]
    ccl.ccl_allreduce(send, recv, op=op, mode=mode)
    torch.cuda.synchronize()
    return [bits(t) for t in recv]


# ------------------------------------------------------------------ pages' examples on the device

def _golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("case", _golden("worked_examples.json"), ids=lambda c: c["name"])
def test_worked_examples_on_gpu(case, mode):
    ins = [np.asarray(r, dtype=np.float32) for r in case["inputs"]]
    exp = [np.asarray(r, dtype=np.float32) for r in case["expected"]]
    N = len(ins)
    kind = case["collective"]
    if kind == "allreduce":
        got = run_allreduce(ins, case["op"], mode)
    elif kind == "reduce_scatter":
        send = [to_dev(r) for r in ins]
        _, ln = ccl.ccl_plan_chunks(ins[0].size, N)
        out = [torch.zeros(ln[r], dtype=torch.float32, device=DEV) for r in range(N)]
        ccl.ccl_reduce_scatter(send, out, op=case["op"], mode=mode)
        got = [bits(t) for t in out]
    elif kind == "broadcast":
        send = [to_dev(r) for r in ins]
        ccl.ccl_broadcast(send, send, root=case["root"], mode=mode)
        got = [bits(t) for t in send]
    elif kind == "allgather":
        send = [to_dev(r) for r in ins]
        out = [torch.zeros(exp[0].size, dtype=torch.float32, device=DEV) for _ in range(N)]
        ccl.ccl_allgather(send, out, mode=mode)
        got = [bits(t) for t in out]
    elif kind == "alltoall":
        send = [to_dev(r) for r in ins]
        out = [torch.zeros_like(s) for s in send]
        ccl.ccl_alltoall(send, out, mode=mode)
        got = [bits(t) for t in out]
    elif kind == "reduce":
        send = [to_dev(r) for r in ins]
        ccl.ccl_reduce(send, send, root=case["root"], op=case["op"], mode=mode)
        got = [bits(t) for t in send]
    elif kind == "gather":
        send = [to_dev(r) for r in ins]
        out = [None] * N
        out[case["root"]] = torch.zeros(exp[0].size, dtype=torch.float32, device=DEV)
        ccl.ccl_gather(send, out, root=case["root"], mode=mode)
        got = [bits(out[case["root"]])]
    else:
        raise AssertionError(kind)
    torch.cuda.synchronize()
    for r in range(len(exp)):
        assert_bits_equal(got[r], exp[r], "%s rank %d" % (case["name"], r))


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("case", _golden("rounding_cases.json"), ids=lambda c: c["name"])
def test_rounding_cases_on_gpu(case, mode):
    dt = np.uint16 if case["dtype"] == "bf16" else np.uint32
    ins = [np.array([int(v, 16) for v in row], dtype=dt) for row in case["inputs_bits"]]
    if case["dtype"] == "fp32":
        ins = [a.view(np.float32) for a in ins]
    exp = np.array([int(v, 16) for v in case["expected_bits"]], dtype=dt)
    got = run_allreduce(ins, case["op"], mode)
    for r, g in enumerate(got):
        assert_bits_equal(g, exp, "%s rank %d" % (case["name"], r))


# ------------------------------------------------------------------ AllReduce sweep

AR_SHAPES = [(1, 5), (2, 1), (2, 4099), (3, 5), (3, 2), (4, 4096), (5, 3), (7, 10007), (8, 3 * 2048 * 8 + 13),
             (8, 70000), (16, 70001), (17, 12345), (33, 4099), (64, 20000)]


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min"])
@pytest.mark.parametrize("N,K", AR_SHAPES, ids=lambda v: str(v))
def test_allreduce_matches_oracle(N, K, op, dtype, mode):
    x = inputs(dtype, N, K, seed=17 * N + K)
    want, _ = oracle.ring_allreduce(x, op)
    got = run_allreduce(x, op, mode, in_place=(K % 2 == 0))
    for r in range(N):
        assert_bits_equal(got[r], want[r], "AR %s %s N=%d K=%d rank %d" % (op, dtype, N, K, r))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("pad", [1, 2, 3])
@pytest.mark.parametrize("N,K", [(3, 1001), (8, 20000), (4, 7)])
def test_allreduce_unaligned_buffers(N, K, pad, dtype):
    """Buffers that are not 16-byte aligned take the element path."""
    x = inputs(dtype, N, K, seed=pad)
    want, _ = oracle.ring_allreduce(x, "sum")
    for in_place in (True, False):
        got = run_allreduce(x, "sum", "fused", in_place=in_place, pad=pad)
        for r in range(N):
            assert_bits_equal(got[r], want[r], "unaligned rank %d" % r)


def test_allreduce_count_zero_and_single_rank():
    t = torch.zeros(0, dtype=torch.bfloat16, device=DEV)
    ccl.ccl_allreduce([t, t.clone()], op="sum")
    # N = 1 AVG divides by 1: NaN payloads become the canonical NaN, the rest is unchanged
    x = W.mixed_bf16(1, 1000, seed_base=3)
    want, _ = oracle.ring_allreduce(list(x), "avg")
    got = run_allreduce(list(x), "avg", "fused")
    assert_bits_equal(got[0], want[0], "N=1 avg")


def test_allreduce_arena_guards_and_launch_count():
    N, K = 8, 70001
    x = W.normal_bf16(N, K, seed_base=2)
    arena = RankArena(N, K, torch.bfloat16, device=DEV, guard_bytes=1024)
    arena.load([r.view(np.int16) for r in x])
    n0 = ccl.ccl_launch_count()
    ccl.ccl_allreduce(arena.ranks, op="avg")
    torch.cuda.synchronize()
    assert ccl.ccl_launch_count() - n0 == 1
    assert arena.guards_intact()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    got = arena.rows_bits()
    for r in range(N):
        assert_bits_equal(got[r].view(np.uint16), want[r], "arena rank %d" % r)
    n0 = ccl.ccl_launch_count()
    ccl.ccl_allreduce(arena.ranks, op="avg", mode="step")
    torch.cuda.synchronize()
    assert ccl.ccl_launch_count() - n0 == 2 * (N - 1) + 1
    assert arena.guards_intact()


# ------------------------------------------------------------------ ReduceScatter / AllGather

RS_SHAPES = [(1, 9), (2, 4099), (3, 10), (4, 4096), (5, 3), (8, 70000), (8, 70003), (16, 16 * 3001 + 11),
             (33, 5000)]


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod"])
@pytest.mark.parametrize("N,K", RS_SHAPES, ids=lambda v: str(v))
def test_reduce_scatter_then_allgather(N, K, op, dtype, mode):
    """ReduceScatter matches the oracle; AllGather of its output equals the
    AllReduce bit for bit (AllReduce = ReduceScatter + AllGather)."""
    x = inputs(dtype, N, K, seed=5 * N + K)
    td = torch_dtype(x)
    _, ln = ccl.ccl_plan_chunks(K, N)
    send = [to_dev(r) for r in x]
    rs = [empty_like_host(ln[r], td) for r in range(N)]
    ccl.ccl_reduce_scatter(send, rs, op=op, mode=mode)
    ag = [empty_like_host(K, td) for _ in range(N)]
    ccl.ccl_allgather(rs, ag, mode=mode)
    torch.cuda.synchronize()
    want_rs = oracle.reduce_scatter(x, op)
    want_ar, _ = oracle.ring_allreduce(x, op)
    for r in range(N):
        assert_bits_equal(bits(rs[r]), want_rs[r], "RS rank %d" % r)
        assert_bits_equal(bits(ag[r]), want_ar[r], "RS+AG rank %d" % r)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,K", [(3, 10), (8, 70003), (4, 4096)])
def test_in_place_reduce_scatter_and_allgather(N, K, dtype):
    """NCCL-style in-place forms: ReduceScatter into send[r] + off_r, and
    AllGather from recv[r] + off_r."""
    x = inputs(dtype, N, K, seed=N * K)
    off, ln = ccl.ccl_plan_chunks(K, N)
    bufs = [to_dev(r) for r in x]
    rs = [bufs[r][off[r]:off[r] + ln[r]] for r in range(N)]
    ccl.ccl_reduce_scatter(bufs, rs, op="sum")
    ccl.ccl_allgather(rs, bufs)
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(x, "sum")
    for r in range(N):
        assert_bits_equal(bits(bufs[r]), want[r], "in-place RS+AG rank %d" % r)


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,K", [(1, 5), (3, 15), (4, 4099), (8, 65536 + 3), (16, 777), (40, 4000)])
def test_allgather_matches_oracle(N, K, dtype, mode):
    off, ln = ccl.ccl_plan_chunks(K, N)
    x = inputs(dtype, N, K, seed=K)
    chunks = [x[r][:ln[r]].copy() for r in range(N)]
    send = [to_dev(c) for c in chunks]
    out = [empty_like_host(K, torch_dtype(x)) for _ in range(N)]
    ccl.ccl_allgather(send, out, mode=mode)
    torch.cuda.synchronize()
    want = oracle.allgather(chunks, K)
    for r in range(N):
        assert_bits_equal(bits(out[r]), want[r], "AG rank %d" % r)


# ------------------------------------------------------------------ Reduce / Gather / Scatter

@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "prod", "min"])
@pytest.mark.parametrize("N,K,root", [(1, 9, 0), (3, 5, 0), (4, 4099, 3), (8, 70003, 5), (16, 777, 15),
                                      (33, 4099, 7)])
def test_reduce_matches_oracle(N, K, root, op, dtype, mode):
    """The root receives the AllReduce's bits; no other buffer is written."""
    x = inputs(dtype, N, K, seed=root * 7 + K)
    want = oracle.reduce(x, root, op)
    send = [to_dev(r) for r in x]
    recv = [None] * N
    recv[root] = empty_like_host(K, torch_dtype(x), pad_elems=root % 2)
    ccl.ccl_reduce(send, recv, root=root, op=op, mode=mode)
    inplace = [to_dev(r) for r in x]
    ccl.ccl_reduce(inplace, inplace, root=root, op=op, mode=mode)
    torch.cuda.synchronize()
    assert_bits_equal(bits(recv[root]), want[root], "reduce root")
    for r in range(N):
        assert_bits_equal(bits(send[r]), x[r], "reduce input %d untouched" % r)
        assert_bits_equal(bits(inplace[r]), want[r], "reduce in place rank %d" % r)


@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,K,root", [(1, 5, 0), (3, 15, 0), (4, 4099, 2), (8, 65536 + 3, 7), (16, 777, 4)])
def test_gather_and_scatter_match_oracle(N, K, root, dtype, mode):
    off, ln = ccl.ccl_plan_chunks(K, N)
    full = inputs(dtype, 1, K, seed=K + root)[0]
    parts = oracle.scatter(full, N)
    # Scatter from root
    send = [None] * N
    send[root] = to_dev(full)
    recv = [empty_like_host(ln[r], torch_dtype([full]), pad_elems=r % 3) for r in range(N)]
    ccl.ccl_scatter(send, recv, root=root, mode=mode)
    # Gather back to root
    out = [None] * N
    out[root] = empty_like_host(K, torch_dtype([full]))
    ccl.ccl_gather(recv, out, root=root, mode=mode)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(recv[r]), parts[r], "scatter rank %d" % r)
    assert_bits_equal(bits(out[root]), oracle.gather(parts, K), "gather")
    assert_bits_equal(bits(out[root]), full, "gather(scatter(x)) = x")


# ------------------------------------------------------------------ Broadcast

@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,K,root", [(1, 7, 0), (3, 5, 0), (4, 4099, 3), (8, 70001, 5), (20, 333, 11)])
def test_broadcast_matches_oracle(N, K, root, dtype, mode):
    x = inputs(dtype, N, K, seed=root + K)
    want = oracle.broadcast(x, root)
    bufs = [to_dev(r) for r in x]
    ccl.ccl_broadcast(bufs, bufs, root=root, mode=mode)  # in place
    out = [empty_like_host(K, torch_dtype(x), pad_elems=1) for _ in range(N)]
    send = [None] * N
    send[root] = to_dev(x[root])
    ccl.ccl_broadcast(send, out, root=root, mode=mode)  # out of place, unaligned outputs
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(bufs[r]), want[r], "bcast in place rank %d" % r)
        assert_bits_equal(bits(out[r]), want[r], "bcast rank %d" % r)


@pytest.mark.parametrize("N", [8, 20])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("shift", [0, 16, 32, 4])
@pytest.mark.parametrize("kind", ["whole32", "whole16", "ragged"])
def test_fanout_vector_widths(kind, shift, dtype, N):
    """The fan-out kernel (Broadcast, AllGather, Gather) moves 32-byte vectors
    when every buffer starts on a 32-byte boundary and the chunk starts on a
    whole 32-byte vector, 16-byte vectors when only 16-byte alignment holds,
    and elements or shifted windows otherwise.  Buffers start `shift` bytes
    past a 512-byte boundary; the chunk length makes chunk offsets whole
    32-byte vectors, whole 16-byte vectors only (odd multiples), or ragged."""
    es = 2 if dtype == "bf16" else 4
    vec = 16 // es
    per = {"whole32": 2 * vec * 300, "whole16": 2 * vec * 300 + vec, "ragged": 2 * vec * 300 + 3}[kind]
    K = N * per + (5 if kind == "ragged" else 0)
    pad = shift // es
    x = inputs(dtype, N, K, seed=K + shift)
    tdt = torch_dtype(x)
    # Broadcast from rank 3, out of place (N = 20: the large parameter block)
    send = [None] * N
    send[3] = to_dev(x[3], pad_elems=pad)
    out = [empty_like_host(K, tdt, pad_elems=pad) for _ in range(N)]
    ccl.ccl_broadcast(send, out, root=3)
    # AllGather of each rank's chunk
    off, ln = ccl.ccl_plan_chunks(K, N)
    chunks = [x[r][off[r]:off[r] + ln[r]].copy() for r in range(N)]
    cs = [to_dev(c, pad_elems=pad) for c in chunks]
    ag = [empty_like_host(K, tdt, pad_elems=pad) for _ in range(N)]
    ccl.ccl_allgather(cs, ag)
    # Gather to rank 5
    g = [None] * N
    g[5] = empty_like_host(K, tdt, pad_elems=pad)
    ccl.ccl_gather(cs, g, root=5)
    torch.cuda.synchronize()
    want_b = oracle.broadcast(x, 3)
    want_ag = oracle.allgather(chunks, K)
    for r in range(N):
        assert_bits_equal(bits(out[r]), want_b[r], "bcast rank %d" % r)
        assert_bits_equal(bits(ag[r]), want_ag[r], "allgather rank %d" % r)
    assert_bits_equal(bits(g[5]), oracle.gather(chunks, K), "gather")


# ------------------------------------------------------------------ AllToAll(v)

@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,maxc", [(1, 50), (2, 9), (3, 1000), (8, 5000), (8, 3), (13, 300)])
def test_alltoallv_matches_oracle(N, maxc, dtype, mode):
    g = np.random.Generator(np.random.PCG64(N * maxc))
    counts = g.integers(0, maxc + 1, size=(N, N))
    counts[0, N - 1] = 0
    sends = [inputs(dtype, 1, int(counts[i].sum()), seed=i)[0] for i in range(N)]
    want = oracle.alltoallv(sends, counts)
    send = [to_dev(s) for s in sends]
    recv = [empty_like_host(int(counts[:, j].sum()), torch_dtype(sends), pad_elems=j % 3) for j in range(N)]
    ccl.ccl_alltoallv(send, recv, counts.tolist(), mode=mode)
    back = [empty_like_host(int(counts[i].sum()), torch_dtype(sends)) for i in range(N)]
    ccl.ccl_alltoallv(recv, back, counts.T.tolist(), mode=mode)
    torch.cuda.synchronize()
    for j in range(N):
        assert_bits_equal(bits(recv[j]), want[j], "A2Av recv %d" % j)
        assert_bits_equal(bits(back[j]), sends[j], "A2Av twice = identity, rank %d" % j)


@pytest.mark.parametrize("N,blk", [(4, 1), (4, 16), (8, 7168)])
def test_alltoall_uniform(N, blk):
    x = [W.random_bits_u16(N * blk, seed=100 + r) for r in range(N)]
    want = oracle.alltoallv(x, np.full((N, N), blk))
    send = [to_dev(r) for r in x]
    recv = [torch.empty_like(s) for s in send]
    ccl.ccl_alltoall(send, recv)
    torch.cuda.synchronize()
    for j in range(N):
        assert_bits_equal(bits(recv[j]), want[j], "A2A rank %d" % j)


# ------------------------------------------------------------------ bucket AllReduce

@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("N,numels,bucket_elems", [
    (3, [5, 17, 3, 40, 1, 26], 13),
    (4, [4096, 4096 * 3 + 5, 11, 4096, 70000], 8192),
    (8, [1000, 20000, 3, 20001, 512], 6000),
    (8, [4096] * 10, 1 << 20),
])
def test_bucket_allreduce_matches_oracle(N, numels, bucket_elems, op, dtype, mode):
    es = 2 if dtype == "bf16" else 4
    grads_h = [[inputs(dtype, 1, n, seed=1000 * r + t)[0] for t, n in enumerate(numels)] for r in range(N)]
    want = oracle.bucket_allreduce(grads_h, bucket_elems, op)
    grads = [[to_dev(g, pad_elems=(t % 2)) for t, g in enumerate(row)] for row in grads_h]
    ccl.ccl_bucket_allreduce(grads, bucket_bytes=bucket_elems * es, op=op, mode=mode)
    torch.cuda.synchronize()
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(bits(grads[r][t]), want[r][t], "bucket rank %d tensor %d" % (r, t))
