"""The named workloads at full size, on the device, in the launch configuration
the benchmark times (fused mode, one launch), checked against the oracle:

  integers   AllReduce SUM, N=4, 4096 fp32 integers in [-8, 8] (exact sums)
  grad-avg   AllReduce AVG, N=8, 64Mi bf16 per rank (128 MiB), Normal(0, 1e-3), in place
  ragged     ReduceScatter then AllGather vs AllReduce, N=16, 16,777,259 fp32, SUM and MAX
  buckets    bucket-fused AllReduce, N=8, 4 Llama layers (809,533,440 bf16 per rank), 25 MiB buckets
  sweep      AllReduce SUM bf16, 1 KiB .. 1 GiB per rank (x4 steps), N in {2,4,8,16,64}, sampled outputs
  moe-a2a    AllToAllv, N=8, 4096 tokens x 7168 bf16 per rank, Zipf(1.2) top-1 routing over 64 experts
"""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W
from ring_allreduce_rank_gb300.arena import RankArena

from accuracy import error_figures, report
from gpu_util import DEV, assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _normwise_ok(y_bits_bf16, x, op, rtol, tag):
    """The relative tolerance, normwise; the elementwise figure is printed
    beside it (tests/accuracy.py)."""
    y = W.bf16_bits_to_f32(y_bits_bf16).astype(np.float64) if y_bits_bf16.dtype == np.uint16 else \
        y_bits_bf16.astype(np.float64)
    y64, absum = oracle.sum_f64(x, op)
    fig = error_figures(y, y64, absum)
    report(tag, fig)
    return fig["normwise"] <= rtol


def test_integers_fp32_n4_exact():
    x = W.integers_fp32(4, 4096, seed=0)
    ref = x.astype(np.float64).sum(axis=0)
    for mode in ("fused", "step"):
        bufs = [to_dev(r) for r in x]
        ccl.ccl_allreduce(bufs, op="sum", mode=mode)
        torch.cuda.synchronize()
        for b in bufs:
            np.testing.assert_array_equal(b.cpu().numpy().astype(np.float64), ref)


def test_grad_avg_bf16_n8_128mib_full():
    N, K = 8, 64 * 1024 * 1024
    x = W.normal_bf16(N, K, std=1e-3, seed_base=0)
    arena = RankArena(N, K, torch.bfloat16, device=DEV, guard_bytes=256)
    arena.load([r.view(np.int16) for r in x])
    ccl.ccl_allreduce(arena.ranks, op="avg")
    torch.cuda.synchronize()
    assert arena.guards_intact()
    got = arena.rows_bits()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(got[r].view(np.uint16), want[r], "grad-avg rank %d" % r)
    assert _normwise_ok(want[0], list(x), "avg", 1e-2, "grad-avg N=8 bf16 64Mi")


@pytest.mark.parametrize("op", ["sum", "max"])
def test_ragged_fp32_n16_rs_ag_equals_ar(op):
    N, K = 16, 16_777_259
    x = W.uniform_fp32(N, K, seed_base=0)
    off, ln = ccl.ccl_plan_chunks(K, N)
    assert ln == [1_048_579] * 11 + [1_048_578] * 5
    send = [to_dev(r) for r in x]
    rs = [torch.empty(ln[r], dtype=torch.float32, device=DEV) for r in range(N)]
    ag = [torch.empty(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    ccl.ccl_reduce_scatter(send, rs, op=op)
    ccl.ccl_allgather(rs, ag)
    ccl.ccl_allreduce(send, op=op)  # in place, after the RS read its inputs
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), op)
    for r in range(N):
        a, g = bits(send[r]), bits(ag[r])
        assert_bits_equal(g, a, "RS+AG vs AR rank %d" % r)
        assert_bits_equal(a, want[r], "ragged AR rank %d" % r)
    if op == "sum":
        assert _normwise_ok(want[0], list(x), "sum", 1e-5, "ragged N=16 fp32 SUM")
    else:
        np.testing.assert_array_equal(want[0], x.max(axis=0))


@pytest.mark.slow
def test_buckets_llama4_bf16_n8_full():
    N = 8
    numels = W.llama_layer_numels(4)
    be = W.bucket_elems(25 * W.MiB, 2)
    grads_h = W.bucket_gradients_bf16(N, numels, std=1e-3, seed_base=0)
    grads = [[to_dev(g) for g in row] for row in grads_h]
    n0 = ccl.ccl_launch_count()
    ccl.ccl_bucket_allreduce(grads, bucket_bytes=25 * W.MiB, op="sum")
    torch.cuda.synchronize()
    launches = ccl.ccl_launch_count() - n0
    assert 1 <= launches <= 2
    got = [[bits(g) for g in row] for row in grads]
    del grads
    torch.cuda.empty_cache()
    want = oracle.bucket_allreduce(grads_h, be, "sum")
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(got[r][t], want[r][t], "bucket rank %d tensor %d" % (r, t))


SWEEP_N = [2, 4, 8, 16, 64]
SWEEP_BYTES = [1 << k for k in range(10, 31, 2)]  # 1 KiB .. 1 GiB


@pytest.mark.slow
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep_allreduce_bf16_sampled(N):
    """Inputs: a Normal(0, 1e-3) pattern of up to 4Mi elements per rank tiled to
    the full length; outputs checked at sampled positions (every chunk's first
    and last element plus random ones) with the oracle's closed form."""
    P = 1 << 22
    g = np.random.Generator(np.random.PCG64(N))
    for S in SWEEP_BYTES:
        K = S // 2
        pat = W.normal_bf16(N, min(K, P), std=1e-3, seed_base=0)
        arena = RankArena(N, K, torch.bfloat16, device=DEV)
        for r in range(N):
            p_dev = to_dev(pat[r])
            reps = (K + p_dev.numel() - 1) // p_dev.numel()
            arena.ranks[r].copy_(p_dev.repeat(reps)[:K])
            del p_dev
        ccl.ccl_allreduce(arena.ranks, op="sum")
        torch.cuda.synchronize()
        off, ln = ccl.ccl_plan_chunks(K, N)
        idx = set(g.integers(0, K, size=2048).tolist())
        for c in range(N):
            if ln[c]:
                idx.update([off[c], off[c] + ln[c] - 1])
        idx = np.array(sorted(idx), dtype=np.int64)
        vals = [pat[r][idx % pat.shape[1]] for r in range(N)]
        want = oracle.ring_allreduce_gathered(vals, K, idx.astype(np.uint64), "sum")
        it = torch.from_numpy(idx).to(DEV)
        for r in (0, N // 2, N - 1):
            got = bits(arena.ranks[r].index_select(0, it))
            assert_bits_equal(got, want, "sweep N=%d S=%d rank %d" % (N, S, r))
        for r in range(1, N):
            assert torch.equal(arena.ranks[r].view(torch.int16), arena.ranks[0].view(torch.int16))
        y64, absum = oracle.sum_f64(vals, "sum")
        fig = error_figures(W.bf16_bits_to_f32(want), y64, absum)
        report("sweep N=%d S=%d (sampled)" % (N, S), fig)
        del arena
        torch.cuda.empty_cache()


def test_moe_alltoallv_n8_full():
    N, T, H = 8, 4096, 7168
    counts_tok = W.zipf_expert_counts(N, T, 64, 1.2, 1000)
    counts = counts_tok * H
    sends = [W.random_bits_u16(T * H, seed=2000 + i) for i in range(N)]
    want = oracle.alltoallv(sends, counts)
    send = [to_dev(s) for s in sends]
    recv = [torch.empty(int(counts[:, j].sum()), dtype=torch.bfloat16, device=DEV) for j in range(N)]
    ccl.ccl_alltoallv(send, recv, counts.tolist())
    torch.cuda.synchronize()
    for j in range(N):
        assert_bits_equal(bits(recv[j]), want[j], "moe a2a rank %d" % j)


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_64bit_indexing_over_2_pow_31_elements(dtype):
    """More than 2^31 elements per rank (N=2, a ragged 2^31 + 4099): every index
    computation has to be 64-bit.  Inputs are a seeded pattern tiled to full
    length; outputs are checked at sampled positions on both sides of 2^31
    and at the chunk boundary."""
    N, K = 2, (1 << 31) + 4099
    P = 1 << 20
    pat = W.normal_bf16(N, P, seed_base=7) if dtype == "bf16" else W.normal_fp32(N, P, seed_base=7)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    arena = RankArena(N, K, td, device=DEV)
    for r in range(N):
        p_dev = to_dev(pat[r])
        arena.ranks[r].copy_(p_dev.repeat((K + P - 1) // P)[:K])
        del p_dev
    ccl.ccl_allreduce(arena.ranks, op="sum")
    torch.cuda.synchronize()
    off, ln = ccl.ccl_plan_chunks(K, N)
    g = np.random.Generator(np.random.PCG64(31))
    idx = set(g.integers(0, K, size=4096).tolist())
    for e in (0, 1, off[1] - 1, off[1], off[1] + 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, K - 8, K - 1):
        idx.add(int(e))
    idx = np.array(sorted(idx), dtype=np.int64)
    vals = [pat[r][idx % P] for r in range(N)]
    want = oracle.ring_allreduce_gathered(vals, K, idx.astype(np.uint64), "sum")
    it = torch.from_numpy(idx).to(DEV)
    for r in range(N):
        assert_bits_equal(bits(arena.ranks[r].index_select(0, it)), want, "K > 2^31 rank %d" % r)
    del arena
    torch.cuda.empty_cache()


@pytest.mark.parametrize("algo", ["ring", "halving_doubling", "tree", "hierarchical"])
def test_maximum_ranks_1024(algo):
    """The largest rank count the ABI accepts: 1024 ranks, ragged length."""
    N, K = 1024, 3001
    x = list(W.mixed_bf16(N, K, seed_base=11))
    group = 32 if algo == "hierarchical" else 0
    if algo == "ring":
        want, _ = oracle.ring_allreduce(x, "sum")
    else:
        want = oracle.allreduce_algo(x, algo, "sum", group)
    bufs = [to_dev(r) for r in x]
    ccl.ccl_allreduce_algo(bufs, op="sum", algo=algo, group_size=group)
    torch.cuda.synchronize()
    for r in (0, 1, 511, 1023):
        assert_bits_equal(bits(bufs[r]), want[r], "%s N=1024 rank %d" % (algo, r))


def test_maximum_ranks_1024_reduce_scatter_allgather_broadcast():
    N, K = 1024, 5000
    x = list(W.normal_bf16(N, K, seed_base=12))
    off, ln = ccl.ccl_plan_chunks(K, N)
    send = [to_dev(r) for r in x]
    rs = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    ag = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    ccl.ccl_reduce_scatter(send, rs, op="avg")
    ccl.ccl_allgather(rs, ag)
    ccl.ccl_broadcast(send, send, root=1023)
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(x, "avg")
    for r in (0, 7, 1023):
        assert_bits_equal(bits(ag[r]), want[r], "RS+AG N=1024 rank %d" % r)
        assert_bits_equal(bits(send[r]), x[1023], "broadcast N=1024 rank %d" % r)
