"""The pre-multiplied AVG (NCCL's pre-multiplied sum, Collective Communication,
libraries section) on the device, bit for bit against the oracle: every
contribution scaled by the correctly rounded reciprocal of N and rounded to the
buffer type, then summed in ring order.  Covers every kernel path that folds
contributions: the exact-N and any-N fused kernels, the element path
(unaligned buffers), the shifted ReduceScatter path, the many-rank small-chunk
kernel, the step-by-step ring, Reduce, bucket fusion, the bucketer and the
host-buffer pipeline; plus the calls that refuse the operator."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, assert_bits_equal, bits, empty_like_host, to_dev, torch_dtype

pytestmark = pytest.mark.gpu
OP = "avg_premul"


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


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("N,K", [(1, 1000), (2, 4099), (3, 10_007), (4, 8192 + 5), (5, 77_777), (8, 65_536 + 13),
                                 (16, 40_001), (17, 9_999), (7, 3)])
def test_allreduce(dtype, mode, N, K):
    x = inputs(dtype, N, K, seed=N * 100 + K % 97)
    want, _ = oracle.ring_allreduce(x, OP)
    send = [to_dev(r) for r in x]
    ccl.ccl_allreduce(send, op=OP, mode=mode)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(send[r]), want[r], "premul AR %s %s N=%d K=%d rank %d" % (dtype, mode, N, K, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(3, 5001), (8, 10_000)])
def test_allreduce_unaligned_out_of_place(dtype, N, K):
    """Buffers one element past a 16-byte boundary take the element path."""
    x = inputs(dtype, N, K, seed=5 + N)
    want, _ = oracle.ring_allreduce(x, OP)
    send = [to_dev(r, pad_elems=1) for r in x]
    recv = [empty_like_host(K, torch_dtype(x), pad_elems=2) for _ in range(N)]
    ccl.ccl_allreduce(send, recv, op=OP)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(recv[r]), want[r], "premul unaligned rank %d" % r)
        assert_bits_equal(bits(send[r]), x[r], "input untouched rank %d" % r)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("mode", ["fused", "step"])
@pytest.mark.parametrize("N,K", [(3, 10_007), (8, 65_536 + 13), (16, 40_001), (5, 4)])
def test_reduce_scatter(dtype, mode, N, K):
    """K not a multiple of N * vector: chunks at unaligned offsets go through
    the shifted ReduceScatter path."""
    x = inputs(dtype, N, K, seed=N + 3 * K)
    want = oracle.reduce_scatter(x, OP)
    send = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    recv = [empty_like_host(int(ln[r]), torch_dtype(x)) for r in range(N)]
    ccl.ccl_reduce_scatter(send, recv, op=OP, mode=mode)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(recv[r]), want[r], "premul RS %s %s N=%d rank %d" % (dtype, mode, N, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K,root", [(3, 10_007, 1), (8, 40_000, 0), (6, 5, 5)])
def test_reduce(dtype, N, K, root):
    x = inputs(dtype, N, K, seed=N * 7 + root)
    want = oracle.reduce(x, root, OP)
    send = [to_dev(r) for r in x]
    recv = [None] * N
    recv[root] = empty_like_host(K, torch_dtype(x))
    ccl.ccl_reduce(send, recv, root=root, op=OP)
    torch.cuda.synchronize()
    assert_bits_equal(bits(recv[root]), want[root], "premul reduce root %d" % root)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(64, 64 * 40 + 7), (100, 1000), (1024, 5000)])
def test_many_ranks_small_chunks(dtype, N, K):
    """More than 16 ranks with at most 64 elements per chunk: the shared-memory
    small-chunk kernel."""
    x = inputs(dtype, N, K, seed=N + K)
    want, _ = oracle.ring_allreduce(x, OP)
    send = [to_dev(r) for r in x]
    ccl.ccl_allreduce(send, op=OP)
    torch.cuda.synchronize()
    for r in (0, N // 2, N - 1):
        assert_bits_equal(bits(send[r]), want[r], "premul small chunks N=%d rank %d" % (N, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N", [3, 8])
def test_bucket_allreduce_and_bucketer(dtype, N):
    numels = [5, 17, 3, 4000, 1, 2600, 129]
    bucket_bytes = 1024 * (2 if dtype == "bf16" else 4)
    es = 2 if dtype == "bf16" else 4
    gen = (lambda n, s: W.mixed_bf16(1, n, seed_base=s)[0]) if dtype == "bf16" else \
        (lambda n, s: W.mixed_fp32(1, n, seed_base=s)[0])
    host = [[gen(n, 100 * r + t) for t, n in enumerate(numels)] for r in range(N)]
    want = oracle.bucket_allreduce(host, bucket_bytes // es, OP)
    dev = [[to_dev(a) for a in row] for row in host]
    ccl.ccl_bucket_allreduce(dev, bucket_bytes=bucket_bytes, op=OP)
    torch.cuda.synchronize()
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(bits(dev[r][t]), want[r][t], "premul bucket rank %d tensor %d" % (r, t))
    dev = [[to_dev(a) for a in row] for row in host]
    b = ccl.CclBucketer(dev, bucket_bytes=bucket_bytes, op=OP)
    for t in reversed(range(len(numels))):
        b.mark_ready(t)
    torch.cuda.synchronize()
    b.close()
    for r in range(N):
        for t in range(len(numels)):
            assert_bits_equal(bits(dev[r][t]), want[r][t], "premul bucketer rank %d tensor %d" % (r, t))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(3, 10_007), (8, 65_536 + 13)])
def test_host_buffers(dtype, N, K):
    x = inputs(dtype, N, K, seed=N * 11)
    want, _ = oracle.ring_allreduce(x, OP)
    td = torch_dtype(x)
    send = [(torch.from_numpy(r.view(np.int16)).view(td) if td == torch.bfloat16 else torch.from_numpy(r))
            .clone().pin_memory() for r in x]
    es = 2 if dtype == "bf16" else 4
    work = torch.empty(3 * N * 1024 * es, dtype=torch.uint8, device=DEV)
    ccl.ccl_allreduce_host(send, op=OP, work=work)
    torch.cuda.synchronize()
    for r in range(N):
        got = send[r].view(torch.int16).numpy().view(np.uint16) if es == 2 else \
            send[r].view(torch.int32).numpy().view(np.uint32)
        assert_bits_equal(got, want[r], "premul host rank %d" % r)


def test_power_of_two_matches_avg_on_device():
    """N = 8 on normal bf16 gradients: the same bits as AVG (1/8 is exact)."""
    N, K = 8, 1 << 20
    x = list(W.normal_bf16(N, K, std=1e-3, seed_base=9))
    a = [to_dev(r) for r in x]
    p = [to_dev(r) for r in x]
    ccl.ccl_allreduce(a, op="avg")
    ccl.ccl_allreduce(p, op=OP)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), p[0].view(torch.int16))


def test_refused_by_other_orders_and_compression():
    x = [to_dev(r) for r in inputs("fp32", 4, 1000, seed=1)]
    for algo in ("halving_doubling", "tree", "hierarchical"):
        with pytest.raises(C.CclError) as ei:
            ccl.ccl_allreduce_algo(x, op=OP, algo=algo, group_size=2)
        assert ei.value.status == 2, algo  # CCL_ERR_UNSUPPORTED
    ccl.ccl_allreduce_algo(x, op=OP, algo="ring")  # the ring order takes it
    res = [torch.zeros(1000, dtype=torch.float32, device=DEV) for _ in range(4)]
    with pytest.raises(C.CclError) as ei:
        ccl.ccl_allreduce_compressed(x, res, op=OP, comp="int8_block", block=128)
    assert ei.value.status == 2
    torch.cuda.synchronize()


@pytest.mark.parametrize("op", ["avg_premul", "min"])
@pytest.mark.parametrize("N", [1, 5])
def test_static_scratch_reduce_scatter(op, N):
    """The allocation-free step-by-step ReduceScatter takes every op the
    step mode takes, the pre-multiplied AVG included (N = 1: one scaling
    launch and no steps)."""
    import ctypes
    fn = ccl.lib().ccl_reduce_scatter_step_static
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, pp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    K = 50_003
    x = inputs("bf16", N, K, seed=N + 40)
    want = oracle.reduce_scatter(x, op)
    send = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    recv = [empty_like_host(int(ln[r]), torch.bfloat16) for r in range(N)]
    ptrs = lambda ts: (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    rc = fn(ptrs(send), ptrs(recv), N, K, 1, C.OPS[op], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, ccl.ccl_status_string(rc)
    torch.cuda.synchronize()
    for r in range(N):
        assert_bits_equal(bits(recv[r]), want[r], "static scratch %s N=%d rank %d" % (op, N, r))
