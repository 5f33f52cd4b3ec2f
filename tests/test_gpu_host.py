"""AllReduce of rank buffers in host memory (ccl_allreduce_host), checked bit
for bit against the oracle, on both of its paths: in place over the host link
(page-locked buffers read and written by the fused kernel) and staged (slices
copied in, reduced with the whole vector's chunk rotation and copied out, so
the result must be the ring AllReduce of the whole vector, whatever the
slicing).  Every test runs with the library's host path set to "staged" (the
default) and to "direct"."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C
from ring_allreduce_rank_gb300 import workloads as W

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


@pytest.fixture(autouse=True, params=["staged", "direct"])
def host_path(request):
    ccl.ccl_set_host_path(request.param)
    yield request.param
    ccl.ccl_set_host_path("staged")


def _host(rows, pinned=True):
    """(N, K) numpy rows -> one host tensor per rank, same bits."""
    out = []
    for row in rows:
        row = np.ascontiguousarray(row)
        t = torch.from_numpy(row.view(np.int16)).view(torch.bfloat16) if row.dtype == np.uint16 else \
            torch.from_numpy(row.astype(np.float32, copy=False))
        t = t.clone()
        out.append(t.pin_memory() if pinned else t)
    return out


def _host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else \
        t.view(torch.int32).numpy().view(np.uint32)


def _work(nbytes):
    return torch.empty(nbytes, dtype=torch.uint8, device=DEV)


def _stage_work(N, es, stage_elems):
    return _work(3 * N * stage_elems * es)


@pytest.mark.parametrize("N,K", [(3, 10_007), (8, 65_536 + 13), (16, 40_001), (5, 4)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "avg", "max", "min", "prod"])
def test_host_allreduce_matches_oracle(N, K, dtype, op):
    """A small work buffer (1024-element stages) forces many slices, ragged
    chunks and slices that straddle chunk boundaries."""
    x = W.mixed_bf16(N, K, seed_base=N) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=N)
    want, _ = oracle.ring_allreduce(list(x), op)
    send = _host(x)
    recv = [torch.empty_like(t).pin_memory() for t in send]
    es = 2 if dtype == "bf16" else 4
    s = torch.cuda.Stream()
    ccl.ccl_allreduce_host(send, recv, op=op, work=_stage_work(N, es, 1024), stream=s)
    s.synchronize()  # the call's copies are joined into its stream
    assert len(ccl.ccl_plan_host_slices(K, N, dtype, 3 * N * 1024 * es)) >= (2 if K > 1024 else 1)
    for r in range(N):
        assert_bits_equal(_host_bits(recv[r]), want[r], "host AR %s %s N=%d rank %d" % (dtype, op, N, r))
        assert_bits_equal(_host_bits(send[r]), x[r], "input untouched rank %d" % r)


def test_host_allreduce_equals_device_allreduce_in_place_and_pageable():
    """In place, in pageable (not page-locked) host memory, and against the
    device-resident AllReduce of the same data."""
    N, K = 8, 300_001
    x = W.normal_bf16(N, K, seed_base=3)
    dev = [to_dev(r) for r in x]
    ccl.ccl_allreduce(dev, op="avg")
    host = _host(x, pinned=False)
    ccl.ccl_allreduce_host(host, op="avg", work=_stage_work(N, 2, 4096))
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(_host_bits(host[r]), bits(dev[r]), "host vs device rank %d" % r)
        assert_bits_equal(_host_bits(host[r]), want[r], "host vs oracle rank %d" % r)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("pad", [0, 24])
def test_host_allreduce_rows_of_one_allocation(dtype, pad):
    """Rank buffers that are equally spaced rows of one pinned allocation move
    with one 2D copy per slice and direction; the output rows here have a
    different pitch (pad elements between them) from the input rows."""
    N, K = 6, 123_457
    x = W.mixed_bf16(N, K, seed_base=7) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=7)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    src = torch.from_numpy(x.view(np.int16) if dtype == "bf16" else x).view(td).clone().pin_memory()
    dst = torch.zeros((N, K + pad), dtype=td).pin_memory()
    send = [src[r] for r in range(N)]
    recv = [dst[r, :K] for r in range(N)]
    ccl.ccl_allreduce_host(send, recv, op="avg", work=_stage_work(N, es, 4096))
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(_host_bits(recv[r].contiguous()), want[r], "rows %s pad %d rank %d" % (dtype, pad, r))
        if pad:
            assert not dst[r, K:].view(torch.int16 if es == 2 else torch.int32).any(), "padding written"
    # in place on the rows
    ccl.ccl_allreduce_host(send, op="sum", work=_stage_work(N, es, 2048))
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), "sum")
    for r in range(N):
        assert_bits_equal(_host_bits(send[r]), want[r], "rows in place %s rank %d" % (dtype, r))


def test_host_allreduce_back_to_back_calls_share_the_work_buffer():
    """Two calls in a row on one stream reuse the stages; each gets its own
    result (the second call's copies-in wait for the first call's copies-out)."""
    N, K = 4, 200_000
    work = _stage_work(N, 4, 2048)
    xa, xb = W.normal_fp32(N, K, seed_base=10), W.uniform_fp32(N, K, seed_base=20)
    sa, sb = _host(xa), _host(xb)
    ra = [torch.empty_like(t).pin_memory() for t in sa]
    rb = [torch.empty_like(t).pin_memory() for t in sb]
    s = torch.cuda.Stream()
    ccl.ccl_allreduce_host(sa, ra, op="sum", work=work, stream=s)
    ccl.ccl_allreduce_host(sb, rb, op="max", work=work, stream=s)
    s.synchronize()
    wa, _ = oracle.ring_allreduce(list(xa), "sum")
    wb, _ = oracle.ring_allreduce(list(xb), "max")
    for r in range(N):
        assert_bits_equal(_host_bits(ra[r]), wa[r], "first call rank %d" % r)
        assert_bits_equal(_host_bits(rb[r]), wb[r], "second call rank %d" % r)


def test_host_allreduce_degenerate_cases():
    # count 0: nothing happens, no work buffer needed
    e = [torch.empty(0, dtype=torch.float32).pin_memory() for _ in range(3)]
    ccl.ccl_allreduce_host(e, op="sum", work=_work(16))
    # one rank, out of place: a copy; AVG divides by 1
    x = W.mixed_fp32(1, 5000, seed_base=1)
    for op in ("sum", "avg"):
        send, recv = _host(x), [torch.empty(5000, dtype=torch.float32).pin_memory()]
        ccl.ccl_allreduce_host(send, recv, op=op, work=_stage_work(1, 4, 256))
        torch.cuda.synchronize()
        want, _ = oracle.ring_allreduce(list(x), op)
        assert_bits_equal(_host_bits(recv[0]), want[0], "N=1 %s" % op)
    # fewer elements than ranks: empty chunks
    x = W.normal_fp32(7, 3, seed_base=2)
    send = _host(x)
    ccl.ccl_allreduce_host(send, op="sum", work=_stage_work(7, 4, 256))
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), "sum")
    for r in range(7):
        assert_bits_equal(_host_bits(send[r]), want[r], "K<N rank %d" % r)


def test_host_allreduce_refuses_stream_capture():
    send = _host(W.normal_fp32(2, 1024, seed_base=4))
    work = _stage_work(2, 4, 256)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            with pytest.raises(C.CclError) as ei:
                ccl.ccl_allreduce_host(send, op="sum", work=work, stream=s)
        finally:
            g.capture_end()
    assert ei.value.status == 2  # CCL_ERR_UNSUPPORTED


@pytest.mark.slow
def test_host_allreduce_headline_size():
    """N=8, 64 Mi bf16 elements per rank, AVG, default work buffer: the
    end-to-end configuration the benchmark times."""
    N, K = 8, 64 * 1024 * 1024
    x = W.normal_bf16(N, K, std=1e-3, seed_base=0)
    send = _host(x)
    recv = [torch.empty_like(t).pin_memory() for t in send]
    ccl.ccl_allreduce_host(send, recv, op="avg", work=_work(C.HOST_WORK_BYTES_DEFAULT))
    torch.cuda.synchronize()
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(_host_bits(recv[r]), want[r], "headline host AR rank %d" % r)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_allreduce_path_taken(host_path, pinned):
    """Page-locked buffers take one fused launch on the "direct" path;
    pageable buffers, or the "staged" path, take the staged pipeline (many
    launches: one reduction per slice).  The bits are the oracle's either way."""
    N, K = 4, 3 * 65_536 + 11
    x = W.normal_bf16(N, K, std=1e-3, seed_base=17)
    send = _host(x, pinned=pinned)
    recv = [torch.empty_like(t).pin_memory() if pinned else torch.empty_like(t) for t in send]
    work = _stage_work(N, 2, 4096)
    n0 = ccl.ccl_launch_count()
    ccl.ccl_allreduce_host(send, recv, op="avg", work=work)
    torch.cuda.synchronize()
    launches = ccl.ccl_launch_count() - n0
    if pinned and host_path == "direct":
        assert launches == 1
    else:
        assert launches > 1
    want, _ = oracle.ring_allreduce(list(x), "avg")
    for r in range(N):
        assert_bits_equal(_host_bits(recv[r]), want[r], "%s pinned=%s rank %d" % (host_path, pinned, r))


def test_host_allreduce_registered_memory(host_path):
    """Pageable host memory page-locked after the fact (cudaHostRegister) is
    what many frameworks hand over: the direct path reads and writes it in
    place like cudaHostAlloc'd memory, and both paths give the oracle's bits."""
    cudart = torch.cuda.cudart()
    N, K = 3, 50_003
    x = W.normal_fp32(N, K, seed_base=61)
    send = [torch.from_numpy(r.copy()) for r in x]  # pageable
    recv = [torch.empty(K, dtype=torch.float32) for _ in range(N)]
    regs = []
    try:
        for t in send + recv:
            assert int(cudart.cudaHostRegister(t.data_ptr(), t.numel() * 4, 0)) == 0
            regs.append(t)
        n0 = ccl.ccl_launch_count()
        ccl.ccl_allreduce_host(send, recv, op="sum", work=_stage_work(N, 4, 1024))
        torch.cuda.synchronize()
        launches = ccl.ccl_launch_count() - n0
        assert (launches == 1) == (host_path == "direct")
        want, _ = oracle.ring_allreduce(list(x), "sum")
        for r in range(N):
            assert_bits_equal(_host_bits(recv[r]), want[r], "registered %s rank %d" % (host_path, r))
    finally:
        for t in regs:
            cudart.cudaHostUnregister(t.data_ptr())
