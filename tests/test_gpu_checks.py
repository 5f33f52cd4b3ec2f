"""Result checks and tracing on the device: ccl_check_identical counts, bit
for bit, the elements where a rank differs from rank 0 (0 after every
AllReduce, exactly the planted differences otherwise), and traced calls
record their shape and the kernels they launched."""
import numpy as np
import pytest
import torch

import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    ccl.lib()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,K,pad", [(8, 70001, 0), (3, 1000, 1), (33, 4099, 0)])
def test_check_identical_counts_planted_differences(N, K, pad, dtype):
    x = W.mixed_bf16(N, K, seed_base=N) if dtype == "bf16" else W.mixed_fp32(N, K, seed_base=N)
    bufs = [to_dev(r, pad_elems=pad) for r in x]
    ccl.ccl_allreduce(bufs, op="sum")
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ccl.ccl_check_identical(bufs, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0
    g = np.random.Generator(np.random.PCG64(K))
    planted = 0
    for r in (1, N - 1):
        for e in sorted(set(g.integers(0, K, size=5).tolist()) | {0, K - 1}):
            v = bufs[r][e:e + 1]
            v.view(torch.int16 if dtype == "bf16" else torch.int32).bitwise_xor_(1)
            planted += 1
    cnt.zero_()
    ccl.ccl_check_identical(bufs, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == planted


def test_trace_records_calls():
    ccl.ccl_trace_clear()
    ccl.ccl_set_trace(True)
    try:
        N, K = 4, 4099
        bufs = [torch.zeros(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
        ccl.ccl_allreduce(bufs, op="avg")
        ccl.ccl_allreduce(bufs, op="sum", mode="step")
        torch.cuda.synchronize()
        recs = ccl.ccl_trace_read()
    finally:
        ccl.ccl_set_trace(False)
    assert [r["collective"] for r in recs] == ["allreduce", "allreduce"]
    assert recs[0]["launches"] == 1 and recs[1]["launches"] == 2 * (N - 1)
    assert all(r["status"] == 0 and r["nranks"] == N and r["count"] == K and r["dtype"] == 1 for r in recs)
    assert recs[0]["op"] == 1 and recs[1]["mode"] == 1 and recs[1]["seq"] == recs[0]["seq"] + 1
    assert all(r["gpu_ns"] > 0 for r in recs)


def test_trace_device_time_agrees_with_events_and_skips_capture():
    """A traced call's device time is that of its work on its stream: it
    agrees with CUDA events taken around the same call by the caller.  Calls
    made during graph capture are traced untimed and the capture still
    works."""
    N, K = 8, 1 << 24  # 32 MiB per rank: about 80 us per AllReduce
    bufs = [torch.zeros(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce(bufs, op="sum")  # warm-up
    torch.cuda.synchronize()
    ccl.ccl_trace_clear()
    ccl.ccl_set_trace(True)
    try:
        times = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # keep the GPU busy while the host enqueues, so that the caller's
            # events time the call's work and not the host's enqueue gap
            torch.cuda._sleep(2_000_000)
            e0.record()
            ccl.ccl_allreduce(bufs, op="sum")
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e6)
        recs = ccl.ccl_trace_read()
        assert len(recs) == 3
        for r, t in zip(recs, times):
            assert r["gpu_ns"] > 0
            assert abs(r["gpu_ns"] - t) <= 0.25 * t + 10_000, (r["gpu_ns"], t)

        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                ccl.ccl_allreduce(bufs, op="sum")
        g.replay()
        torch.cuda.synchronize()
        rec = ccl.ccl_trace_read()[-1]
        assert rec["collective"] == "allreduce" and rec["status"] == 0 and rec["gpu_ns"] == 0
    finally:
        ccl.ccl_set_trace(False)


def test_automatic_checks_follow_each_collective():
    """With checks on, every AllReduce (fused, step, another order, the
    compressed one), AllGather and Broadcast enqueues one comparison of its
    outputs: one extra launch each, and no mismatch on correct results.  Off,
    nothing extra is launched."""
    N, K = 6, 20_011
    x = list(W.mixed_bf16(N, K, seed_base=41))
    bufs = [to_dev(r) for r in x]
    _, ln = ccl.ccl_plan_chunks(K, N)
    parts = [torch.empty(ln[r], dtype=torch.bfloat16, device=DEV) for r in range(N)]
    full = [torch.empty(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    grads = [to_dev(r) for r in W.normal_bf16(N, K, std=1e-2, seed_base=3)]
    res = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    ccl.ccl_allreduce_compressed(grads, res, op="avg")  # its one-time set-up, outside the counted region
    torch.cuda.synchronize()
    ccl.ccl_set_check(True)
    try:
        ccl.ccl_check_read(reset=True)
        n0 = ccl.ccl_launch_count()
        ccl.ccl_allreduce(bufs, op="sum")
        ccl.ccl_allreduce_algo(bufs, op="max", algo="tree")
        ccl.ccl_reduce_scatter(bufs, parts, op="sum")          # not checked: outputs differ by design
        ccl.ccl_allgather(parts, full)
        ccl.ccl_broadcast(bufs, full, root=2)
        ccl.ccl_allreduce_compressed(grads, res, op="avg")
        fused = ccl.ccl_launch_count() - n0
        assert ccl.ccl_check_read() == 0
        n1 = ccl.ccl_launch_count()
        ccl.ccl_allreduce(bufs, op="avg", mode="step")
        step = ccl.ccl_launch_count() - n1
        assert ccl.ccl_check_read() == 0
    finally:
        ccl.ccl_set_check(False)
    n2 = ccl.ccl_launch_count()
    ccl.ccl_allreduce(bufs, op="sum")
    ccl.ccl_allreduce_compressed(grads, res, op="avg")
    plain = ccl.ccl_launch_count() - n2
    # checked: AR 1+1, tree 1+1, RS 1, AG 1+1, broadcast 1+1, compressed (pipe + tail) 2+1
    assert fused == 2 + 2 + 1 + 2 + 2 + 3
    assert step == 2 * (N - 1) + 1 + 1  # in place: 2(N-1) steps, the AVG scale, the check
    assert plain == 1 + 2
    torch.cuda.synchronize()
