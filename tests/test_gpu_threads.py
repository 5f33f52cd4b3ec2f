"""Several host threads calling the library at once, each on its own stream.

Fused collectives share nothing on the device; the host-side state (launch
counter, trace buffer, the host-buffer AllReduce's copy streams, the bucket
planner) is shared and locked.  ctypes releases the GIL around each call, so
the threads really are inside the library together.  Every thread's results
must equal the oracle's bit for bit, and the trace and launch counts must add
up over all threads."""
import threading

import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu
ITERS = 12


def _rows_bits(rows):
    return [np.asarray(r).view(np.uint16) if np.asarray(r).dtype == np.uint16 else np.asarray(r).view(np.uint32)
            for r in rows]


def test_threads_on_their_own_streams_get_the_oracles_bits():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    # one workload per thread: (ranks, count, dtype, op)
    specs = [(8, 3 * 65536 + 13, "bf16", "avg"), (5, 100_003, "fp32", "sum"),
             (16, 40_000, "bf16", "max"), (3, 77_777, "fp32", "prod")]
    cases = []
    for i, (N, K, dt, op) in enumerate(specs):
        x = list(W.mixed_bf16(N, K, seed_base=50 + 10 * i) if dt == "bf16" else W.mixed_fp32(N, K, seed_base=50 + 10 * i))
        ar, _ = oracle.ring_allreduce(x, op)
        numels = [K // 3, K - K // 3]
        grads_h = [[r[:numels[0]], r[numels[0]:]] for r in x]
        bk = oracle.bucket_allreduce(grads_h, 4096, op)
        cases.append(dict(N=N, K=K, dt=dt, op=op, x=x, ar=ar, numels=numels, bucket=bk))

    prior_trace = ccl.ccl_get_config()["trace"]
    ccl.ccl_set_trace(True)
    ccl.ccl_trace_clear()
    launches0 = ccl.ccl_launch_count()
    errors = []
    results = [None] * len(cases)
    barrier = threading.Barrier(len(cases), timeout=300)

    def worker(i):
        try:
            c = cases[i]
            N, K = c["N"], c["K"]
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                pristine = [to_dev(r) for r in c["x"]]
                bufs = [torch.empty_like(p) for p in pristine]
                _, ln = ccl.ccl_plan_chunks(K, N)
                parts = [torch.empty(ln[r], dtype=pristine[0].dtype, device="cuda:0") for r in range(N)]
                full = [torch.empty_like(p) for p in pristine]
                host = [torch.empty(K, dtype=pristine[0].dtype).pin_memory() for _ in range(N)]
                work = torch.empty(3 * N * 4096 * 4, dtype=torch.uint8, device="cuda:0")
                grads = [[torch.empty(n, dtype=pristine[0].dtype, device="cuda:0") for n in c["numels"]]
                         for _ in range(N)]
                s.synchronize()
                barrier.wait()
                for _ in range(ITERS):
                    for b, p in zip(bufs, pristine):
                        b.copy_(p)
                    ccl.ccl_allreduce(bufs, op=c["op"], stream=s)
                    ccl.ccl_reduce_scatter(pristine, parts, op=c["op"], stream=s)
                    ccl.ccl_allgather(parts, full, stream=s)
                    for r in range(N):
                        grads[r][0].copy_(pristine[r][:c["numels"][0]])
                        grads[r][1].copy_(pristine[r][c["numels"][0]:])
                    ccl.ccl_bucket_allreduce(grads, bucket_bytes=4096 * pristine[0].element_size(), op=c["op"],
                                             stream=s)
                    for h, p in zip(host, pristine):
                        h.copy_(p, non_blocking=True)
                    ccl.ccl_allreduce_host(host, op=c["op"], work=work, stream=s)
                s.synchronize()
                results[i] = dict(ar=[bits(b) for b in bufs], ag=[bits(f) for f in full],
                                  bucket=[[bits(g) for g in row] for row in grads],
                                  host=[bits(h) for h in host])
        except Exception as e:  # reported by the main thread
            errors.append((i, repr(e)))
            barrier.abort()  # the others stop waiting for this thread

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    torch.cuda.synchronize()
    try:
        assert not any(t.is_alive() for t in threads)
        assert not errors, errors
        recs = ccl.ccl_trace_read()
    finally:
        ccl.ccl_set_trace(prior_trace)

    for i, c in enumerate(cases):
        got, want = results[i], _rows_bits(c["ar"])
        for r in range(c["N"]):
            assert_bits_equal(got["ar"][r], want[r], "thread %d AllReduce rank %d" % (i, r))
            assert_bits_equal(got["ag"][r], want[r], "thread %d ReduceScatter+AllGather rank %d" % (i, r))
            assert_bits_equal(got["host"][r], want[r], "thread %d host-buffer AllReduce rank %d" % (i, r))
            for t in range(2):
                assert_bits_equal(got["bucket"][r][t], _rows_bits([c["bucket"][r][t]])[0],
                                  "thread %d bucket rank %d tensor %d" % (i, r, t))

    # five traced calls per iteration per thread, none lost, all successful;
    # their launches add up to the library's counter
    calls = 5 * ITERS * len(cases)
    assert len(recs) == calls
    assert all(r["status"] == 0 for r in recs)
    assert sorted(r["seq"] for r in recs) == list(range(recs[0]["seq"], recs[0]["seq"] + calls))
    assert sum(r["launches"] for r in recs) == ccl.ccl_launch_count() - launches0
    per = {}
    for r in recs:
        per[r["collective"]] = per.get(r["collective"], 0) + 1
    assert per == {"allreduce": ITERS * len(cases), "reduce_scatter": ITERS * len(cases),
                   "allgather": ITERS * len(cases), "bucket_allreduce": ITERS * len(cases),
                   "allreduce_host": ITERS * len(cases)}
