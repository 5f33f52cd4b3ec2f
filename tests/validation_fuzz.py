"""Randomised overlap validation, run by test_validation_fuzz.py in a child
process with CUDA_VISIBLE_DEVICES="": the pointers are fake, so a call that
passed validation can only fail its launch (no device), never touch memory.

The expected outcome comes from the header's contract, restated here: the
buffers a call writes must not overlap one another, and a buffer it reads may
overlap a buffer it writes only in that call's documented in-place form
(AllReduce: send[r] == recv[r]; ReduceScatter: recv[r] == send[r] + off_r
elements; AllGather: send[r] == recv[r] + off_r elements)."""
import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import ring_allreduce_rank_gb300 as ccl  # noqa: E402

FAKE = 0x7f0000000000
OVERLAP, CUDA_ERR = 3, 4


def _pp(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def _meets(a, b):
    return a[0] < b[1] and b[0] < a[1] and a[0] < a[1] and b[0] < b[1]


def expected_overlap(kind, send, recv, K, es):
    N = len(send)
    q, rem = K // N, K % N
    ln = [q + (1 if c < rem else 0) for c in range(N)]
    off = [sum(ln[:c]) for c in range(N)]
    if kind == "allreduce":
        W = [(recv[r], recv[r] + K * es) for r in range(N)]
        R = [(send[r], send[r] + K * es) for r in range(N)]
        in_place = lambda r: send[r] == recv[r]
    elif kind == "reduce_scatter":
        W = [(recv[r], recv[r] + ln[r] * es) for r in range(N)]
        R = [(send[r], send[r] + K * es) for r in range(N)]
        in_place = lambda r: recv[r] == send[r] + off[r] * es
    else:  # allgather
        W = [(recv[r], recv[r] + K * es) for r in range(N)]
        R = [(send[r], send[r] + ln[r] * es) for r in range(N)]
        in_place = lambda r: send[r] == recv[r] + off[r] * es
    return _violates(W, R, lambda i, j: i == j and in_place(i))


def _violates(W, R, allowed):
    """W, R: lists of (lo, hi) write / read ranges; allowed(i, j): read i may
    overlap write j."""
    for i in range(len(W)):
        for j in range(i + 1, len(W)):
            if _meets(W[i], W[j]):
                return True
    for i in range(len(R)):
        for j in range(len(W)):
            if _meets(R[i], W[j]) and not allowed(i, j):
                return True
    return False


def expected_overlap_rooted(kind, send, recv, root, K, es):
    """Reduce: writes recv[root], reads every send[r], in place when
    send[root] == recv[root].  Broadcast: writes every recv[r], reads
    send[root], in place when recv[root] == send[root].  Gather: writes
    recv[root], reads every send[r] (len_r), which may sit at recv[root] +
    off_r.  Scatter: writes every recv[r] (len_r), reads send[root], and recv[r]
    may sit at send[root] + off_r."""
    N = len(send)
    q, rem = K // N, K % N
    ln = [q + (1 if c < rem else 0) for c in range(N)]
    off = [sum(ln[:c]) for c in range(N)]
    if kind == "reduce":
        W = [(recv[root], recv[root] + K * es)]
        R = [(send[r], send[r] + K * es) for r in range(N)]
        return _violates(W, R, lambda i, j: i == root and send[root] == recv[root])
    if kind == "broadcast":
        W = [(recv[r], recv[r] + K * es) for r in range(N)]
        R = [(send[root], send[root] + K * es)]
        return _violates(W, R, lambda i, j: j == root and send[root] == recv[root])
    if kind == "gather":
        W = [(recv[root], recv[root] + K * es)]
        R = [(send[r], send[r] + ln[r] * es) for r in range(N)]
        return _violates(W, R, lambda i, j: send[i] == recv[root] + off[i] * es)
    W = [(recv[r], recv[r] + ln[r] * es) for r in range(N)]  # scatter
    R = [(send[root], send[root] + K * es)]
    return _violates(W, R, lambda i, j: recv[j] == send[root] + off[j] * es)


def main(iters=3000):
    L = ccl.lib()
    g = np.random.default_rng(20261202)
    seen = {OVERLAP: 0, "accepted": 0}
    stream = ctypes.c_void_p(0)
    for it in range(iters):
        kind = ["allreduce", "reduce_scatter", "allgather"][it % 3]
        N = int(g.integers(1, 7))
        K = int(g.integers(1, 40))
        dt = int(g.integers(0, 2))
        es = 4 if dt == 0 else 2
        window = int(g.choice([64, 512, 4096]))
        send = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        recv = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        q, rem = K // N, K % N
        off = [c * q + min(c, rem) for c in range(N)]
        for r in range(N):  # often take the call's in-place form for some ranks
            if g.random() < 0.3:
                if kind == "allreduce":
                    recv[r] = send[r]
                elif kind == "reduce_scatter":
                    recv[r] = send[r] + off[r] * es
                else:
                    send[r] = recv[r] + off[r] * es
        want = expected_overlap(kind, send, recv, K, es)
        fn = {"allreduce": lambda: L.ccl_allreduce(_pp(send), _pp(recv), N, K, dt, 0, 0, stream),
              "reduce_scatter": lambda: L.ccl_reduce_scatter(_pp(send), _pp(recv), N, K, dt, 0, 0, stream),
              "allgather": lambda: L.ccl_allgather(_pp(send), _pp(recv), N, K, dt, 0, stream)}[kind]
        got = fn()
        if want:
            assert got == OVERLAP, (kind, N, K, es, send, recv, got)
            seen[OVERLAP] += 1
        else:
            # accepted: nothing to do (0) or a launch that fails without a device
            assert got in (0, CUDA_ERR), (kind, N, K, es, send, recv, got)
            seen["accepted"] += 1
    assert seen[OVERLAP] > iters // 10 and seen["accepted"] > iters // 10, seen
    rooted = {OVERLAP: 0, "accepted": 0}
    for it in range(iters):
        kind = ["reduce", "broadcast", "gather", "scatter"][it % 4]
        N = int(g.integers(1, 7))
        K = int(g.integers(1, 40))
        root = int(g.integers(0, N))
        dt = int(g.integers(0, 2))
        es = 4 if dt == 0 else 2
        window = int(g.choice([64, 512, 4096]))
        send = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        recv = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        q, rem = K // N, K % N
        off = [c * q + min(c, rem) for c in range(N)]
        for r in range(N):  # the documented in-place forms, often
            if g.random() < 0.3:
                if kind in ("reduce", "broadcast") and r == root:
                    recv[root] = send[root]
                elif kind == "gather":
                    send[r] = recv[root] + off[r] * es
                elif kind == "scatter":
                    recv[r] = send[root] + off[r] * es
        want = expected_overlap_rooted(kind, send, recv, root, K, es)
        fn = {"reduce": lambda: L.ccl_reduce(_pp(send), _pp(recv), N, root, K, dt, 0, 0, stream),
              "broadcast": lambda: L.ccl_broadcast(_pp(send), _pp(recv), N, root, K, dt, 0, stream),
              "gather": lambda: L.ccl_gather(_pp(send), _pp(recv), N, root, K, dt, 0, stream),
              "scatter": lambda: L.ccl_scatter(_pp(send), _pp(recv), N, root, K, dt, 0, stream)}[kind]
        got = fn()
        if want:
            assert got == OVERLAP, (kind, N, root, K, es, send, recv, got)
            rooted[OVERLAP] += 1
        else:
            assert got in (0, CUDA_ERR), (kind, N, root, K, es, send, recv, got)
            rooted["accepted"] += 1
    assert rooted[OVERLAP] > iters // 10 and rooted["accepted"] > iters // 10, rooted
    # AllToAllv: no in-place form (every read disjoint from every write);
    # bucket AllReduce: in place on the tensors, which must all be disjoint
    other = {OVERLAP: 0, "accepted": 0}
    for it in range(iters):
        N = int(g.integers(1, 6))
        dt = int(g.integers(0, 2))
        es = 4 if dt == 0 else 2
        window = int(g.choice([64, 512, 4096]))
        if it % 2 == 0:
            counts = g.integers(0, 6, size=(N, N))
            stot, rtot = counts.sum(axis=1), counts.sum(axis=0)
            send = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
            recv = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
            W = [(recv[j], recv[j] + int(rtot[j]) * es) for j in range(N)]
            R = [(send[i], send[i] + int(stot[i]) * es) for i in range(N)]
            want = _violates(W, R, lambda i, j: False)
            cts = (ctypes.c_size_t * (N * N))(*[int(c) for c in counts.ravel()])
            got = L.ccl_alltoallv(_pp(send), _pp(recv), N, cts, dt, 0, stream)
            what = ("alltoallv", N, counts.tolist(), send, recv, got)
        else:
            T = int(g.integers(1, 5))
            numels = [int(v) for v in g.integers(0, 20, size=T)]
            ptrs = [FAKE + es * int(g.integers(0, window)) for _ in range(N * T)]
            W = [(ptrs[r * T + t], ptrs[r * T + t] + numels[t] * es) for r in range(N) for t in range(T)]
            want = _violates(W, [], lambda i, j: False)
            nums = (ctypes.c_size_t * T)(*numels)
            got = L.ccl_bucket_allreduce(_pp(ptrs), nums, T, N, 0, dt, 0, 0, stream)
            what = ("bucket", N, numels, ptrs, got)
        if want:
            assert got == OVERLAP, what
            other[OVERLAP] += 1
        else:
            assert got in (0, CUDA_ERR), what
            other["accepted"] += 1
    assert other[OVERLAP] > iters // 10 and other["accepted"] > iters // 10, other
    # compressed and Top-k AllReduce: gradients, residuals (and Top-k's work
    # buffer) all disjoint; host-buffer AllReduce: outputs and the work buffer
    # disjoint, an input overlapping an output only as send[r] == recv[r]
    comp = {OVERLAP: 0, "accepted": 0}
    topk_wb = ctypes.c_size_t()
    for it in range(iters):
        N = int(g.integers(1, 6))
        K = int(g.integers(1, 40))
        dt = int(g.integers(0, 2))
        es = 4 if dt == 0 else 2
        window = int(g.choice([64, 512, 4096]))
        far = FAKE + (1 << 32)
        kind = ["compressed", "topk", "host"][it % 3]
        if kind in ("compressed", "topk"):
            grads = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
            res = [FAKE + 4 * int(g.integers(0, window)) for _ in range(N)]
            W = [(p, p + K * es) for p in grads] + [(p, p + K * 4) for p in res]
            if kind == "compressed":
                got = L.ccl_allreduce_compressed(_pp(grads), _pp(res), N, K, dt, 0, 0, 128, ctypes.c_float(0.5),
                                                 stream)
            else:
                assert L.ccl_plan_topk_work_bytes(N, ctypes.byref(topk_wb)) == 0
                work = far if g.random() < 0.7 else FAKE + 16 * int(g.integers(0, window))
                W.append((work, work + topk_wb.value))
                got = L.ccl_allreduce_topk(_pp(grads), _pp(res), N, K, dt, 0, 3, ctypes.c_void_p(work),
                                           topk_wb.value, stream)
            want = _violates(W, [], lambda i, j: False)
            what = (kind, N, K, es, grads, res, got)
        else:
            send = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
            recv = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
            for r in range(N):
                if g.random() < 0.3:
                    recv[r] = send[r]
            wbytes = 3 * N * 256 * es
            work = far if g.random() < 0.7 else FAKE + 16 * int(g.integers(0, window))
            W = [(recv[r], recv[r] + K * es) for r in range(N)] + [(work, work + wbytes)]
            R = [(send[r], send[r] + K * es) for r in range(N)]
            want = _violates(W, R, lambda i, j: j == i and send[i] == recv[i])
            got = L.ccl_allreduce_host(_pp(send), _pp(recv), N, K, dt, 0, ctypes.c_void_p(work), wbytes, stream)
            what = (kind, N, K, es, send, recv, work, got)
        if want:
            assert got == OVERLAP, what
            comp[OVERLAP] += 1
        else:
            assert got in (0, CUDA_ERR), what
            comp["accepted"] += 1
    assert comp[OVERLAP] > iters // 10 and comp["accepted"] > iters // 10, comp
    # the ReduceScatter that allocates nothing promises ccl_reduce_scatter's
    # error checks: both must answer every layout the same way
    same = {OVERLAP: 0, "accepted": 0}
    for it in range(iters):
        N = int(g.integers(1, 7))
        K = int(g.integers(1, 40))
        dt = int(g.integers(0, 2))
        es = 4 if dt == 0 else 2
        window = int(g.choice([64, 512, 4096]))
        send = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        recv = [FAKE + es * int(g.integers(0, window)) for _ in range(N)]
        q, rem = K // N, K % N
        for r in range(N):
            if g.random() < 0.3:
                recv[r] = send[r] + (r * q + min(r, rem)) * es
        want = expected_overlap("reduce_scatter", send, recv, K, es)
        a = L.ccl_reduce_scatter(_pp(send), _pp(recv), N, K, dt, 0, 1, stream)
        b = L.ccl_reduce_scatter_step_static(_pp(send), _pp(recv), N, K, dt, 0, stream)
        assert (a == OVERLAP) == want and (b == OVERLAP) == want, (N, K, es, send, recv, a, b)
        same[OVERLAP if want else "accepted"] += 1
    assert same[OVERLAP] > iters // 10 and same["accepted"] > iters // 10, same
    # NULL entries: allowed for zero-element buffers and for the entries a
    # call ignores, rejected (CCL_ERR_INVALID_ARG) everywhere else.  Buffers
    # sit far apart here, so no layout overlaps.
    nulls = {"rejected": 0, "accepted": 0}
    for it in range(iters):
        kind = ["reduce_scatter", "allgather", "gather", "scatter", "broadcast", "reduce", "allreduce"][it % 7]
        N = int(g.integers(1, 7))
        K = int(g.integers(1, 9))  # often fewer elements than ranks: empty chunks
        root = int(g.integers(0, N))
        q, rem = K // N, K % N
        ln = [q + (1 if c < rem else 0) for c in range(N)]
        send = [FAKE + (2 * r) * (1 << 20) for r in range(N)]
        recv = [FAKE + (2 * r + 1) * (1 << 20) for r in range(N)]
        for r in range(N):
            if g.random() < 0.25:
                send[r] = None
            if g.random() < 0.25:
                recv[r] = None
        need_send = {"reduce_scatter": [True] * N, "allgather": [ln[r] > 0 for r in range(N)],
                     "gather": [ln[r] > 0 for r in range(N)], "scatter": [r == root for r in range(N)],
                     "broadcast": [r == root for r in range(N)], "reduce": [True] * N,
                     "allreduce": [True] * N}[kind]
        need_recv = {"reduce_scatter": [ln[r] > 0 for r in range(N)], "allgather": [True] * N,
                     "gather": [r == root for r in range(N)], "scatter": [ln[r] > 0 for r in range(N)],
                     "broadcast": [True] * N, "reduce": [r == root for r in range(N)],
                     "allreduce": [True] * N}[kind]
        want_reject = any(need_send[r] and send[r] is None for r in range(N)) or \
            any(need_recv[r] and recv[r] is None for r in range(N))
        fn = {"reduce_scatter": lambda: L.ccl_reduce_scatter(_pp(send), _pp(recv), N, K, 0, 0, 0, stream),
              "allgather": lambda: L.ccl_allgather(_pp(send), _pp(recv), N, K, 0, 0, stream),
              "gather": lambda: L.ccl_gather(_pp(send), _pp(recv), N, root, K, 0, 0, stream),
              "scatter": lambda: L.ccl_scatter(_pp(send), _pp(recv), N, root, K, 0, 0, stream),
              "broadcast": lambda: L.ccl_broadcast(_pp(send), _pp(recv), N, root, K, 0, 0, stream),
              "reduce": lambda: L.ccl_reduce(_pp(send), _pp(recv), N, root, K, 0, 0, 0, stream),
              "allreduce": lambda: L.ccl_allreduce(_pp(send), _pp(recv), N, K, 0, 0, 0, stream)}[kind]
        got = fn()
        if want_reject:
            assert got == 1, (kind, N, K, root, send, recv, got)
            nulls["rejected"] += 1
        else:
            assert got in (0, CUDA_ERR), (kind, N, K, root, send, recv, got)
            nulls["accepted"] += 1
    assert nulls["rejected"] > iters // 10 and nulls["accepted"] > iters // 10, nulls
    print("validation fuzz ok", seen, rooted, other, comp, same, nulls)


if __name__ == "__main__":
    assert os.environ.get("CUDA_VISIBLE_DEVICES") == "", "run with CUDA_VISIBLE_DEVICES=''"
    main()
