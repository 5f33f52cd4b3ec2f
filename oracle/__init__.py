"""CPU oracle for the ring collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under test never does: it
shares no code with it, and a product path that reached this module would void
every parity claim.

The arithmetic lives in ``ring_oracle.c`` (plain C, built here with gcc
``-O2 -ffp-contract=off``); this module only compiles it and marshals numpy
arrays.  ``ring_py.py`` is a second, pure-Python statement of every collective
here (not of the alternative formulations -- threaded ring, closed forms, the
fp64 sum), for small inputs, written apart from the C code; the tests require
the two to agree bit for bit.  Buffers are numpy arrays: ``np.float32`` for fp32, ``np.uint16`` bit
patterns for bf16 (the oracle never needs a bf16 numpy type).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ring_oracle.c")
# ORACLE_LIB: a prebuilt copy to load instead (the mutation tests point it at
# copies of ring_oracle.c with one planted mistake each)
OVERRIDE = os.environ.get("ORACLE_LIB") or None
LIB = OVERRIDE or os.path.join(HERE, "_build", "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra"]

FP32, BF16 = 0, 1
SUM, AVG, MAX, PROD, MIN, AVG_PREMUL = 0, 1, 2, 3, 4, 5
OPS = {"sum": SUM, "avg": AVG, "max": MAX, "prod": PROD, "min": MIN, "avg_premul": AVG_PREMUL}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ring_oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    if OVERRIDE:
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc"] + CFLAGS + ["-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            u64, i32, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
            pp = ctypes.POINTER(ctypes.c_void_p)
            p64 = ctypes.POINTER(ctypes.c_uint64)
            L.oracle_round_bf16.argtypes = [ctypes.c_uint32]
            L.oracle_round_bf16.restype = ctypes.c_uint16
            L.oracle_round_bf16_array.argtypes = [vp, vp, u64]
            L.oracle_round_bf16_array.restype = None
            L.oracle_partition.argtypes = [u64, i32, p64, p64]
            L.oracle_partition.restype = None
            L.oracle_ring_schedule.argtypes = [i32, ctypes.POINTER(ctypes.c_int32)]
            L.oracle_ring_schedule.restype = None
            L.oracle_ring_allreduce.argtypes = [pp, i32, u64, i32, i32, p64]
            L.oracle_ring_allreduce_threads.argtypes = [pp, i32, u64, i32, i32, i32]
            L.oracle_ring_allreduce_threads_ex.argtypes = [pp, i32, u64, i32, i32, i32, i32, ctypes.c_long]
            L.oracle_ring_allreduce_closed.argtypes = [pp, pp, i32, u64, i32, i32]
            L.oracle_ring_allreduce_at.argtypes = [pp, i32, u64, i32, i32, p64, u64, vp]
            L.oracle_ring_allreduce_gathered.argtypes = [pp, i32, u64, i32, i32, p64, u64, vp]
            L.oracle_reduce_scatter.argtypes = [pp, pp, i32, u64, i32, i32]
            L.oracle_allgather.argtypes = [pp, pp, i32, u64, i32]
            L.oracle_reduce.argtypes = [pp, pp, i32, i32, u64, i32, i32]
            L.oracle_allreduce_compressed.argtypes = [pp, pp, i32, u64, i32, i32, i32, i32, ctypes.c_float]
            L.oracle_allreduce_compressed_k.argtypes = [pp, pp, i32, u64, i32, i32, i32, i32, ctypes.c_float, u64]
            L.oracle_allreduce_hd.argtypes = [pp, i32, u64, i32, i32]
            L.oracle_allreduce_tree.argtypes = [pp, i32, u64, i32, i32]
            L.oracle_allreduce_hier.argtypes = [pp, i32, i32, u64, i32, i32]
            L.oracle_allreduce_order_at.argtypes = [pp, i32, u64, i32, i32, i32, i32, p64, u64, vp]
            L.oracle_gather.argtypes = [pp, vp, i32, u64, i32]
            L.oracle_scatter.argtypes = [vp, pp, i32, u64, i32]
            L.oracle_broadcast.argtypes = [pp, pp, i32, i32, u64, i32]
            L.oracle_alltoallv.argtypes = [pp, pp, i32, p64, i32]
            L.oracle_bucket_allreduce.argtypes = [pp, p64, i32, i32, u64, i32, i32]
            L.oracle_sum_f64.argtypes = [pp, i32, u64, i32, i32, vp, vp]
            for name in ("oracle_ring_allreduce", "oracle_ring_allreduce_closed", "oracle_ring_allreduce_at",
                         "oracle_ring_allreduce_gathered", "oracle_reduce_scatter", "oracle_reduce", "oracle_gather",
                         "oracle_scatter", "oracle_allreduce_hd", "oracle_allreduce_tree", "oracle_allreduce_hier",
                         "oracle_allreduce_order_at", "oracle_allreduce_compressed", "oracle_allreduce_compressed_k",
                         "oracle_allgather", "oracle_broadcast", "oracle_alltoallv",
                         "oracle_bucket_allreduce", "oracle_sum_f64"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return FP32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("oracle buffers are float32 or uint16 (bf16 bit patterns), got %s" % a.dtype)


def _ptrs(arrs) -> ctypes.Array:
    for a in arrs:
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle buffers must be C-contiguous")
    return (ctypes.c_void_p * max(1, len(arrs)))(*[a.ctypes.data for a in arrs])


def _u64(vals) -> ctypes.Array:
    vals = list(vals)
    return (ctypes.c_uint64 * max(1, len(vals)))(*vals)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError("%s failed with code %d" % (what, rc))


def _op(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


# ---------------------------------------------------------------- API

def round_bf16(bits_f32: int) -> int:
    """fp32 bit pattern -> bf16 bit pattern, round to nearest even."""
    return int(lib().oracle_round_bf16(ctypes.c_uint32(bits_f32)))


def round_bf16_array(bits_f32: np.ndarray) -> np.ndarray:
    src = np.ascontiguousarray(bits_f32, dtype=np.uint32).ravel()
    out = np.empty(src.size, dtype=np.uint16)
    lib().oracle_round_bf16_array(src.ctypes.data, out.ctypes.data, src.size)
    return out


def partition(K: int, N: int):
    off, ln = (ctypes.c_uint64 * N)(), (ctypes.c_uint64 * N)()
    lib().oracle_partition(K, N, off, ln)
    return list(off), list(ln)


def ring_schedule(N: int) -> np.ndarray:
    """[phase][s][rank] -> (send chunk, recv chunk, source rank)."""
    steps = max(N - 1, 0)
    tab = np.zeros((2, steps, N, 3), dtype=np.int32)
    lib().oracle_ring_schedule(N, tab.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return tab


def ring_allreduce(bufs, op="sum"):
    """Step-faithful ring AllReduce.  Returns (outputs, elements sent per rank)."""
    outs = [np.array(b, copy=True, order="C") for b in bufs]
    N, K = len(outs), outs[0].size
    sent = (ctypes.c_uint64 * N)()
    _check(lib().oracle_ring_allreduce(_ptrs(outs), N, K, _dtype_code(outs[0]), _op(op), sent),
           "oracle_ring_allreduce")
    return outs, list(sent)


def ring_allreduce_threads(bufs, op="sum", threads: int = 0):
    """The step-by-step ring with the ranks spread over `threads` threads (0:
    one per rank) and a barrier per step; the same bits as ring_allreduce."""
    outs = [np.array(b, copy=True, order="C") for b in bufs]
    N, K = len(outs), outs[0].size
    _check(lib().oracle_ring_allreduce_threads(_ptrs(outs), N, K, _dtype_code(outs[0]), _op(op), threads or N),
           "oracle_ring_allreduce_threads")
    return outs


TIMED_OUT = 3


def ring_allreduce_threads_status(bufs, op="sum", threads: int = 0, withhold: int = -1, timeout_ms: int = 60000):
    """As ring_allreduce_threads, with the thread owning rank `withhold` leaving
    before its first send (a failed rank).  Returns (outputs, code): 0, or
    TIMED_OUT when the others' bounded waits ran out."""
    outs = [np.array(b, copy=True, order="C") for b in bufs]
    N, K = len(outs), outs[0].size
    rc = lib().oracle_ring_allreduce_threads_ex(_ptrs(outs), N, K, _dtype_code(outs[0]), _op(op), threads or N,
                                                withhold, timeout_ms)
    if rc not in (0, TIMED_OUT):
        _check(rc, "oracle_ring_allreduce_threads_ex")
    return outs, rc


def ring_allreduce_closed(bufs, op="sum"):
    ins = [np.ascontiguousarray(b) for b in bufs]
    outs = [np.empty_like(b) for b in ins]
    _check(lib().oracle_ring_allreduce_closed(_ptrs(ins), _ptrs(outs), len(ins), ins[0].size,
                                              _dtype_code(ins[0]), _op(op)), "oracle_ring_allreduce_closed")
    return outs


def ring_allreduce_at(bufs, idx, op="sum") -> np.ndarray:
    ins = [np.ascontiguousarray(b) for b in bufs]
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=ins[0].dtype)
    _check(lib().oracle_ring_allreduce_at(_ptrs(ins), len(ins), ins[0].size, _dtype_code(ins[0]), _op(op),
                                          idx.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), idx.size,
                                          out.ctypes.data), "oracle_ring_allreduce_at")
    return out


def ring_allreduce_gathered(vals, K: int, idx, op="sum") -> np.ndarray:
    """vals[r] = rank r's elements at the indices idx (of K-element buffers)."""
    ins = [np.ascontiguousarray(v) for v in vals]
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=ins[0].dtype)
    _check(lib().oracle_ring_allreduce_gathered(_ptrs(ins), len(ins), K, _dtype_code(ins[0]), _op(op),
                                                idx.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), idx.size,
                                                out.ctypes.data), "oracle_ring_allreduce_gathered")
    return out


def reduce_scatter(bufs, op="sum"):
    ins = [np.ascontiguousarray(b) for b in bufs]
    N, K = len(ins), ins[0].size
    _, ln = partition(K, N)
    outs = [np.empty(ln[r], dtype=ins[0].dtype) for r in range(N)]
    _check(lib().oracle_reduce_scatter(_ptrs(ins), _ptrs(outs), N, K, _dtype_code(ins[0]), _op(op)),
           "oracle_reduce_scatter")
    return outs


ALGOS = {"ring": 0, "halving_doubling": 1, "tree": 2, "hierarchical": 3}


def allreduce_algo(bufs, algo: str, op="sum", group: int = 0):
    """Step-by-step AllReduce under another schedule: halving_doubling, tree or
    hierarchical (group = ranks per group)."""
    outs = [np.array(b, copy=True, order="C") for b in bufs]
    N, K = len(outs), outs[0].size
    dt = _dtype_code(outs[0])
    if algo == "ring":
        return ring_allreduce(outs, op)[0]
    if algo == "halving_doubling":
        rc = lib().oracle_allreduce_hd(_ptrs(outs), N, K, dt, _op(op))
    elif algo == "tree":
        rc = lib().oracle_allreduce_tree(_ptrs(outs), N, K, dt, _op(op))
    elif algo == "hierarchical":
        rc = lib().oracle_allreduce_hier(_ptrs(outs), N, group, K, dt, _op(op))
    else:
        raise ValueError(algo)
    _check(rc, "oracle_allreduce_" + algo)
    return outs


def allreduce_algo_at(bufs, algo: str, idx, op="sum", group: int = 0) -> np.ndarray:
    """Closed form of another schedule's result at the listed indices."""
    ins = [np.ascontiguousarray(b) for b in bufs]
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=ins[0].dtype)
    _check(lib().oracle_allreduce_order_at(_ptrs(ins), len(ins), ins[0].size, _dtype_code(ins[0]), _op(op),
                                           ALGOS[algo], group, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                           idx.size, out.ctypes.data), "oracle_allreduce_order_at")
    return out


COMPRESSORS = {"int8_block": 0, "threshold": 1, "topk": 2}


def allreduce_compressed(grads, residuals, op="sum", comp="int8_block", block=128, threshold=0.5, k=0):
    """One compressed AllReduce step with error feedback.  Returns (new grads,
    new residuals); inputs are not modified.  k: elements kept per rank by the
    "topk" compressor."""
    g = [np.array(x, copy=True, order="C") for x in grads]
    e = [np.array(x, dtype=np.float32, copy=True, order="C") for x in residuals]
    N, K = len(g), g[0].size
    _check(lib().oracle_allreduce_compressed_k(_ptrs(g), _ptrs(e), N, K, _dtype_code(g[0]), _op(op),
                                               COMPRESSORS[comp], int(block), ctypes.c_float(threshold), int(k)),
           "oracle_allreduce_compressed_k")
    return g, e


def reduce(bufs, root: int, op="sum"):
    """Only rank root's buffer changes (to the AllReduce result); returns all N."""
    ins = [np.ascontiguousarray(b) for b in bufs]
    outs = [np.array(b, copy=True) for b in ins]
    _check(lib().oracle_reduce(_ptrs(ins), _ptrs(outs), len(ins), root, ins[0].size, _dtype_code(ins[0]), _op(op)),
           "oracle_reduce")
    return outs


def gather(chunks, K: int) -> np.ndarray:
    """chunks[r] = rank r's slice; returns the root's concatenation."""
    ins = [np.ascontiguousarray(c) for c in chunks]
    out = np.zeros(K, dtype=ins[0].dtype)
    _check(lib().oracle_gather(_ptrs(ins), out.ctypes.data, len(ins), K, _dtype_code(ins[0])), "oracle_gather")
    return out


def scatter(root_buf, N: int):
    src = np.ascontiguousarray(root_buf)
    _, ln = partition(src.size, N)
    outs = [np.zeros(ln[r], dtype=src.dtype) for r in range(N)]
    _check(lib().oracle_scatter(src.ctypes.data, _ptrs(outs), N, src.size, _dtype_code(src)), "oracle_scatter")
    return outs


def allgather(chunks, K: int):
    """chunks[r] = rank r's contribution (chunk r of the K-element result)."""
    ins = [np.ascontiguousarray(c) for c in chunks]
    N = len(ins)
    outs = [np.zeros(K, dtype=ins[0].dtype) for _ in range(N)]
    _check(lib().oracle_allgather(_ptrs(ins), _ptrs(outs), N, K, _dtype_code(ins[0])), "oracle_allgather")
    return outs


def broadcast(bufs, root: int):
    ins = [np.ascontiguousarray(b) for b in bufs]
    outs = [np.array(b, copy=True) for b in ins]
    _check(lib().oracle_broadcast(_ptrs(ins), _ptrs(outs), len(ins), root, ins[0].size, _dtype_code(ins[0])),
           "oracle_broadcast")
    return outs


def alltoallv(sends, counts: np.ndarray):
    """counts[i, j] elements from rank i to rank j."""
    ins = [np.ascontiguousarray(s) for s in sends]
    N = len(ins)
    counts = np.asarray(counts, dtype=np.uint64).reshape(N, N)
    outs = [np.zeros(int(counts[:, j].sum()), dtype=ins[0].dtype) for j in range(N)]
    _check(lib().oracle_alltoallv(_ptrs(ins), _ptrs(outs), N, _u64(counts.ravel()), _dtype_code(ins[0])),
           "oracle_alltoallv")
    return outs


def bucket_allreduce(tensors, bucket_elems: int, op="sum"):
    """tensors[r][t] = rank r's t-th registered gradient (flat arrays).  Returns new arrays."""
    N, T = len(tensors), len(tensors[0])
    outs = [[np.array(tensors[r][t], copy=True) for t in range(T)] for r in range(N)]
    flat = [outs[r][t] for r in range(N) for t in range(T)]
    numels = [outs[0][t].size for t in range(T)]
    _check(lib().oracle_bucket_allreduce(_ptrs(flat), _u64(numels), T, N, bucket_elems,
                                         _dtype_code(flat[0]), _op(op)), "oracle_bucket_allreduce")
    return outs


def sum_f64(bufs, op="sum"):
    """fp64 plain sum (or mean) and sum of |x| per element."""
    ins = [np.ascontiguousarray(b) for b in bufs]
    K = ins[0].size
    y, a = np.empty(K, np.float64), np.empty(K, np.float64)
    _check(lib().oracle_sum_f64(_ptrs(ins), len(ins), K, _dtype_code(ins[0]), _op(op), y.ctypes.data,
                                a.ctypes.data), "oracle_sum_f64")
    return y, a
