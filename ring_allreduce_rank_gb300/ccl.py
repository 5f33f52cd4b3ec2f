"""Thin Python binding of libccl.so (include/ccl.h).

Argument marshalling only: torch tensors become device pointers, element
counts and dtype codes, and the call goes straight to the C ABI, which runs
every step in the library's own CUDA kernels.  There is no fallback: if the
library is not built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from .build import LIB as _LIB_PATH

FP32, BF16 = 0, 1
SUM, AVG, MAX, PROD, MIN, AVG_PREMUL = 0, 1, 2, 3, 4, 5
FUSED, STEP = 0, 1
OPS = {"sum": SUM, "avg": AVG, "max": MAX, "prod": PROD, "min": MIN, "avg_premul": AVG_PREMUL}
MODES = {"fused": FUSED, "step": STEP}
ALGOS = {"ring": 0, "halving_doubling": 1, "tree": 2, "hierarchical": 3}
COMPRESSORS = {"int8_block": 0, "threshold": 1, "topk": 2}
STATUS = {0: "CCL_OK", 1: "CCL_ERR_INVALID_ARG", 2: "CCL_ERR_UNSUPPORTED", 3: "CCL_ERR_OVERLAP",
          4: "CCL_ERR_CUDA", 5: "CCL_ERR_NO_MEMORY", 6: "CCL_ERR_TIMEOUT", 7: "CCL_ERR_CHECK_FAILED"}
MAX_RANKS = 1024
DEFAULT_BUCKET_BYTES = 25 * 1024 * 1024
HOST_WORK_BYTES_DEFAULT = 192 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class Config(ctypes.Structure):
    """ccl_config_t."""
    _fields_ = [("mode_override", ctypes.c_int), ("trace", ctypes.c_int), ("check", ctypes.c_int),
                ("host_path", ctypes.c_int), ("default_bucket_bytes", ctypes.c_size_t)]


class CclError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s" % (where, STATUS.get(status, status)))


def lib() -> ctypes.CDLL:
    """Load libccl.so (built in-tree); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            # CCL_LIBRARY: another build of this library to load (the
            # bounds-checking debug build, libccl_debug.so)
            path = os.environ.get("CCL_LIBRARY") or _LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError("libccl.so is not built (%s); run `python -m ring_allreduce_rank_gb300.build` "
                                   "or __graft_entry__.build()" % path)
            L = ctypes.CDLL(path)
            vp, pp, i32, sz = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_size_t
            psz = ctypes.POINTER(ctypes.c_size_t)
            sig = {
                "ccl_allreduce": [pp, pp, i32, sz, i32, i32, i32, vp],
                "ccl_reduce_scatter": [pp, pp, i32, sz, i32, i32, i32, vp],
                "ccl_allgather": [pp, pp, i32, sz, i32, i32, vp],
                "ccl_broadcast": [pp, pp, i32, i32, sz, i32, i32, vp],
                "ccl_reduce": [pp, pp, i32, i32, sz, i32, i32, i32, vp],
                "ccl_allreduce_algo": [pp, pp, i32, sz, i32, i32, i32, i32, vp],
                "ccl_allreduce_compressed": [pp, pp, i32, sz, i32, i32, i32, i32, ctypes.c_float, vp],
                "ccl_plan_compressed_bytes": [sz, i32, i32, psz],
                "ccl_allreduce_topk": [pp, pp, i32, sz, i32, i32, sz, vp, sz, vp],
                "ccl_plan_topk_work_bytes": [i32, psz],
                "ccl_plan_topk_sample": [sz, sz, ctypes.POINTER(ctypes.c_uint32)],
                "ccl_plan_topk_bytes": [sz, sz, psz],
                "ccl_gather": [pp, pp, i32, i32, sz, i32, i32, vp],
                "ccl_scatter": [pp, pp, i32, i32, sz, i32, i32, vp],
                "ccl_alltoall": [pp, pp, i32, sz, i32, i32, vp],
                "ccl_alltoallv": [pp, pp, i32, psz, i32, i32, vp],
                "ccl_bucket_allreduce": [pp, psz, i32, i32, sz, i32, i32, i32, vp],
                "ccl_plan_chunks": [sz, i32, psz, psz],
                "ccl_plan_ring_schedule": [i32, ctypes.POINTER(ctypes.c_int32)],
                "ccl_plan_buckets": [psz, i32, sz, psz, sz, psz],
                "ccl_plan_alltoallv": [i32, psz, psz, psz],
                "ccl_arena_layout": [i32, sz, sz, psz, psz],
                "ccl_allreduce_host": [pp, pp, i32, sz, i32, i32, vp, sz, vp],
                "ccl_plan_host_slices": [sz, i32, i32, sz, psz, psz, sz, psz],
                "ccl_finalize": [],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.ccl_bucketer_create.argtypes = [pp, psz, i32, i32, sz, i32, i32, i32, ctypes.POINTER(vp)]
            L.ccl_bucketer_mark_ready.argtypes = [vp, i32, vp, vp]
            L.ccl_bucketer_reset.argtypes = [vp]
            L.ccl_bucketer_status.argtypes = [vp, psz, psz]
            L.ccl_bucketer_destroy.argtypes = [vp]
            for name in ("ccl_bucketer_create", "ccl_bucketer_mark_ready", "ccl_bucketer_reset",
                         "ccl_bucketer_status", "ccl_bucketer_destroy"):
                getattr(L, name).restype = ctypes.c_int
            L.ccl_check_identical.argtypes = [pp, i32, sz, i32, vp, vp]
            L.ccl_check_identical.restype = ctypes.c_int
            L.ccl_debug_faults.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_ulonglong)]
            L.ccl_debug_faults.restype = ctypes.c_int
            L.ccl_set_check.argtypes = [i32]
            L.ccl_set_check.restype = None
            L.ccl_check_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
            L.ccl_check_read.restype = ctypes.c_int
            L.ccl_set_trace.argtypes = [i32]
            L.ccl_set_trace.restype = None
            L.ccl_trace_read.argtypes = [vp, sz]
            L.ccl_trace_read.restype = sz
            L.ccl_trace_clear.argtypes = []
            L.ccl_trace_clear.restype = None
            L.ccl_step_sent.argtypes = [i32, ctypes.POINTER(ctypes.c_ulonglong), i32]
            L.ccl_step_sent.restype = ctypes.c_int
            L.ccl_get_config.argtypes = [ctypes.POINTER(Config)]
            L.ccl_get_config.restype = ctypes.c_int
            L.ccl_set_mode_override.argtypes = [i32]
            L.ccl_set_mode_override.restype = ctypes.c_int
            L.ccl_set_default_bucket_bytes.argtypes = [sz]
            L.ccl_set_default_bucket_bytes.restype = ctypes.c_int
            L.ccl_set_host_path.argtypes = [i32]
            L.ccl_set_host_path.restype = ctypes.c_int
            L.ccl_status_string.argtypes = [ctypes.c_int]
            L.ccl_status_string.restype = ctypes.c_char_p
            L.ccl_version.argtypes = []
            L.ccl_version.restype = ctypes.c_int
            L.ccl_launch_count.argtypes = []
            L.ccl_launch_count.restype = ctypes.c_ulonglong
            _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise CclError(status, where)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return FP32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("ccl supports float32 and bfloat16 tensors, got %s" % t.dtype)


def _ptrs(ts: Sequence[Optional[torch.Tensor]]) -> ctypes.Array:
    vals = []
    for t in ts:
        if t is None:
            vals.append(None)
            continue
        if not t.is_contiguous():
            raise ValueError("rank buffers must be contiguous")
        vals.append(t.data_ptr())
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _op(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _sizes(vals) -> ctypes.Array:
    vals = [int(v) for v in vals]
    return (ctypes.c_size_t * max(1, len(vals)))(*vals)


# ------------------------------------------------------------------ collectives

def ccl_allreduce(send: Sequence[torch.Tensor], recv: Optional[Sequence[torch.Tensor]] = None, op="sum",
                  mode="fused", stream=None) -> None:
    """AllReduce over len(send) simulated ranks; recv=None means in place."""
    recv = send if recv is None else recv
    n = len(send)
    _check(lib().ccl_allreduce(_ptrs(send), _ptrs(recv), n, send[0].numel(), _dtype(send[0]), _op(op), _mode(mode),
                               _stream(stream)), "ccl_allreduce")


def ccl_allreduce_host(send: Sequence[torch.Tensor], recv: Optional[Sequence[torch.Tensor]] = None, op="sum",
                       work: Optional[torch.Tensor] = None, stream=None) -> None:
    """AllReduce of rank buffers in host memory (CPU tensors; pinned ones let
    the copies overlap), staged through `work`, a contiguous CUDA tensor the
    caller owns (HOST_WORK_BYTES_DEFAULT bytes run at the link's speed)."""
    if work is None or not work.is_cuda or not work.is_contiguous():
        raise ValueError("ccl_allreduce_host needs a contiguous CUDA work tensor")
    recv = send if recv is None else recv
    _check(lib().ccl_allreduce_host(_ptrs(send), _ptrs(recv), len(send), send[0].numel(), _dtype(send[0]), _op(op),
                                    ctypes.c_void_p(work.data_ptr()), work.numel() * work.element_size(),
                                    _stream(stream)), "ccl_allreduce_host")


def ccl_allreduce_algo(send: Sequence[torch.Tensor], recv: Optional[Sequence[torch.Tensor]] = None, op="sum",
                       algo="halving_doubling", group_size: int = 0, stream=None) -> None:
    """AllReduce under another schedule's summation order (one pass)."""
    recv = send if recv is None else recv
    a = ALGOS[algo] if isinstance(algo, str) else int(algo)
    _check(lib().ccl_allreduce_algo(_ptrs(send), _ptrs(recv), len(send), send[0].numel(), _dtype(send[0]), _op(op),
                                    a, int(group_size), _stream(stream)), "ccl_allreduce_algo")


def ccl_allreduce_compressed(grads: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor], op="sum",
                             comp="int8_block", block: int = 128, threshold: float = 0.5, stream=None) -> None:
    """One compressed AllReduce step with error feedback, in place on grads
    and residuals (fp32, one per rank)."""
    for e in residuals:
        if e.dtype != torch.float32:
            raise TypeError("residuals are float32")
    c = COMPRESSORS[comp] if isinstance(comp, str) else int(comp)
    _check(lib().ccl_allreduce_compressed(_ptrs(grads), _ptrs(residuals), len(grads), grads[0].numel(),
                                          _dtype(grads[0]), _op(op), c, int(block), ctypes.c_float(threshold),
                                          _stream(stream)), "ccl_allreduce_compressed")


def ccl_allreduce_topk(grads: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor], k: int, op="sum",
                       work: Optional[torch.Tensor] = None, stream=None) -> None:
    """One Top-k sparsified AllReduce step with error feedback, in place on
    grads and residuals (fp32, one per rank).  work: a device buffer of at
    least ccl_plan_topk_work_bytes(N) bytes (allocated here when omitted)."""
    for e in residuals:
        if e.dtype != torch.float32:
            raise TypeError("residuals are float32")
    if work is None:
        work = torch.empty(ccl_plan_topk_work_bytes(len(grads)), dtype=torch.uint8, device=grads[0].device)
    _check(lib().ccl_allreduce_topk(_ptrs(grads), _ptrs(residuals), len(grads), grads[0].numel(), _dtype(grads[0]),
                                    _op(op), int(k), ctypes.c_void_p(work.data_ptr()), work.numel() * work.element_size(),
                                    _stream(stream)), "ccl_allreduce_topk")


def ccl_plan_topk_work_bytes(nranks: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().ccl_plan_topk_work_bytes(int(nranks), ctypes.byref(out)), "ccl_plan_topk_work_bytes")
    return out.value


def ccl_plan_topk_sample(count: int, k: int) -> int:
    """One run of 256 elements in this many is sampled by ccl_allreduce_topk
    (aligned buffers); 0 when it takes no sample."""
    out = ctypes.c_uint32()
    _check(lib().ccl_plan_topk_sample(int(count), int(k), ctypes.byref(out)), "ccl_plan_topk_sample")
    return out.value


def ccl_plan_topk_bytes(count: int, k: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().ccl_plan_topk_bytes(int(count), int(k), ctypes.byref(out)), "ccl_plan_topk_bytes")
    return out.value


def ccl_plan_compressed_bytes(count: int, comp="int8_block", block: int = 128) -> int:
    out = ctypes.c_size_t()
    c = COMPRESSORS[comp] if isinstance(comp, str) else int(comp)
    _check(lib().ccl_plan_compressed_bytes(count, c, block, ctypes.byref(out)), "ccl_plan_compressed_bytes")
    return out.value


def ccl_reduce_scatter(send: Sequence[torch.Tensor], recv: Sequence[torch.Tensor], op="sum", mode="fused",
                       stream=None) -> None:
    """recv[r] (len_r elements) receives chunk r of the ring reduction of send."""
    _check(lib().ccl_reduce_scatter(_ptrs(send), _ptrs(recv), len(send), send[0].numel(), _dtype(send[0]), _op(op),
                                    _mode(mode), _stream(stream)), "ccl_reduce_scatter")


def ccl_allgather(send: Sequence[torch.Tensor], recv: Sequence[torch.Tensor], mode="fused", stream=None) -> None:
    """send[r] is chunk r (len_r elements); every recv[q] gets all chunks."""
    _check(lib().ccl_allgather(_ptrs(send), _ptrs(recv), len(recv), recv[0].numel(), _dtype(recv[0]), _mode(mode),
                               _stream(stream)), "ccl_allgather")


def ccl_broadcast(send: Sequence[Optional[torch.Tensor]], recv: Sequence[torch.Tensor], root: int = 0,
                  mode="fused", stream=None) -> None:
    _check(lib().ccl_broadcast(_ptrs(send), _ptrs(recv), len(recv), int(root), recv[0].numel(), _dtype(recv[0]),
                               _mode(mode), _stream(stream)), "ccl_broadcast")


def ccl_reduce(send: Sequence[torch.Tensor], recv: Sequence[Optional[torch.Tensor]], root: int = 0, op="sum",
               mode="fused", stream=None) -> None:
    """Only recv[root] receives the reduction (the AllReduce's bits)."""
    n = len(send)
    _check(lib().ccl_reduce(_ptrs(send), _ptrs(recv), n, int(root), send[0].numel(), _dtype(send[0]), _op(op),
                            _mode(mode), _stream(stream)), "ccl_reduce")


def ccl_gather(send: Sequence[torch.Tensor], recv: Sequence[Optional[torch.Tensor]], root: int = 0, mode="fused",
               stream=None) -> None:
    """recv[root] receives every rank's slice (chunk r = send[r]) in rank order."""
    out = recv[root]
    _check(lib().ccl_gather(_ptrs(send), _ptrs(recv), len(send), int(root), out.numel(), _dtype(out), _mode(mode),
                            _stream(stream)), "ccl_gather")


def ccl_scatter(send: Sequence[Optional[torch.Tensor]], recv: Sequence[torch.Tensor], root: int = 0, mode="fused",
                stream=None) -> None:
    """send[root] is split into the N chunks; chunk r goes to recv[r]."""
    src = send[root]
    _check(lib().ccl_scatter(_ptrs(send), _ptrs(recv), len(recv), int(root), src.numel(), _dtype(src), _mode(mode),
                             _stream(stream)), "ccl_scatter")


def ccl_alltoall(send: Sequence[torch.Tensor], recv: Sequence[torch.Tensor], mode="fused", stream=None) -> None:
    n = len(send)
    if send[0].numel() % n:
        raise ValueError("uniform AllToAll needs numel divisible by the number of ranks")
    _check(lib().ccl_alltoall(_ptrs(send), _ptrs(recv), n, send[0].numel() // n, _dtype(send[0]), _mode(mode),
                              _stream(stream)), "ccl_alltoall")


def ccl_alltoallv(send: Sequence[torch.Tensor], recv: Sequence[torch.Tensor], counts, mode="fused",
                  stream=None) -> None:
    """counts[i][j] elements go from rank i to rank j (host data)."""
    n = len(send)
    flat = [int(counts[i][j]) for i in range(n) for j in range(n)]
    dt = _dtype(next(t for t in list(send) + list(recv) if t is not None))
    _check(lib().ccl_alltoallv(_ptrs(send), _ptrs(recv), n, _sizes(flat), dt, _mode(mode), _stream(stream)),
           "ccl_alltoallv")


def ccl_bucket_allreduce(tensors: Sequence[Sequence[torch.Tensor]], bucket_bytes: int = 0,
                         op="sum", mode="fused", stream=None) -> None:
    """tensors[r][t]: rank r's t-th gradient in registration order (in place).
    bucket_bytes = 0 takes the library's default bucket size (25 MiB, or
    CCL_BUCKET_MB / ccl_set_default_bucket_bytes)."""
    nranks, nt = len(tensors), len(tensors[0])
    flat = [tensors[r][t] for r in range(nranks) for t in range(nt)]
    numels = [tensors[0][t].numel() for t in range(nt)]
    _check(lib().ccl_bucket_allreduce(_ptrs(flat), _sizes(numels), nt, nranks, int(bucket_bytes),
                                      _dtype(flat[0]), _op(op), _mode(mode), _stream(stream)),
           "ccl_bucket_allreduce")


def ccl_check_identical(bufs: Sequence[torch.Tensor], mismatches: torch.Tensor, stream=None) -> None:
    """Adds to mismatches (a one-element int64 device tensor) the number of
    elements whose bits differ from rank 0's, over ranks 1..N-1."""
    if mismatches.dtype != torch.int64 or mismatches.numel() != 1 or not mismatches.is_cuda:
        raise TypeError("mismatches must be a one-element int64 CUDA tensor")
    _check(lib().ccl_check_identical(_ptrs(bufs), len(bufs), bufs[0].numel(), _dtype(bufs[0]),
                                     ctypes.c_void_p(mismatches.data_ptr()), _stream(stream)), "ccl_check_identical")


class TraceRecord(ctypes.Structure):
    _fields_ = [("collective", ctypes.c_char * 24), ("nranks", ctypes.c_int), ("dtype", ctypes.c_int),
                ("op", ctypes.c_int), ("mode", ctypes.c_int), ("status", ctypes.c_int), ("launches", ctypes.c_uint),
                ("count", ctypes.c_ulonglong), ("host_ns", ctypes.c_ulonglong), ("seq", ctypes.c_ulonglong),
                ("gpu_ns", ctypes.c_ulonglong)]


def ccl_debug_faults():
    """(accesses skipped, first address) in a bounds-checking debug build;
    raises CclError (CCL_ERR_UNSUPPORTED) in a release build."""
    n, a = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    _check(lib().ccl_debug_faults(ctypes.byref(n), ctypes.byref(a)), "ccl_debug_faults")
    return int(n.value), int(a.value)


def ccl_set_check(enabled: bool) -> None:
    """Automatic result checks after AllReduce, AllGather and Broadcast."""
    lib().ccl_set_check(1 if enabled else 0)


def ccl_check_read(reset: bool = True) -> int:
    """Mismatches counted by the automatic checks on the current device."""
    n = ctypes.c_ulonglong()
    _check(lib().ccl_check_read(ctypes.byref(n), 1 if reset else 0), "ccl_check_read")
    return int(n.value)


def ccl_set_trace(enabled: bool) -> None:
    lib().ccl_set_trace(1 if enabled else 0)


def ccl_trace_read(max_records: int = 4096):
    """The newest traced calls, oldest first, as dicts."""
    n = lib().ccl_trace_read(None, 0)
    n = min(n, max_records)
    buf = (TraceRecord * max(1, n))()
    n = lib().ccl_trace_read(ctypes.cast(buf, ctypes.c_void_p), n)
    return [{"collective": r.collective.decode(), "nranks": r.nranks, "dtype": r.dtype, "op": r.op, "mode": r.mode,
             "status": r.status, "launches": r.launches, "count": r.count, "host_ns": r.host_ns, "seq": r.seq,
             "gpu_ns": r.gpu_ns}
            for r in buf[:n]]


def ccl_trace_clear() -> None:
    lib().ccl_trace_clear()


def ccl_step_sent(nranks: int, reset: bool = True) -> list:
    """Elements each rank sent in the ring steps of this thread's step-mode
    calls since the last reset."""
    buf = (ctypes.c_ulonglong * nranks)()
    _check(lib().ccl_step_sent(int(nranks), buf, 1 if reset else 0), "ccl_step_sent")
    return [int(v) for v in buf]


def ccl_get_config() -> dict:
    """The library's settings: mode override ("fused", "step" or None),
    trace, check, default bucket bytes, the host-buffer AllReduce's path
    ("staged" or "direct")."""
    c = Config()
    _check(lib().ccl_get_config(ctypes.byref(c)), "ccl_get_config")
    names = {v: k for k, v in MODES.items()}
    return {"mode_override": names.get(c.mode_override), "trace": bool(c.trace), "check": bool(c.check),
            "default_bucket_bytes": int(c.default_bucket_bytes),
            "host_path": {v: k for k, v in HOST_PATHS.items()}.get(c.host_path, c.host_path)}


def ccl_set_mode_override(mode: Optional[str]) -> None:
    """Force "fused" or "step" on every call that takes a mode; None removes
    the override."""
    _check(lib().ccl_set_mode_override(-1 if mode is None else _mode(mode)), "ccl_set_mode_override")


HOST_PATHS = {"staged": 0, "direct": 1}


def ccl_set_host_path(path: str) -> None:
    """ccl_allreduce_host's path: "staged" (the default) or "direct" (in
    place over the host link when every buffer is page-locked host memory,
    else staged)."""
    if path not in HOST_PATHS:
        raise ValueError("host path must be 'staged' or 'direct', not %r" % (path,))
    _check(lib().ccl_set_host_path(HOST_PATHS[path]), "ccl_set_host_path")


def ccl_set_default_bucket_bytes(nbytes: int) -> None:
    """Bucket size for bucket_bytes = 0 (0 restores 25 MiB)."""
    _check(lib().ccl_set_default_bucket_bytes(int(nbytes)), "ccl_set_default_bucket_bytes")


class CclBucketer:
    """ccl_bucketer_*: per-bucket AllReduce launched as gradients become ready.
    tensors[r][t] as for ccl_bucket_allreduce; keep them alive while in use."""

    def __init__(self, tensors: Sequence[Sequence[torch.Tensor]], bucket_bytes: int = 0,
                 op="sum", max_ctas: int = 0):
        nranks, nt = len(tensors), len(tensors[0])
        self._tensors = tensors
        flat = [tensors[r][t] for r in range(nranks) for t in range(nt)]
        numels = [tensors[0][t].numel() for t in range(nt)]
        h = ctypes.c_void_p()
        _check(lib().ccl_bucketer_create(_ptrs(flat), _sizes(numels), nt, nranks, int(bucket_bytes), _dtype(flat[0]),
                                         _op(op), int(max_ctas), ctypes.byref(h)), "ccl_bucketer_create")
        self._h = h

    def mark_ready(self, tensor: int, event: Optional[torch.cuda.Event] = None, comm_stream=None) -> None:
        ev = ctypes.c_void_p(event.cuda_event) if event is not None else ctypes.c_void_p(0)
        _check(lib().ccl_bucketer_mark_ready(self._h, int(tensor), ev, _stream(comm_stream)), "ccl_bucketer_mark_ready")

    def reset(self) -> None:
        _check(lib().ccl_bucketer_reset(self._h), "ccl_bucketer_reset")

    def status(self):
        nb, nl = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().ccl_bucketer_status(self._h, ctypes.byref(nb), ctypes.byref(nl)), "ccl_bucketer_status")
        return nb.value, nl.value

    def close(self) -> None:
        if self._h:
            lib().ccl_bucketer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ planner

def ccl_plan_chunks(count: int, nranks: int):
    off, ln = (ctypes.c_size_t * nranks)(), (ctypes.c_size_t * nranks)()
    _check(lib().ccl_plan_chunks(count, nranks, off, ln), "ccl_plan_chunks")
    return list(off), list(ln)


def ccl_plan_ring_schedule(nranks: int):
    steps = max(nranks - 1, 0)
    n = max(1, 2 * steps * nranks * 3)
    buf = (ctypes.c_int32 * n)()
    _check(lib().ccl_plan_ring_schedule(nranks, buf), "ccl_plan_ring_schedule")
    flat = list(buf)[:2 * steps * nranks * 3]
    return [[[tuple(flat[((ph * steps + s) * nranks + i) * 3:((ph * steps + s) * nranks + i) * 3 + 3])
              for i in range(nranks)] for s in range(steps)] for ph in range(2)]


def ccl_plan_buckets(numels, bucket_elems: int):
    nb = ctypes.c_size_t()
    _check(lib().ccl_plan_buckets(_sizes(numels), len(numels), bucket_elems, None, 0, ctypes.byref(nb)),
           "ccl_plan_buckets")
    starts = (ctypes.c_size_t * (nb.value + 1))()
    _check(lib().ccl_plan_buckets(_sizes(numels), len(numels), bucket_elems, starts, nb.value, ctypes.byref(nb)),
           "ccl_plan_buckets")
    return list(starts)


def ccl_plan_alltoallv(counts):
    n = len(counts)
    flat = [int(counts[i][j]) for i in range(n) for j in range(n)]
    sd, rd = (ctypes.c_size_t * (n * n))(), (ctypes.c_size_t * (n * n))()
    _check(lib().ccl_plan_alltoallv(n, _sizes(flat), sd, rd), "ccl_plan_alltoallv")
    return [list(sd)[i * n:(i + 1) * n] for i in range(n)], [list(rd)[j * n:(j + 1) * n] for j in range(n)]


def ccl_plan_host_slices(count: int, nranks: int, dtype: str = "bf16", work_bytes: int = HOST_WORK_BYTES_DEFAULT):
    """[(off, len)] slices of ccl_allreduce_host, in elements per rank."""
    dt = {"fp32": FP32, "bf16": BF16}[dtype]
    n = ctypes.c_size_t()
    _check(lib().ccl_plan_host_slices(count, nranks, dt, work_bytes, None, None, 0, ctypes.byref(n)),
           "ccl_plan_host_slices")
    off, ln = (ctypes.c_size_t * max(1, n.value))(), (ctypes.c_size_t * max(1, n.value))()
    _check(lib().ccl_plan_host_slices(count, nranks, dt, work_bytes, off, ln, n.value, ctypes.byref(n)),
           "ccl_plan_host_slices")
    return list(zip(list(off)[:n.value], list(ln)[:n.value]))


def ccl_arena_layout(nranks: int, bytes_per_rank: int, align: int = 256):
    stride, total = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().ccl_arena_layout(nranks, bytes_per_rank, align, ctypes.byref(stride), ctypes.byref(total)),
           "ccl_arena_layout")
    return stride.value, total.value


def ccl_status_string(status: int) -> str:
    return lib().ccl_status_string(status).decode()


def ccl_launch_count() -> int:
    return int(lib().ccl_launch_count())


def ccl_finalize() -> None:
    _check(lib().ccl_finalize(), "ccl_finalize")
