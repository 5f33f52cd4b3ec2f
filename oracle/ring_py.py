"""Tiny pure-Python ring collectives -- TEST INFRASTRUCTURE ONLY, small cases.

A second statement of the ring AllReduce, in Python loops over Python
integers (bit patterns), written independently of ``ring_oracle.c``.  The tests
compare the two bit for bit on small inputs and check this one against the
pages' worked examples.  Like the rest of ``oracle/`` it may be used only by
``tests/``.

The schedule (Collectives and sharded matmul, slides "ring ReduceScatter" and
"ring AllGather"; Lesson 3, reference solution, which snapshots every send of a
step before any receive is applied):

  ReduceScatter step s = 0..N-2: rank i sends its current chunk (i-s) mod N to
  rank i+1; rank i combines the chunk (i-1-s) mod N arriving from rank i-1
  into its own copy (local first, then incoming).
  AllGather step s = 0..N-2: rank i sends chunk (i+1-s) mod N; rank i stores
  the chunk (i-s) mod N arriving from rank i-1.

Chunk c of K elements holds K // N + (c < K % N) elements.  Each combination
is one IEEE binary32 operation rounded to nearest-even, then a round to the
buffer type.  A binary32 sum, product or quotient of two binary32 values is
taken here in binary64 and rounded once to binary32; 53 >= 2 * 24 + 2, so that
double rounding gives the correctly rounded binary32 result.  Readings where
the pages are silent: a NaN result is the quiet NaN 0x7FFFFFFF; MAX and MIN
return NaN if either side is NaN, else the larger (smaller) value, with +0
beating -0 in MAX and -0 beating +0 in MIN; AVG divides the finished chunk once
by N at the rank that holds it; the pre-multiplied AVG scales every
contribution by the binary32 reciprocal of N first, rounds it to the buffer
type, and sums.
"""
from __future__ import annotations

import math
import struct

import numpy as np

NAN32 = 0x7FFFFFFF


def f32_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))[0]


def f32_bits(x: float) -> int:
    """Round a binary64 value to binary32 (nearest-even, overflow to infinity)."""
    if math.isnan(x):
        return NAN32
    if math.isinf(x):
        return 0x7F800000 if x > 0 else 0xFF800000
    with np.errstate(over="ignore"):
        y = np.float32(x)  # IEEE conversion, round to nearest-even
    return int(np.array([y], dtype=np.float32).view(np.uint32)[0])


def bf16_from_f32(bits: int) -> int:
    """Round a binary32 bit pattern to bfloat16, nearest-even; a NaN keeps its
    sign and top payload bits and becomes quiet."""
    if (bits & 0x7F800000) == 0x7F800000 and (bits & 0x007FFFFF):
        return ((bits >> 16) | 0x0040) & 0xFFFF
    upper, lower = bits >> 16, bits & 0xFFFF
    if lower > 0x8000 or (lower == 0x8000 and (upper & 1)):
        upper += 1
    return upper & 0xFFFF


def _is_nan(bits: int) -> bool:
    return (bits & 0x7F800000) == 0x7F800000 and (bits & 0x007FFFFF) != 0


def _binop(a: int, b: int, op: str) -> int:
    """One binary32 operation on binary32 bit patterns."""
    if op in ("max", "min"):
        if _is_nan(a) or _is_nan(b):
            return NAN32
        x, y = f32_value(a), f32_value(b)
        if x == y:  # equal values: only +0 / -0 can differ in bits
            return (a & b) if op == "max" else (a | b)
        return a if (x > y) == (op == "max") else b
    x, y = f32_value(a), f32_value(b)
    r = x * y if op == "prod" else x + y
    return f32_bits(r)


def _canon(bits: int) -> int:
    return NAN32 if _is_nan(bits) else bits


class _Type:
    def __init__(self, bf16: bool):
        self.bf16 = bf16

    def widen(self, v: int) -> int:
        return (v << 16) if self.bf16 else v

    def narrow(self, bits: int) -> int:
        return bf16_from_f32(bits) if self.bf16 else bits


def partition(K: int, N: int):
    lens = [K // N + (1 if c < K % N else 0) for c in range(N)]
    offs = [sum(lens[:c]) for c in range(N)]
    return offs, lens


def reduce_scatter(bufs, op: str = "sum"):
    """ReduceScatter as the ring computes it: the ReduceScatter phase leaves
    chunk c finished at rank c-1, which hands it to rank c.  Returns one
    array per rank (chunk r for rank r)."""
    buf, T, offs, lens, _ = _reduce_scatter_phase(bufs, op)
    N = len(buf)
    out = []
    for r in range(N):
        row = buf[(r - 1) % N][offs[r]:offs[r] + lens[r]]
        out.append(np.array(row, dtype=np.uint16) if T.bf16 else np.array(row, dtype=np.uint32).view(np.float32))
    return out


def _reduce_scatter_phase(bufs, op):
    """The N-1 ReduceScatter steps (and AVG's one division at each holder) on
    copies of bufs.  Returns (buffers as bit patterns, type, offsets, lengths,
    elements sent per rank)."""
    arrs = [np.ascontiguousarray(b) for b in bufs]
    bf16 = arrs[0].dtype == np.uint16
    T = _Type(bf16)
    N, K = len(arrs), arrs[0].size
    buf = [[int(v) for v in (a if bf16 else a.view(np.uint32))] for a in arrs]
    offs, lens = partition(K, N)
    sent = [0] * N
    ring_op = "sum" if op in ("avg", "avg_premul") else op

    if op == "avg_premul":  # every contribution scaled by rn(1/N) and rounded to the type
        inv = f32_value(f32_bits(1.0 / N))
        buf = [[T.narrow(_canon(f32_bits(f32_value(T.widen(v)) * inv))) for v in row] for row in buf]

    def chunk(c):
        return range(offs[c], offs[c] + lens[c])

    for s in range(N - 1):
        msgs = [[buf[i][e] for e in chunk((i - s) % N)] for i in range(N)]
        for i in range(N):
            c = (i - 1 - s) % N
            incoming = msgs[(i - 1) % N]
            for k, e in enumerate(chunk(c)):
                buf[i][e] = T.narrow(_canon(_binop(T.widen(buf[i][e]), T.widen(incoming[k]), ring_op)))
            sent[(i - 1) % N] += lens[c]
    if op == "avg":  # once, at the rank holding the finished chunk (i+1) mod N
        for i in range(N):
            for e in chunk((i + 1) % N):
                buf[i][e] = T.narrow(_canon(f32_bits(f32_value(T.widen(buf[i][e])) / N)))
    return buf, T, offs, lens, sent


def ring_allreduce(bufs, op: str = "sum"):
    """bufs: N equal-length numpy arrays (float32, or uint16 bf16 bit patterns).
    Returns (outputs as arrays of the same kind, elements sent per rank)."""
    buf, T, offs, lens, sent = _reduce_scatter_phase(bufs, op)
    N = len(buf)
    bf16 = T.bf16

    def chunk(c):
        return range(offs[c], offs[c] + lens[c])

    for s in range(N - 1):  # AllGather phase
        msgs = [[buf[i][e] for e in chunk((i + 1 - s) % N)] for i in range(N)]
        for i in range(N):
            c = (i - s) % N
            incoming = msgs[(i - 1) % N]
            for k, e in enumerate(chunk(c)):
                buf[i][e] = incoming[k]
            sent[(i - 1) % N] += lens[c]

    if bf16:
        outs = [np.array(row, dtype=np.uint16) for row in buf]
    else:
        outs = [np.array(row, dtype=np.uint32).view(np.float32) for row in buf]
    return outs, sent


# ------------------------------------------------------------------ compressed AllReduce with error feedback
# (Collective Communication: "Blockwise quantization for gradient
# communication", the greedy 1-bit compressor of Tables 3 and 4, "Top-k
# sparsification", and error feedback, Definition 1.4: e_{t+1} = g_t + e_t - v_t.)
# Each rank compresses u = g + e (binary32) to the transmitted v and keeps
# e' = u - v; the v's are AllReduced by the ring above in binary32 (SUM, or AVG
# dividing once by N) and the result is rounded once to the gradient type.
# numpy binary32 array operations are single IEEE operations (round to
# nearest-even, no contraction); NaN results are made the quiet NaN 0x7FFFFFFF.

def _canon_f32(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32).copy()
    a.view(np.uint32)[np.isnan(a)] = NAN32
    return a


def _int8_block(u: np.ndarray, block: int) -> np.ndarray:
    """v for one rank: per block of `block` elements s = max|u| / 127 (NaN if
    the block holds a NaN), q = u / s rounded to an integer with ties to even
    (0 when s = 0), v = q * s."""
    v = np.empty_like(u)
    with np.errstate(all="ignore"):
        for b0 in range(0, u.size, block):
            blk = u[b0:b0 + block]
            if np.isnan(blk).any():
                s = np.float32(np.nan)
            else:
                s = _canon_f32(np.abs(blk).max(initial=np.float32(0)) / np.float32(127))[()]
            if s > 0:
                q = np.rint(_canon_f32(blk / s))  # IEEE roundToIntegralTiesToEven
            elif s == 0:
                q = np.zeros_like(blk)
            else:  # NaN scale
                q = np.full_like(blk, s)
            v[b0:b0 + block] = _canon_f32(_canon_f32(q) * s)
    return v


def _top_k(u: np.ndarray, k: int) -> np.ndarray:
    """v = u where the magnitude key (the bit pattern of |u|, so NaN ranks
    above every number) reaches the k-th largest key, else 0."""
    keys = u.view(np.uint32) & np.uint32(0x7FFFFFFF)
    if k <= 0 or u.size == 0:
        return np.zeros_like(u)
    tau = np.sort(keys)[::-1][min(k, u.size) - 1]
    return np.where(keys >= tau, u, np.float32(0)).astype(np.float32)


def allreduce_compressed(grads, residuals, op: str = "sum", comp: str = "int8_block", block: int = 128,
                         threshold: float = 0.5, k: int = 0):
    """One step.  grads: N arrays (float32, or uint16 bf16 patterns); residuals:
    N float32 arrays.  Returns (new grads, new residuals); inputs untouched."""
    if op not in ("sum", "avg"):
        raise ValueError("compressed AllReduce takes SUM or AVG")
    bf16 = np.asarray(grads[0]).dtype == np.uint16
    sent, res = [], []
    with np.errstate(all="ignore"):
        for g, e in zip(grads, residuals):
            g32 = (np.asarray(g, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32) if bf16 \
                else np.asarray(g, dtype=np.float32)
            u = _canon_f32(g32 + np.asarray(e, dtype=np.float32))
            if comp == "int8_block":
                v = _int8_block(u, block)
            elif comp == "threshold":
                v = np.where(u >= np.float32(threshold), np.float32(1), np.float32(0)).astype(np.float32)
            elif comp == "topk":
                v = _top_k(u, k)
            else:
                raise ValueError(comp)
            res.append(_canon_f32(u - v))
            sent.append(v)
    total, _ = ring_allreduce(sent, op)
    if bf16:
        out = [np.array([bf16_from_f32(int(b)) for b in t.view(np.uint32)], dtype=np.uint16) for t in total]
    else:
        out = [t.copy() for t in total]
    return out, res


# ------------------------------------------------------------------ other schedules, step by step
# The fold orders of the other AllReduce schedules the pages describe, each
# simulated step by step on whole buffers (the C oracle has its own step
# simulations and per-element closed forms; this is a third statement).

def _load(bufs):
    arrs = [np.ascontiguousarray(b) for b in bufs]
    bf16 = arrs[0].dtype == np.uint16
    return [[int(v) for v in (a if bf16 else a.view(np.uint32))] for a in arrs], _Type(bf16)


def _store(buf, T):
    if T.bf16:
        return [np.array(row, dtype=np.uint16) for row in buf]
    return [np.array(row, dtype=np.uint32).view(np.float32) for row in buf]


def _combine(T, a, b, op):
    return T.narrow(_canon(_binop(T.widen(a), T.widen(b), op)))


def _divide(T, a, n):
    return T.narrow(_canon(f32_bits(f32_value(T.widen(a)) / n)))


def allreduce_halving_doubling(bufs, op: str = "sum"):
    """Recursive halving then doubling (Collective Communication, "Recursive
    halving-doubling"; distance doubling: round k pairs rank v with v XOR 2^k,
    and the rank whose bit k is 0 keeps the lower half of its current range,
    rounded up).  N not a power of two: with P the largest power of two <= N
    and r = N - P, rank 2v+1 first adds rank 2v's buffer (v < r) and stands in
    for both; the virtual ranks are 2v+1 (v < r) and v + r (v >= r); rank 2v
    receives the result at the end.  AVG divides once by N."""
    if op not in ("sum", "avg", "max", "min", "prod"):
        raise ValueError(op)
    buf, T = _load(bufs)
    N, K = len(buf), len(buf[0])
    sop = "sum" if op == "avg" else op
    P = 1
    while P * 2 <= N:
        P *= 2
    r = N - P
    for v in range(r):
        buf[2 * v + 1] = [_combine(T, a, b, sop) for a, b in zip(buf[2 * v + 1], buf[2 * v])]
    real = [2 * v + 1 if v < r else v + r for v in range(P)]
    lo, hi = [0] * P, [K] * P
    rounds = P.bit_length() - 1
    for k in range(rounds):  # halving: exchange and combine half of the current range
        snap = [list(buf[real[v]]) for v in range(P)]
        for v in range(P):
            p = v ^ (1 << k)
            mid = lo[v] + (hi[v] - lo[v] + 1) // 2
            keep = (lo[v], mid) if not v & (1 << k) else (mid, hi[v])
            row = buf[real[v]]
            for e in range(*keep):
                row[e] = _combine(T, row[e], snap[p][e], sop)
            lo[v], hi[v] = keep
    if op == "avg":
        for v in range(P):
            row = buf[real[v]]
            for e in range(lo[v], hi[v]):
                row[e] = _divide(T, row[e], N)
    for k in reversed(range(rounds)):  # doubling: exchange the finished ranges
        snap = [list(buf[real[v]]) for v in range(P)]
        rng = list(zip(lo, hi))
        for v in range(P):
            p = v ^ (1 << k)
            row = buf[real[v]]
            for e in range(*rng[p]):
                row[e] = snap[p][e]
            lo[v], hi[v] = min(rng[v][0], rng[p][0]), max(rng[v][1], rng[p][1])
    for v in range(r):
        buf[2 * v] = list(buf[2 * v + 1])
    return _store(buf, T)


def allreduce_binomial_tree(bufs, op: str = "sum"):
    """Reduce up a binomial tree rooted at rank 0, then broadcast down
    (Collective Communication, "Tree AllReduce"): at level k every rank i that
    is a multiple of 2^(k+1) adds rank i + 2^k's buffer, if that rank exists.
    AVG divides once by N at the root."""
    if op not in ("sum", "avg", "max", "min", "prod"):
        raise ValueError(op)
    buf, T = _load(bufs)
    N = len(buf)
    sop = "sum" if op == "avg" else op
    step = 1
    while step < N:
        for i in range(0, N, 2 * step):
            if i + step < N:
                buf[i] = [_combine(T, a, b, sop) for a, b in zip(buf[i], buf[i + step])]
        step *= 2
    if op == "avg":
        buf[0] = [_divide(T, a, N) for a in buf[0]]
    return _store([list(buf[0]) for _ in range(N)], T)


def allreduce_hierarchical(bufs, L: int, op: str = "sum"):
    """Two-level AllReduce (AllReduce survey, two-level table): groups of L
    consecutive ranks; a ring ReduceScatter inside every group over L chunks
    (chunk c finished at local rank c-1); a ring AllReduce of chunk c across
    the groups' holders, chunk c cut into G = N / L sub-chunks; then a ring
    AllGather inside every group.  AVG divides once by N."""
    if op not in ("sum", "avg", "max", "min", "prod"):
        raise ValueError(op)
    arrs = [np.ascontiguousarray(b) for b in bufs]
    N, K = len(arrs), arrs[0].size
    if L < 1 or N % L:
        raise ValueError("group size must divide the rank count")
    G = N // L
    sop = "sum" if op == "avg" else op
    offs, lens = partition(K, L)
    T = _Type(arrs[0].dtype == np.uint16)
    out = [None] * N
    # 1. ring ReduceScatter inside every group
    grp = []
    for g in range(G):
        b, _, _, _, _ = _reduce_scatter_phase(arrs[g * L:(g + 1) * L], sop)
        grp.append(b)
    result = [0] * K
    # 2. ring AllReduce of every chunk across the groups' holders
    for c in range(L):
        holder = (c - 1) % L
        rows = [grp[g][holder][offs[c]:offs[c] + lens[c]] for g in range(G)]
        rows = [np.array(rw, dtype=np.uint16) if T.bf16 else np.array(rw, dtype=np.uint32).view(np.float32)
                for rw in rows]
        red, _ = ring_allreduce(rows, sop)
        vals = [int(v) for v in (red[0] if T.bf16 else red[0].view(np.uint32))]
        if op == "avg":
            vals = [_divide(T, a, N) for a in vals]
        result[offs[c]:offs[c] + lens[c]] = vals
    # 3. ring AllGather inside every group: every rank receives every chunk
    for i in range(N):
        out[i] = list(result)
    return _store(out, T)


# ------------------------------------------------------------------ the other collectives

def reduce(bufs, root: int, op: str = "sum"):
    """Reduce(root): the root receives the AllReduce's bits, the other ranks
    keep their buffers (Lesson 3, core concepts: AllReduce = Reduce followed by
    Broadcast)."""
    out = [np.array(b, copy=True) for b in bufs]
    out[root] = ring_allreduce(bufs, op)[0][root]
    return out


def allgather(chunks, K: int):
    """Every rank receives the concatenation, in rank order, of the ranks'
    chunks (chunk r of the K-element partition comes from rank r)."""
    offs, lens = partition(K, len(chunks))
    full = np.concatenate([np.asarray(c)[:lens[r]] for r, c in enumerate(chunks)]) if K else \
        np.zeros(0, dtype=np.asarray(chunks[0]).dtype)
    return [full.copy() for _ in chunks]


def gather(chunks, K: int) -> np.ndarray:
    """The root's concatenation of the ranks' chunks."""
    return allgather(chunks, K)[0]


def scatter(root_buf, N: int):
    """Rank r receives chunk r of the root's buffer."""
    src = np.asarray(root_buf)
    offs, lens = partition(src.size, N)
    return [src[offs[r]:offs[r] + lens[r]].copy() for r in range(N)]


def broadcast(bufs, root: int):
    return [np.array(bufs[root], copy=True) for _ in bufs]


def alltoallv(sends, counts):
    """recv_j holds, in source order, the counts[i][j] elements rank i sends to
    rank j; send_i holds its blocks in destination order."""
    counts = np.asarray(counts, dtype=np.int64)
    N = len(sends)
    recv = []
    for j in range(N):
        parts = []
        for i in range(N):
            start = int(counts[i, :j].sum())
            parts.append(np.asarray(sends[i])[start:start + int(counts[i, j])])
        recv.append(np.concatenate(parts) if parts else np.zeros(0, dtype=np.asarray(sends[0]).dtype))
    return recv


def bucket_allreduce(tensors, bucket_elems: int, op: str = "sum"):
    """Bucket fusion (Collective Communication, "Bucket fusion"): every rank's
    tensors are laid end to end in reverse registration order, the stream is
    cut into buckets of bucket_elems (the last one partial; a tensor may span
    buckets) and every bucket is ring-AllReduced on its own, with its own chunk
    partition.  tensors[r][t]; returns new arrays."""
    N, T = len(tensors), len(tensors[0])
    streams = [np.concatenate([np.asarray(tensors[r][t]) for t in reversed(range(T))]) for r in range(N)]
    total = streams[0].size
    for b0 in range(0, total, bucket_elems):
        b1 = min(b0 + bucket_elems, total)
        red, _ = ring_allreduce([s[b0:b1] for s in streams], op)
        for r in range(N):
            streams[r][b0:b1] = red[r]
    out = []
    for r in range(N):
        row, pos = [None] * T, 0
        for t in reversed(range(T)):
            n = np.asarray(tensors[r][t]).size
            row[t] = streams[r][pos:pos + n].copy()
            pos += n
        out.append(row)
    return out
