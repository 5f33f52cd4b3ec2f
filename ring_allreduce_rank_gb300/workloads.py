"""Seeded synthetic inputs for the ring collectives.

This module only draws random numbers and lays them out; it holds none of the
collectives' arithmetic.  Both the CUDA path and the CPU oracle are fed from
here, so they always see identical input bits.  Everything is generated on the
host with numpy's PCG64 generator (one generator per rank, seeded with
``seed_base + rank``) and returned as numpy arrays: ``float32`` for fp32 and
``uint16`` bit patterns for bf16 (fp32 draws rounded to bf16 with torch's CPU
round-to-nearest-even conversion).

The shapes follow the workloads the pages discuss: data-parallel gradient
buffers (Collective Communication, Definition 1.1: gradient synchronisation),
Llama-style layer gradients grouped into buckets (Collective Communication,
"Bucket fusion"), and top-1 MoE token dispatch over 64 experts on 8 ranks
(Collective Communication, the AllToAll napkin math for expert parallelism).
"""
from __future__ import annotations

import numpy as np
import torch

MiB = 1 << 20


def _gen(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), torch CPU RNE conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def integers_fp32(N: int, K: int, seed: int = 0, lo: int = -8, hi: int = 8) -> np.ndarray:
    """(N, K) uniform integers in [lo, hi] stored as fp32, one generator, rank-major.
    Every sum of up to 2^20 such values is exact in fp32."""
    return _gen(seed).integers(lo, hi + 1, size=(N, K)).astype(np.float32)


def normal_bf16(N: int, K: int, std: float = 1e-3, seed_base: int = 0) -> np.ndarray:
    """(N, K) bf16 bit patterns of Normal(0, std), rank r drawn from seed_base + r."""
    out = np.empty((N, K), dtype=np.uint16)
    for r in range(N):
        x = _gen(seed_base + r).standard_normal(K, dtype=np.float32)
        x *= np.float32(std)
        out[r] = to_bf16_bits(x)
    return out


def normal_fp32(N: int, K: int, std: float = 1.0, seed_base: int = 0) -> np.ndarray:
    out = np.empty((N, K), dtype=np.float32)
    for r in range(N):
        out[r] = _gen(seed_base + r).standard_normal(K, dtype=np.float32) * np.float32(std)
    return out


def uniform_fp32(N: int, K: int, lo: float = -1.0, hi: float = 1.0, seed_base: int = 0) -> np.ndarray:
    """(N, K) Uniform(lo, hi) fp32, rank r drawn from seed_base + r."""
    out = np.empty((N, K), dtype=np.float32)
    for r in range(N):
        u = _gen(seed_base + r).random(K, dtype=np.float32)
        out[r] = u * np.float32(hi - lo) + np.float32(lo)
    return out


def special_values_fp32() -> np.ndarray:
    """Edge values for the arithmetic: signed zeros, subnormals, extremes, inf, NaN."""
    bits = np.array([
        0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007fffff, 0x00800000, 0x3f800000,
        0xbf800000, 0x7f7fffff, 0xff7fffff, 0x7f800000, 0xff800000, 0x7fc00000, 0x7fa00001,
        0xffc00123, 0x3f808000, 0x3f818000, 0x00008000, 0x00018000, 0x7f7f8000, 0x7f7f7fff,
    ], dtype=np.uint32)
    return bits.view(np.float32)


def mixed_fp32(N: int, K: int, seed_base: int = 0, special_frac: float = 0.05) -> np.ndarray:
    """Normal values of widely varying magnitude with a sprinkle of special values."""
    out = np.empty((N, K), dtype=np.float32)
    sp = special_values_fp32()
    for r in range(N):
        g = _gen(seed_base + r)
        x = g.standard_normal(K, dtype=np.float32) * np.exp2(g.integers(-30, 30, size=K)).astype(np.float32)
        m = g.random(K) < special_frac
        x[m] = sp[g.integers(0, sp.size, size=int(m.sum()))]
        out[r] = x
    return out


def mixed_bf16(N: int, K: int, seed_base: int = 0, special_frac: float = 0.05) -> np.ndarray:
    return np.stack([to_bf16_bits(row) for row in mixed_fp32(N, K, seed_base, special_frac)]) if N else \
        np.empty((0, K), np.uint16)


# ------------------------------------------------------------------ buckets

LLAMA_HIDDEN = 4096
LLAMA_FFN = 11008


def llama_layer_numels(n_layers: int = 4, hidden: int = LLAMA_HIDDEN, ffn: int = LLAMA_FFN) -> list[int]:
    """Gradient tensor sizes in registration (forward) order, per layer:
    attention norm, q, k, v, o, FFN norm, gate, up, down."""
    per_layer = [hidden, hidden * hidden, hidden * hidden, hidden * hidden, hidden * hidden,
                 hidden, hidden * ffn, hidden * ffn, ffn * hidden]
    return per_layer * n_layers


def bucket_elems(bucket_bytes: int, elem_size: int) -> int:
    return bucket_bytes // elem_size


def bucket_gradients_bf16(N: int, numels: list[int], std: float = 1e-3, seed_base: int = 0):
    """tensors[r][t]: Normal(0, std) bf16 gradients, rank r from seed_base + r,
    tensors drawn in registration order."""
    out = []
    for r in range(N):
        g = _gen(seed_base + r)
        row = []
        for n in numels:
            x = g.standard_normal(n, dtype=np.float32)
            x *= np.float32(std)
            row.append(to_bf16_bits(x))
        out.append(row)
    return out


# ------------------------------------------------------------------ all-to-all

def zipf_expert_counts(N: int = 8, tokens: int = 4096, experts: int = 64, s: float = 1.2,
                       seed_base: int = 1000) -> np.ndarray:
    """counts[i, j] = tokens of rank i routed (top-1) to an expert on rank j.
    Expert e is picked with probability proportional to (e+1)^-s and lives on
    rank e // (experts / N)."""
    assert experts % N == 0
    p = (np.arange(1, experts + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    counts = np.zeros((N, N), dtype=np.int64)
    for i in range(N):
        e = _gen(seed_base + i).choice(experts, size=tokens, p=p)
        counts[i] = np.bincount(e // (experts // N), minlength=N)
    return counts


def random_bits_u16(n: int, seed: int) -> np.ndarray:
    """Arbitrary 16-bit payloads (for copies, where values carry no arithmetic)."""
    return _gen(seed).integers(0, 1 << 16, size=n, dtype=np.uint16)
