"""Rank-buffer arena: N simulated ranks' buffers in one device allocation.

One ``torch.empty`` of ``nranks * stride`` bytes holds every rank; rank r's
buffer starts at ``r * stride`` (``stride`` = buffer bytes plus an optional
guard band, rounded up to ``align``, from ``ccl_arena_layout``), so every rank
buffer is at least 256-byte aligned and the collectives take their 16-byte
vector paths.  The guard band after each buffer is filled with a poison byte
and can be checked after a call: a kernel that wrote past a rank's end would
show up there.
"""
from __future__ import annotations

import torch

from .ccl import ccl_arena_layout

POISON = 0xA5


class RankArena:
    def __init__(self, nranks: int, count: int, dtype: torch.dtype, device="cuda", align: int = 256,
                 guard_bytes: int = 0):
        self.nranks, self.count, self.dtype = nranks, count, dtype
        self.elem_size = torch.empty((), dtype=dtype).element_size()
        self.nbytes = count * self.elem_size
        self.guard_bytes = guard_bytes
        self.stride, self.total = ccl_arena_layout(nranks, self.nbytes + guard_bytes, align)
        self.storage = torch.empty(self.total, dtype=torch.uint8, device=device)
        self.ranks = [self.storage[r * self.stride:r * self.stride + self.nbytes].view(dtype)
                      for r in range(nranks)]
        if guard_bytes:
            for r in range(nranks):
                self.guard(r).fill_(POISON)

    def guard(self, r: int) -> torch.Tensor:
        return self.storage[r * self.stride + self.nbytes:(r + 1) * self.stride]

    def guards_intact(self) -> bool:
        return all(bool((self.guard(r) == POISON).all()) for r in range(self.nranks))

    def first_damage(self):
        """(rank, byte offset into that rank's guard band) of the first guard
        byte that no longer holds the poison value, or None."""
        for r in range(self.nranks):
            bad = torch.nonzero(self.guard(r) != POISON)
            if bad.numel():
                return r, int(bad[0, 0])
        return None

    def load(self, host_rows) -> None:
        """Copy host rows (one per rank; numpy or torch, matching bytes) into the arena."""
        for r in range(self.nranks):
            src = host_rows[r]
            if not isinstance(src, torch.Tensor):
                src = torch.from_numpy(src)
            self.ranks[r].view(torch.uint8).copy_(src.contiguous().view(torch.uint8).reshape(-1))

    def rows_bits(self):
        """Every rank's buffer as raw bits on the host (uint16 for bf16, uint32 for fp32)."""
        it = torch.int16 if self.elem_size == 2 else torch.int32
        return [t.view(it).cpu().numpy() for t in self.ranks]
