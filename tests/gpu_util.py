"""Helpers for the GPU parity tests: move seeded host inputs to the device and
bring results back as raw bits for exact comparison with the oracle."""
import numpy as np
import torch

DEV = "cuda:0"


def torch_dtype(rows) -> torch.dtype:
    a = rows[0] if isinstance(rows, (list, tuple)) else rows
    return torch.bfloat16 if np.asarray(a).dtype == np.uint16 else torch.float32


def to_dev(row: np.ndarray, dtype: torch.dtype = None, pad_elems: int = 0) -> torch.Tensor:
    """Host row (float32, or uint16 bf16 bits) -> device tensor of the same bits.
    pad_elems > 0 returns a view that starts pad_elems elements into a larger
    allocation (an unaligned buffer)."""
    row = np.ascontiguousarray(row)
    if row.dtype == np.uint16:
        t = torch.from_numpy(row.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(row.astype(np.float32, copy=False))
    if pad_elems:
        big = torch.empty(row.size + pad_elems, dtype=t.dtype, device=DEV)
        v = big[pad_elems:]
        v.copy_(t)
        return v
    return t.to(DEV)


def empty_like_host(n: int, dtype: torch.dtype, pad_elems: int = 0, fill_bits: int = 0x5a5a) -> torch.Tensor:
    big = torch.empty(n + pad_elems, dtype=dtype, device=DEV)
    if dtype == torch.bfloat16:
        big.view(torch.int16).fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
    else:
        big.view(torch.int32).fill_(int(np.uint32((fill_bits << 16) | fill_bits).view(np.int32)))
    return big[pad_elems:]


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def host_bits(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    got, want = host_bits(got), host_bits(want)
    if got.shape != want.shape:
        raise AssertionError("%s: shape %s vs %s" % (what, got.shape, want.shape))
    bad = np.nonzero(got != want)[0]
    if bad.size:
        i = bad[0]
        raise AssertionError("%s: %d of %d elements differ; first at %d: got 0x%x want 0x%x"
                             % (what, bad.size, got.size, i, int(got[i]), int(want[i])))
