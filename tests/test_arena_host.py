"""The rank arena on the host: layout (every rank buffer aligned, strides that
hold the buffer and its guard band, ranks disjoint) and the guard bands that
catch a write past a rank's end.  The arena is plain torch memory plus the
library's host-only layout planner, so this runs on the CPU; a mistake is
planted by writing one element past a rank's end, as an out-of-bounds kernel
store would."""
import numpy as np
import pytest
import torch

from ring_allreduce_rank_gb300 import workloads as W
from ring_allreduce_rank_gb300.arena import POISON, RankArena


@pytest.fixture(scope="module", autouse=True)
def _built():
    from ring_allreduce_rank_gb300 import build
    build.build()


@pytest.mark.parametrize("N,K,dtype,guard", [(8, 1000, torch.bfloat16, 256), (3, 7, torch.float32, 64),
                                             (16, 4099, torch.float32, 1), (1, 0, torch.bfloat16, 16)])
def test_layout(N, K, dtype, guard):
    a = RankArena(N, K, dtype, device="cpu", guard_bytes=guard)
    es = a.elem_size
    assert a.stride % 256 == 0 and a.stride >= K * es + guard and a.total == N * a.stride
    base = a.storage.data_ptr()
    for r in range(N):
        assert a.ranks[r].numel() == K
        if K:  # torch gives an empty view a null data pointer
            assert a.ranks[r].data_ptr() == base + r * a.stride
        assert a.guard(r).numel() == a.stride - K * es >= guard
    assert a.guards_intact() and a.first_damage() is None


def test_in_bounds_writes_keep_the_guards():
    N, K = 5, 1003
    a = RankArena(N, K, torch.float32, device="cpu", guard_bytes=256)
    x = W.uniform_fp32(N, K, seed_base=1)
    a.load(x)
    for r in range(N):
        a.ranks[r].fill_(float("nan"))  # every byte of every rank written
    assert a.guards_intact()
    a.load(x)
    got = a.rows_bits()
    for r in range(N):
        np.testing.assert_array_equal(got[r], x[r].view(np.int32))


@pytest.mark.parametrize("r", [0, 2, 4])
def test_one_element_past_a_rank_is_caught(r):
    N, K = 5, 1003
    a = RankArena(N, K, torch.bfloat16, device="cpu", guard_bytes=256)
    end = r * a.stride + K * a.elem_size
    a.storage[end:end + a.elem_size] = 0  # the store one element past rank r's end
    assert not a.guards_intact()
    assert a.first_damage() == (r, 0)
    a.storage[end:end + a.elem_size] = POISON
    assert a.guards_intact()


def test_damage_deep_in_a_guard_is_located():
    a = RankArena(4, 100, torch.float32, device="cpu", guard_bytes=512)
    g = a.guard(3)
    g[g.numel() - 1] = 0  # the last guard byte of the last rank
    assert a.first_damage() == (3, g.numel() - 1)
