"""The library's host planners over many seeded random shapes (no GPU): the
chunk partition and the ring schedule against the oracle's own, and the bucket,
AllToAllv and host-slice plans against the definitions their callers rely on."""
import numpy as np
import pytest

import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C

RNG_SEED = 20261202


@pytest.fixture(scope="module", autouse=True)
def _built():
    from ring_allreduce_rank_gb300 import build
    build.build()
    ccl.lib()


def _random_counts(g, n):
    """A mix of empty, tiny, fewer-than-ranks, ordinary and very large counts."""
    kind = g.integers(0, 5, size=n)
    K = np.where(kind == 0, 0,
        np.where(kind == 1, g.integers(1, 8, size=n),
        np.where(kind == 2, g.integers(1, 2000, size=n),
        np.where(kind == 3, g.integers(1, 1 << 28, size=n, dtype=np.int64),
                 g.integers(1 << 31, 1 << 41, size=n, dtype=np.int64)))))
    return [int(k) for k in K]


def test_partition_matches_the_oracle(oracle_mod):
    g = np.random.default_rng(RNG_SEED)
    Ks = _random_counts(g, 600)
    Ns = [int(n) for n in g.integers(1, C.MAX_RANKS + 1, size=600)]
    for K, N in zip(Ks, Ns):
        off, ln = ccl.ccl_plan_chunks(K, N)
        assert (off, ln) == oracle_mod.partition(K, N), (K, N)
        assert sum(ln) == K and max(ln) - min(ln) <= 1


def test_ring_schedule_matches_the_oracle_for_every_small_rank_count(oracle_mod):
    for N in range(1, 81):
        tab = np.array(ccl.ccl_plan_ring_schedule(N), dtype=np.int32).reshape(2, max(N - 1, 0), N, 3)
        np.testing.assert_array_equal(tab, oracle_mod.ring_schedule(N), err_msg="N=%d" % N)


def test_bucket_plan_cuts_the_reversed_stream_into_fixed_buckets():
    g = np.random.default_rng(RNG_SEED + 1)
    for _ in range(300):
        T = int(g.integers(1, 60))
        numels = [int(v) for v in np.where(g.random(T) < 0.1, 0, g.integers(1, 1 << 20, size=T))]
        total = sum(numels)
        B = int(g.choice([1, 7, 4096, 1 << 16, 13_107_200, int(g.integers(1, 1 << 22))]))
        B = max(B, -(-total // 4000))  # at most a few thousand buckets per plan
        starts = ccl.ccl_plan_buckets(numels, B)
        assert starts[0] == 0 and starts[-1] == total
        sizes = np.diff(starts)
        if total == 0:
            assert len(sizes) == 0
            continue
        assert len(sizes) == -(-total // B)
        assert (sizes[:-1] == B).all() and 0 < sizes[-1] <= B


def test_alltoallv_displacements_are_the_prefix_sums():
    g = np.random.default_rng(RNG_SEED + 2)
    for _ in range(200):
        N = int(g.integers(1, 33))
        counts = g.integers(0, 1 << 20, size=(N, N))
        counts[g.random((N, N)) < 0.2] = 0
        sd, rd = ccl.ccl_plan_alltoallv(counts.tolist())
        for i in range(N):
            # send[i]: blocks ordered by destination
            assert sd[i] == [int(counts[i, :j].sum()) for j in range(N)]
        for j in range(N):
            # recv[j]: blocks ordered by source
            assert rd[j] == [int(counts[:i, j].sum()) for i in range(N)]


def test_host_slices_tile_the_vector_within_a_stage():
    g = np.random.default_rng(RNG_SEED + 3)
    for _ in range(300):
        N = int(g.integers(1, 65))
        dt = str(g.choice(["bf16", "fp32"]))
        es = 2 if dt == "bf16" else 4
        min_work = 3 * N * 256 * es
        work = int(g.choice([min_work, min_work + int(g.integers(0, 1 << 20)), 192 << 20,
                             int(g.integers(min_work, 1 << 28))]))
        K = int(g.choice([0, int(g.integers(1, 300)), int(g.integers(1, 1 << 24)), int(g.integers(1, 1 << 30))]))
        stage = work // (3 * N * es) // 256 * 256
        K = min(K, 4000 * stage)  # at most a few thousand slices per plan
        sl = ccl.ccl_plan_host_slices(K, N, dt, work)
        pos = 0
        for off, ln in sl:
            assert off == pos and 0 < ln <= stage and off % 256 == 0, (K, N, dt, work)
            pos += ln
        assert pos == K
