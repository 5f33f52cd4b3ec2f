"""Host-side checks of libccl.so that need no GPU: the library loads and exports
every entry point include/ccl.h declares, the planner agrees with the oracle's
tables, and argument validation rejects bad calls before anything is launched
(these calls never reach a kernel, so no device is touched)."""
import ctypes
import os
import re

import numpy as np
import pytest

import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C
from ring_allreduce_rank_gb300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ccl.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ccl_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from ring_allreduce_rank_gb300 import build
    build.build()
    return ccl.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.ccl_version() >= 10000
    for s in range(8):
        assert ccl.ccl_status_string(s)


@pytest.mark.parametrize("K,N", [(0, 1), (5, 3), (16777259, 16), (67108864, 8), (3, 8), (1 << 33, 7)])
def test_planner_partition_matches_oracle(oracle_mod, L, K, N):
    assert ccl.ccl_plan_chunks(K, N) == oracle_mod.partition(K, N)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 16, 64])
def test_planner_schedule_matches_oracle(oracle_mod, L, N):
    tab = np.array(ccl.ccl_plan_ring_schedule(N), dtype=np.int32).reshape(2, max(N - 1, 0), N, 3)
    np.testing.assert_array_equal(tab, oracle_mod.ring_schedule(N))


def test_planner_buckets_c4(L):
    numels = W.llama_layer_numels(4)
    starts = ccl.ccl_plan_buckets(numels, W.bucket_elems(25 * W.MiB, 2))
    assert len(starts) == 63
    sizes = np.diff(starts)
    assert list(sizes[:-1]) == [13_107_200] * 61 and sizes[-1] == 9_994_240


def test_planner_alltoallv_displacements(L):
    counts = W.zipf_expert_counts(8, 4096, 64, 1.2, 1000)
    sd, rd = ccl.ccl_plan_alltoallv(counts.tolist())
    for i in range(8):
        assert sd[i] == [int(counts[i, :j].sum()) for j in range(8)]
    for j in range(8):
        assert rd[j] == [int(counts[:i, j].sum()) for i in range(8)]


def test_zipf_counts_shape():
    counts = W.zipf_expert_counts(8, 4096, 64, 1.2, 1000)
    assert counts.shape == (8, 8) and (counts.sum(axis=1) == 4096).all()
    # experts 0..7 (the most popular) live on rank 0: it receives the most tokens
    assert counts[:, 0].sum() == counts.sum(axis=0).max()


def test_planner_compressed_bytes(L):
    """Blockwise INT8: codes plus one fp32 scale per block, 4b/(b+4) = 3.88
    times fewer bytes than fp32 at b = 128 (Collective Communication,
    blockwise quantization)."""
    d = 128 * 4096
    assert ccl.ccl_plan_compressed_bytes(d, "int8_block", 128) == d + 4 * 4096
    assert round(4 * d / ccl.ccl_plan_compressed_bytes(d, "int8_block", 128), 2) == 3.88
    assert ccl.ccl_plan_compressed_bytes(1001, "int8_block", 64) == 1001 + 4 * 16
    assert ccl.ccl_plan_compressed_bytes(1001, "threshold", 0) == 126


def test_planner_topk_bytes(L):
    """Top-k with fp32 values and int32 indices: 8 bytes per kept element,
    ratio d / (2k) over dense fp32 -- 500x for k = 0.001 d (Collective
    Communication, "Top-k sparsification")."""
    d = 1_000_000
    assert ccl.ccl_plan_topk_bytes(d, d // 1000) == 8000
    assert 4 * d / ccl.ccl_plan_topk_bytes(d, d // 1000) == 500
    assert ccl.ccl_plan_topk_bytes(10, 50) == 80  # k beyond count keeps count
    assert ccl.ccl_plan_topk_bytes(10, 0) == 0
    # per rank: 4096-bin top histograms (u64 exact, u32 sampled), four window
    # low histograms and the fallback's (2^19 u32 bins each), 256 block sums,
    # a 32-byte state record and the threshold
    assert ccl.ccl_plan_topk_work_bytes(8) == 8 * (4096 * 8 + 4096 * 4 + 5 * (1 << 19) * 4 + 256 * 8 + 32 + 4)
    for n in (0, 17):
        with pytest.raises(C.CclError):
            ccl.ccl_plan_topk_work_bytes(n)
    with pytest.raises(C.CclError):
        ccl.ccl_plan_compressed_bytes(1000, "topk", 10)


@pytest.mark.parametrize("count,k,every", [
    (64 << 20, 671_088, 128),      # the bench's Top-k row: 1 % of 64 Mi
    (16 << 20, 167_772, 32), (16 << 20, 300_000, 64), (20 << 20, 600_000, 128),
    ((16 << 20) + 13, 300_000, 64),
    (1 << 20, 10_486, 16),         # too few keys above the k-th for a sparser sample
    (1 << 20, 1 << 19, 16), (16 << 20, 1 << 23, 16),  # the median: the rank band rule keeps 16
    (100, 5, 0),                   # too small for the sample to place a window
    (1000, 0, 0), (1000, 1000, 0), (1000, 5000, 0)])  # tau is known without a select
def test_planner_topk_sample(L, count, k, every):
    """The sample density ccl_allreduce_topk uses: the same cases the GPU
    test checks by counting the keys the sample histogrammed."""
    assert ccl.ccl_plan_topk_sample(count, k) == every


def test_planner_topk_sample_rule(L):
    """Over a grid of sizes: the density is one of 16, 32, 64, 128 (or 0),
    a sparser sample still expects 4096 keys at or above the k-th, and the
    standard deviation of its rank estimate stays within count / 2048."""
    for count in (1 << 16, 1 << 20, 3 << 22, 64 << 20, (1 << 32) - 1):
        for frac in (1e-4, 1e-3, 1e-2, 0.05, 0.3, 0.5, 0.9):
            k = max(1, int(count * frac))
            e = ccl.ccl_plan_topk_sample(count, k)
            assert e in (0, 16, 32, 64, 128), (count, k, e)
            if e > 16:
                assert k // e >= 4096 and k * e <= (count // 2048) ** 2, (count, k, e)
    with pytest.raises(C.CclError):
        ccl.ccl_plan_topk_sample(1 << 32, 10)
    out = ctypes.c_uint32()
    assert L.ccl_plan_topk_sample(1000, 10, None) == 1
    assert L.ccl_plan_topk_sample(1000, 10, ctypes.byref(out)) == 0


def test_arena_layout(L):
    assert ccl.ccl_arena_layout(8, 134217728) == (134217728, 8 * 134217728)
    assert ccl.ccl_arena_layout(3, 1000, 256) == (1024, 3072)
    with pytest.raises(C.CclError):
        ccl.ccl_arena_layout(3, 1000, 100)


@pytest.mark.parametrize("K,N,dt,work", [(64 << 20, 8, "bf16", 192 << 20), (12_345_678, 16, "fp32", 1 << 20),
                                         (100_000, 8, "bf16", 3 * 8 * 256 * 2), (1000, 3, "fp32", 192 << 20),
                                         (3 * 1024 * 1024 + 7, 5, "bf16", 3 * 5 * 4096 * 2 + 100)])
def test_planner_host_slices(L, K, N, dt, work):
    """Slices of the host-buffer AllReduce tile [0, K) in order, fit a stage,
    start on 256-element boundaries, and ramp up (and down) by doubling."""
    es = 2 if dt == "bf16" else 4
    stage = work // (3 * N * es) // 256 * 256
    sl = ccl.ccl_plan_host_slices(K, N, dt, work)
    pos = 0
    for off, ln in sl:
        assert off == pos and 0 < ln <= stage and off % 256 == 0
        pos += ln
    assert pos == K
    lens = [ln for _, ln in sl]
    first = max(256, stage // 16 // 256 * 256)
    if K >= 4 * stage:
        assert lens[0] == first and lens[-1] <= first
        k = 0
        while lens[k] < stage:  # head: doubling up to the stage length
            assert lens[k + 1] == min(2 * lens[k], stage)
            k += 1
        assert max(lens) == stage


def test_planner_host_slices_rejects_small_work(L):
    with pytest.raises(C.CclError):
        ccl.ccl_plan_host_slices(1000, 8, "fp32", 3 * 8 * 256 * 4 - 1)
    assert ccl.ccl_plan_host_slices(0, 8, "fp32", 0) == []


# ------------------------------------------------------------------ validation (no launch)
# The cases live in tests/validation_cases.py and run in a child process that
# sees no GPU (CUDA_VISIBLE_DEVICES=""): their pointers are fake, so a case that
# wrongly passed validation would get "no device" instead of touching memory.

def test_invalid_arguments_and_overlaps_rejected(L):
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    here = os.path.dirname(os.path.abspath(__file__))
    res = subprocess.run([sys.executable, os.path.join(here, "validation_cases.py")], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "validation cases ok" in res.stdout


def test_step_sent_counter_without_a_device(L):
    """The step-mode traffic counter is host state: zero before any step-mode
    launch, and its arguments are validated."""
    assert ccl.ccl_step_sent(8) == [0] * 8
    assert ccl.ccl_step_sent(C.MAX_RANKS, reset=False) == [0] * C.MAX_RANKS
    buf = (ctypes.c_ulonglong * 1)()
    assert L.ccl_step_sent(0, buf, 1) == 1
    assert L.ccl_step_sent(C.MAX_RANKS + 1, buf, 1) == 1
    assert L.ccl_step_sent(4, None, 1) == 1
