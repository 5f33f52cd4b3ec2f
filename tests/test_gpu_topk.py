"""Top-k sparsified AllReduce with error feedback on the device
(ccl_allreduce_topk), bit for bit against the oracle: gradients and residuals
after one or several steps, ties at the k-th magnitude, special values (a NaN
counts as the largest magnitude), unaligned buffers (the element paths), the
degenerate k, CUDA-graph capture, and the argument checks."""
import numpy as np
import pytest
import torch

import oracle
import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C
from ring_allreduce_rank_gb300 import workloads as W

from gpu_util import DEV, assert_bits_equal, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ccl.lib()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _grads(dtype, N, K, seed):
    return list(W.mixed_bf16(N, K, seed_base=seed)) if dtype == "bf16" else list(W.mixed_fp32(N, K, seed_base=seed))


def _res(N, K, seed):
    return [W.normal_fp32(1, K, std=1e-3, seed_base=seed + r)[0] for r in range(N)]


def _run(g_host, e_host, k, op, pad=0):
    g = [to_dev(x, pad_elems=pad) for x in g_host]
    e = [to_dev(x, pad_elems=pad) for x in e_host]
    ccl.ccl_allreduce_topk(g, e, k, op=op)
    torch.cuda.synchronize()
    return [bits(x) for x in g], [bits(x) for x in e]


def _check(got_g, got_e, want_g, want_e, what):
    for r in range(len(got_g)):
        assert_bits_equal(got_g[r], want_g[r], "%s grads rank %d" % (what, r))
        assert_bits_equal(got_e[r], np.asarray(want_e[r]).view(np.uint32), "%s residual rank %d" % (what, r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("N,K,k", [(1, 1000, 7), (3, 10_007, 100), (8, 65_536 + 13, 655), (16, 40_001, 1),
                                   (5, 4, 2), (4, 5000, 0), (4, 5000, 5000), (4, 5000, 6000), (2, 300_001, 299_999),
                                   (8, 1 << 20, 10_486)])
def test_matches_oracle(dtype, op, N, K, k):
    g = _grads(dtype, N, K, seed=N * 100 + K % 89)
    e = _res(N, K, seed=K % 1000)
    want_g, want_e = oracle.allreduce_compressed(g, e, op, "topk", k=k)
    got_g, got_e = _run(g, e, k, op)
    _check(got_g, got_e, want_g, want_e, "topk %s %s N=%d K=%d k=%d" % (dtype, op, N, K, k))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("k", [1, 50, 333, 1000, 3999])
def test_ties_at_the_kth_magnitude(dtype, k):
    """Integers in [-6, 6] with zero residuals: thousands of equal magnitudes,
    so the k-th falls inside a tie group and every tied value is sent."""
    N, K = 4, 4000
    x = W.integers_fp32(N, K, seed=k, lo=-6, hi=6)
    g = [W.to_bf16_bits(r) for r in x] if dtype == "bf16" else list(x)
    e = [np.zeros(K, np.float32) for _ in range(N)]
    want_g, want_e = oracle.allreduce_compressed(g, e, "sum", "topk", k=k)
    got_g, got_e = _run(g, e, k, "sum")
    _check(got_g, got_e, want_g, want_e, "ties k=%d" % k)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_three_steps_carry_the_residual(dtype):
    N, K, k = 6, 50_003, 500
    e_host = [np.zeros(K, np.float32) for _ in range(N)]
    e_dev = [to_dev(x) for x in e_host]
    for step in range(3):
        g = _grads(dtype, N, K, seed=1000 * step + 1)
        gd = [to_dev(x) for x in g]
        ccl.ccl_allreduce_topk(gd, e_dev, k, op="avg")
        want_g, e_host = oracle.allreduce_compressed(g, e_host, "avg", "topk", k=k)
        torch.cuda.synchronize()
        _check([bits(x) for x in gd], [bits(x) for x in e_dev], want_g, e_host, "step %d" % step)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("pad", [1, 3])
def test_unaligned_buffers(dtype, pad):
    N, K, k = 3, 20_011, 77
    g = _grads(dtype, N, K, seed=pad)
    e = _res(N, K, seed=pad + 50)
    want_g, want_e = oracle.allreduce_compressed(g, e, "sum", "topk", k=k)
    got_g, got_e = _run(g, e, k, "sum", pad=pad)
    _check(got_g, got_e, want_g, want_e, "unaligned pad %d" % pad)


def _window_record(work, N):
    """The select's per-rank record in the work buffer (the layout of
    topk.cu: top u64[N][4096], sample u32[N][4096], low u32[N][5][2^19],
    block sums u64[N][256], then one 32-byte record per rank whose 5th word
    is the window's first top digit (all ones when the sample placed none)
    and whose 7th says whether the window held the k-th key's top digit).
    Returns (hit, window placed) per rank."""
    off = N * (4096 * 8 + 4096 * 4 + 5 * (1 << 19) * 4 + 256 * 8)
    rec = work[off:off + 32 * N].cpu().numpy().view(np.uint32).reshape(N, 8)
    return rec[:, 6].tolist(), [int(w != 0xFFFFFFFF) for w in rec[:, 4].tolist()]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_sampled_window_hit_miss_and_none(dtype):
    """Every way through the select gives the oracle's bits.
    - Normal data: the sample (one run in 16 at this k) places a window of top digits around the
      k-th key's (one full pass; hit).
    - Zero residuals and sampled runs (the first 256 elements of every 4096)
      that all hold +-1e-6: the sample puts the window on that one digit, far
      below the k-th key; the fallback pass counts the right digit (miss).
    - Sampled runs whose values spread over many binades: the sample's bounds
      fall more than one digit apart, no window is placed, and the fallback
      pass counts the k-th key's digit."""
    N, K, k = 4, 1 << 20, 10_486
    base = _grads(dtype, N, K, seed=123)
    idx = np.arange(K)
    sampled = (idx // 256) % 16 == 0
    g = np.random.Generator(np.random.PCG64(77))

    def rig(fill):
        out = []
        for r in range(N):
            x = (W.bf16_bits_to_f32(base[r]) if dtype == "bf16" else base[r]).copy()
            x[sampled] = fill(int(sampled.sum()))
            out.append(W.to_bf16_bits(x) if dtype == "bf16" else x.astype(np.float32))
        return out

    normal = list(W.normal_bf16(N, K, seed_base=5)) if dtype == "bf16" else list(W.normal_fp32(N, K, seed_base=5))
    tiny = rig(lambda n: np.where(g.random(n) < 0.5, -1e-6, 1e-6).astype(np.float32))
    spread = rig(lambda n: (np.exp2(g.uniform(-60, 60, n)) * np.where(g.random(n) < 0.5, -1, 1)).astype(np.float32))
    zeros = [np.zeros(K, np.float32) for _ in range(N)]
    work = torch.empty(ccl.ccl_plan_topk_work_bytes(N), dtype=torch.uint8, device=DEV)
    for name, data, e, want_rec in (("hit", normal, _res(N, K, seed=9), (1, 1)), ("miss", tiny, zeros, (0, 1)),
                                    ("no window", spread, zeros, (0, 0))):
        want_g, want_e = oracle.allreduce_compressed(data, e, "avg", "topk", k=k)
        gd = [to_dev(x) for x in data]
        ed = [to_dev(x) for x in e]
        ccl.ccl_allreduce_topk(gd, ed, k, op="avg", work=work)
        torch.cuda.synchronize()
        hit, placed = _window_record(work, N)
        assert (hit, placed) == ([want_rec[0]] * N, [want_rec[1]] * N), name
        _check([bits(x) for x in gd], [bits(x) for x in ed], want_g, want_e, name)


def _sampled_keys(work, N):
    """Keys the sample counted, per rank: the sums of its 4096-bin histograms
    (u32[N][4096] after the exact u64[N][4096] ones in the work buffer)."""
    h = work[N * 4096 * 8:N * 4096 * 12].cpu().numpy().view(np.uint32).reshape(N, 4096)
    return h.sum(axis=1, dtype=np.int64).tolist()


@pytest.mark.parametrize("dtype,K,k,every", [("fp32", 16 << 20, 167_772, 32), ("bf16", 16 << 20, 300_000, 64),
                                             ("fp32", 20 << 20, 600_000, 128), ("bf16", 20 << 20, 600_000, 128),
                                             ("bf16", 1 << 20, 1 << 19, 16), ("fp32", 16 << 20, 1 << 23, 16),
                                             ("bf16", (16 << 20) + 13, 300_000, 64)])
def test_sample_density(dtype, K, k, every):
    """The sample takes one 256-element run in 16, or in 32, 64 or 128 when the
    sparser sample still expects 4096 keys at or above the k-th and
    sqrt(k * every) <= K / 2048.  k = 1 % of 16 Mi allows 32; 300,000 allows 64
    and 600,000 of 20 Mi 128; half of 1 Mi or of 16 Mi (the median, where a
    band of ranks spans many digits) keeps 16.  Each time the sample counts
    exactly its runs' keys, its window holds the k-th key's digit, and the
    result is the oracle's.  The ragged size ends in a run of one group of 8
    elements (sampled: 65,536 is a multiple of 64) and 5 elements outside any
    group (never sampled)."""
    N = 2
    assert ccl.ccl_plan_topk_sample(K, k) == every
    g = list(W.normal_bf16(N, K, seed_base=k % 101)) if dtype == "bf16" else list(W.normal_fp32(N, K, seed_base=k % 101))
    e = _res(N, K, seed=k % 103)
    want_g, want_e = oracle.allreduce_compressed(g, e, "avg", "topk", k=k)
    gd = [to_dev(x) for x in g]
    ed = [to_dev(x) for x in e]
    work = torch.empty(ccl.ccl_plan_topk_work_bytes(N), dtype=torch.uint8, device=DEV)
    ccl.ccl_allreduce_topk(gd, ed, k, op="avg", work=work)
    torch.cuda.synchronize()
    groups = K // 8                   # whole groups of 8 elements
    runs = (groups + 31) // 32        # runs of 32 groups, the last maybe partial
    sampled = sum(min(32, groups - 32 * q) for q in range(0, runs, every))
    assert _sampled_keys(work, N) == [8 * sampled] * N
    assert _window_record(work, N) == ([1] * N, [1] * N)
    _check([bits(x) for x in gd], [bits(x) for x in ed], want_g, want_e, "K=%d k=%d" % (K, k))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_window_widths(dtype):
    """The sample's window covers the top digits between its two bounds, one
    to four of them: narrow where the sample pins the k-th key down (many
    elements), wider where it cannot (few).  Every width gives the oracle's
    bits, and the sizes below produce windows of one or two digits and of
    three or four."""
    N = 4
    widths = set()
    work = torch.empty(ccl.ccl_plan_topk_work_bytes(N), dtype=torch.uint8, device=DEV)
    off = N * (4096 * 8 + 4096 * 4 + 5 * (1 << 19) * 4 + 256 * 8)
    for K, k in ((1 << 20, 10_486), (1 << 18, 2_621), (65_536 + 13, 655), (40_000, 400), (30_000, 1_500)):
        g = list(W.normal_bf16(N, K, seed_base=K % 97)) if dtype == "bf16" else list(W.normal_fp32(N, K, seed_base=K % 97))
        e = _res(N, K, seed=K % 89)
        want_g, want_e = oracle.allreduce_compressed(g, e, "avg", "topk", k=k)
        gd = [to_dev(x) for x in g]
        ed = [to_dev(x) for x in e]
        ccl.ccl_allreduce_topk(gd, ed, k, op="avg", work=work)
        torch.cuda.synchronize()
        rec = work[off:off + 32 * N].cpu().numpy().view(np.uint32).reshape(N, 8)
        widths.update(int(w) for w in rec[:, 7])
        _check([bits(x) for x in gd], [bits(x) for x in ed], want_g, want_e, "K=%d k=%d" % (K, k))
    assert widths & {1, 2} and widths & {3, 4}, widths


def test_nan_is_sent_first():
    N, K = 3, 4096
    g = list(W.normal_fp32(N, K, seed_base=8))
    g[2][100] = np.float32("nan")
    e = [np.zeros(K, np.float32) for _ in range(N)]
    want_g, want_e = oracle.allreduce_compressed(g, e, "sum", "topk", k=1)
    got_g, got_e = _run(g, e, 1, "sum")
    _check(got_g, got_e, want_g, want_e, "nan")
    assert got_g[0][100] == 0x7FFFFFFF


def test_graph_capture_and_replay():
    """The whole call -- work reset, selection passes, compressed pass -- is
    device-only work: captured once, replayed twice, it equals two oracle
    steps (the residual carries from the first replay into the second)."""
    N, K, k = 4, 100_000, 1000
    x = _grads("bf16", N, K, seed=77)
    g = [to_dev(r) for r in x]
    e = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    work = torch.empty(ccl.ccl_plan_topk_work_bytes(N), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        gr.capture_begin()
        ccl.ccl_allreduce_topk(g, e, k, op="sum", work=work, stream=s)
        gr.capture_end()
    torch.cuda.synchronize()
    want_g, want_e = list(x), [np.zeros(K, np.float32) for _ in range(N)]
    for step in range(2):
        for r in range(N):
            g[r].copy_(to_dev(x[r]))
        gr.replay()
        torch.cuda.synchronize()
        want_g, want_e = oracle.allreduce_compressed(list(x), want_e, "sum", "topk", k=k)
        _check([bits(t) for t in g], [bits(t) for t in e], want_g, want_e, "graph replay %d" % step)


def test_argument_errors():
    N, K = 4, 1000
    g = [torch.zeros(K, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    e = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(N)]
    wb = ccl.ccl_plan_topk_work_bytes(N)
    work = torch.empty(wb + 64, dtype=torch.uint8, device=DEV)

    def status(fn):
        with pytest.raises(C.CclError) as ei:
            fn()
        return ei.value.status

    assert status(lambda: ccl.ccl_allreduce_topk(g, e, 10, op="avg_premul", work=work)) == 2  # unsupported
    assert status(lambda: ccl.ccl_allreduce_topk(g, e, 10, op="max", work=work)) == 1
    assert status(lambda: ccl.ccl_allreduce_topk(g, e, 10, work=work[:wb - 1])) == 1  # too small
    assert status(lambda: ccl.ccl_allreduce_topk(g, e, 10, work=work[1:])) == 1  # not 16-byte aligned
    big = [torch.zeros(K, dtype=torch.bfloat16, device=DEV) for _ in range(17)]
    bige = [torch.zeros(K, dtype=torch.float32, device=DEV) for _ in range(17)]
    assert status(lambda: ccl.ccl_allreduce_topk(big, bige, 10)) == 1  # more than 16 ranks
    # the work buffer inside a residual
    K2 = wb // 4 + 16  # a residual large enough to hold the whole work buffer
    g2 = [torch.zeros(K2, dtype=torch.bfloat16, device=DEV) for _ in range(N)]
    e2 = [torch.zeros(K2, dtype=torch.float32, device=DEV) for _ in range(N)]
    assert status(lambda: ccl.ccl_allreduce_topk(g2, e2, 10, work=e2[1].view(torch.uint8)[:wb])) == 3
    assert status(lambda: ccl.ccl_allreduce_compressed(g, e, comp="topk")) == 1
    ccl.ccl_allreduce_topk([t[:0] for t in g], [t[:0] for t in e], 10, work=work)  # count 0: nothing to do
    torch.cuda.synchronize()
