"""Benchmark: fused ring-order AllReduce, N=8 simulated ranks, bf16, AVG,
64Mi elements (128 MiB) per rank, in place, on one GB300.

One step = one ccl_allreduce call over the whole arena (the ReduceScatter
phase, the AVG scaling and the AllGather phase, computed in one launch).
Metric: algorithmic HBM bytes (N*M read + N*M written = 2 GiB per step) per
second.  Inputs (1 GiB read per step) are larger than the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--gpus N > 1 runs N independent replicas (one per GPU, launched by
torch.distributed.run): the path has no cross-GPU exchange.  --impl reference
times the CPU oracle on the host cores on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AllReduce HBM GB/s & % of peak, N=8 bf16 128 MB/rank, 1 GB300"
UNIT = "GB/s"
NRANKS = 8
COUNT = 64 * 1024 * 1024  # bf16 elements per rank (128 MiB)
DEFAULT_COUNT = COUNT
ELEM = 2
ALG_BYTES = 2 * NRANKS * COUNT * ELEM  # N*M read + N*M written
HOST_WORK_BYTES = 192 * 1024 * 1024  # device stages of the end-to-end (host-buffer) leg
WORKLOAD = "allreduce-avg N=8 bf16 64Mi elements/rank (128 MiB), in place, fused ring order"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_allreduce_bf16_n8_128mib.traffic")
KERNEL_SOURCES = ["ring_allreduce_rank_gb300/csrc/reduce.cu", "ring_allreduce_rank_gb300/csrc/ccl_device.cuh",
                  "ring_allreduce_rank_gb300/csrc/fused.h"]


def set_count(count: int) -> None:
    global COUNT, ALG_BYTES, WORKLOAD
    COUNT = count
    ALG_BYTES = 2 * NRANKS * COUNT * ELEM
    WORKLOAD = "allreduce-avg N=8 bf16 %d elements/rank (profiling size), in place, fused ring order" % count


def kernel_digest() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style torch copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


SPEC_HBM_GBS = 8000.0  # NVIDIA's GB300 HBM3e figure (vendor spec, not a measurement)


def recorded_ncu():
    """DRAM bytes per launch and ncu's DRAM throughput (% of its own peak) from
    the committed full-size ncu capture, if it was taken on the current kernel
    sources; else (None, None)."""
    try:
        kv = dict(line.split("=", 1) for line in open(TRAFFIC_FILE).read().split() if "=" in line)
        if kv.get("kernel_digest") != kernel_digest():
            return None, None
        pct = kv.get("gpu_dram_throughput_pct")
        return int(kv["dram_bytes_per_launch"]), (float(pct) if pct else None)
    except Exception:
        return None, None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = [l.split(",") for l in open(self.file.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ multi-replica timing

def max_over_ranks(dist, ms: float, device) -> float:
    """The slowest replica's time (the job finishes when the last one does)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: bytes every replica moved over the slowest replica's time."""
    return world * bytes_per_step * steps / (ms / 1e3) / 1e9


# ------------------------------------------------------------------ oracle timing (CPU)

def oracle_sample_gbs(target_s: float, max_count: int = COUNT, threads: int = 1):
    """Time the CPU oracle (step-by-step ring simulation) on a sample of the
    workload: N=8 ranks, the first k elements of each rank's buffer, k sized
    from a short probe to take about target_s seconds.  threads = 1: the
    one-thread simulation; more: the ranks spread over that many threads with
    a barrier per step (the same bits).  Returns (GB/s, seconds, k)."""
    import oracle
    from ring_allreduce_rank_gb300 import workloads as W

    oracle.build()

    def run(x):
        if threads > 1:
            oracle.ring_allreduce_threads(x, "avg", threads)
        else:
            oracle.ring_allreduce(x, "avg")

    k = min(1 << 18, max_count)
    x = list(W.normal_bf16(NRANKS, k, std=1e-3, seed_base=0))
    t0 = time.perf_counter()
    run(x)
    dt = time.perf_counter() - t0
    k = int(min(max_count, max(1 << 12, k * target_s / max(dt, 1e-4)))) // 8 * 8
    x = list(W.normal_bf16(NRANKS, k, std=1e-3, seed_base=0))
    t0 = time.perf_counter()
    run(x)
    dt = time.perf_counter() - t0
    return 2 * NRANKS * k * ELEM / dt / 1e9, dt, k


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


# ------------------------------------------------------------------ the other collectives' workloads

ROWS = {
    "allreduce-step": "AllReduce AVG, N=8 bf16 64Mi/rank, in place, step mode (2(N-1) launches + 1 AVG scale)",
    "reduce-scatter": "ReduceScatter SUM, N=16 fp32, 16,777,259 elements/rank (ragged chunks)",
    "allgather": "AllGather, N=16 fp32, 16,777,259 elements total (ragged chunks)",
    "broadcast": "Broadcast from rank 0, N=8 bf16 64Mi elements, in place",
    "alltoallv": "AllToAllv MoE dispatch, N=8, 4096 tokens x 7168 bf16/rank, Zipf(1.2) top-1 over 64 experts",
    "bucket": "bucket-fused AllReduce SUM, N=8 bf16, 4 Llama layers (809,533,440 elements/rank), 25 MiB buckets",
    "allreduce-hd": "AllReduce AVG in halving-doubling order, N=8 bf16 64Mi/rank, in place, one pass",
    "allreduce-tree": "AllReduce AVG in binomial-tree order, N=8 bf16 64Mi/rank, in place, one pass",
    "allreduce-hier": "AllReduce AVG in two-level hierarchical order (2 groups of 4), N=8 bf16 64Mi/rank, in place",
    "allreduce-premul": "AllReduce AVG by pre-multiplication (each contribution times 1/N, then SUM), N=8 bf16 "
                        "64Mi/rank, in place, fused ring order",
    "allreduce-topk": "Top-k sparsified AllReduce AVG with error feedback, k = 1% of each rank's 64Mi bf16 "
                      "elements (671,088), N=8; threshold by on-device radix select",
    "allreduce-int8": "compressed AllReduce AVG with error feedback, blockwise INT8 (b=128), N=8 bf16 64Mi/rank",
    "overlap": "bucket AllReduce (4 Llama layers, N=8 bf16, 25 MiB buckets) overlapped with a synthetic backward "
               "pass of per-rank gradient GEMMs (4096 tokens); bucket kernels on a second stream as gradients finish",
    "reduce": "Reduce SUM to rank 0, N=8 bf16 64Mi elements/rank, out of place",
    "gather": "Gather to rank 0, N=8 bf16, 64Mi elements total (8 slices of 8Mi; --count sets the total)",
    "scatter": "Scatter from rank 0, N=8 bf16, 64Mi elements total (8 slices of 8Mi; --count sets the total)",
    "sweep": "AllReduce SUM bf16, 1 KiB..1 GiB per rank (x4), N in {2,4,8,16,64}; device time per call from "
             "CUDA-graph replay; points whose N*S fits in L2 are marked l2_resident (replays hit L2, not HBM)",
}


def _timed(torch, ccl, step, steps, warmup, stream, dev):
    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = ccl.ccl_launch_count()
    t0.record(stream)
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    per = [a.elapsed_time(b) for a, b in ev]
    # whole-run time of the back-to-back steps (the line's value), and each
    # launch's own duration (the roofline's achieved bandwidth)
    return t0.elapsed_time(t1), per, ccl.ccl_launch_count() - n0


def graph_call_seconds(torch, ccl, call, nbytes, dev) -> float:
    """Device time per call: R calls captured once in a CUDA graph and
    replayed, so the host's per-call cost (Python, argument checks, launch)
    is not in the measurement.  R (at most 20) keeps each replay short."""
    R = int(max(1, min(20, 2e10 / max(nbytes, 1) / 1e3)))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            call(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream(dev)
        for _ in range(R):
            call(st)
    g.replay()
    torch.cuda.synchronize(dev)
    reps = 5
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize(dev)
    del g
    return a.elapsed_time(b) / 1e3 / (R * reps)


def run_row(args, name, local):
    """One of the other collectives' workloads, printed as its own JSON line.
    Inputs come from a seeded torch generator on the device (values do not
    change the timing; parity at these sizes is covered by the GPU tests)."""
    import torch

    import ring_allreduce_rank_gb300 as ccl
    from ring_allreduce_rank_gb300 import workloads as W
    from ring_allreduce_rank_gb300.arena import RankArena

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ccl.lib()
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    peak, peak_src = measured_peak()
    clocks = ClockSampler(local)

    def randn_bf16(n):
        return (torch.randn(n, generator=g, device=dev) * 1e-3).to(torch.bfloat16)

    def line(metric, alg, per_ms, launches, kernel, dtype, config, extra=None, total_ms=None):
        """value: whole-run throughput (total_ms over the back-to-back steps,
        else the sum of the per-launch times); roofline.achieved: algorithmic
        bytes over the average per-launch time."""
        tot = total_ms if total_ms is not None else sum(per_ms)
        val = alg * len(per_ms) / (tot / 1e3) / 1e9
        ach = alg * len(per_ms) / (sum(per_ms) / 1e3) / 1e9
        d = {"metric": metric, "value": round(val, 2), "unit": UNIT, "n_gpus": 1, "steps": len(per_ms),
             "warmup": max(args.warmup, 3), "ms_per_step": round(tot / len(per_ms), 5), "higher_is_better": True,
             "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
             "config": dict(config, workload=ROWS[name]),
             "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(ach / peak, 4), "traffic": None, "algorithmic_bytes_per_step": alg,
                          "peak_source": peak_src, "kernel": kernel,
                          "achieved_median": round(alg / (statistics.median(per_ms) / 1e3) / 1e9, 1)},
             "cpu_baseline": None, "e2e": None, "gpu_launches": int(launches)}
        if extra:
            d.update(extra)
        return d

    if name == "sweep":
        points = []
        for N in (2, 4, 8, 16, 64):
            for S in [1 << k for k in range(10, 31, 2)]:
                K = S // 2
                arena = RankArena(N, K, torch.bfloat16, device=dev)
                for r in range(N):
                    arena.ranks[r].copy_(randn_bf16(K))
                t = graph_call_seconds(torch, ccl, lambda st: ccl.ccl_allreduce(arena.ranks, op="sum", stream=st),
                                       S * N, dev)
                alg = 2 * N * S
                points.append({"N": N, "bytes_per_rank": S, "us": round(t * 1e6, 3),
                               "l2_resident": N * S <= 96 * 1024 * 1024,
                               "GBs": round(alg / t / 1e9, 2), "frac": round(alg / t / 1e9 / peak, 4),
                               "algbw_GBs": round(S / t / 1e9, 3), "busbw_GBs": round(S / t / 1e9 * 2 * (N - 1) / N, 3)})
                del arena
                torch.cuda.empty_cache()
        # the line's value: N=8 at 1 GiB per rank (HBM-bound); every point is listed
        big = [p for p in points if p["N"] == 8 and p["bytes_per_rank"] == 1 << 30][0]
        d = line("AllReduce sweep HBM GB/s, bf16, 1 KiB..1 GiB per rank, N in {2,4,8,16,64}, 1 GB300", 2 * big["N"] *
                 big["bytes_per_rank"], [big["us"] / 1e3], 1, "fused_reduce_kernel<bf16, SUM, N>", "bf16",
                 {"op": "sum", "mode": "fused"}, {"points": points})
        print(json.dumps(d))
        return

    if name in ("allreduce-hd", "allreduce-tree", "allreduce-hier"):
        N, K = 8, 64 * 1024 * 1024
        arena = RankArena(N, K, torch.bfloat16, device=dev)
        for r in range(N):
            arena.ranks[r].copy_(randn_bf16(K))
        algo = {"allreduce-hd": "halving_doubling", "allreduce-tree": "tree", "allreduce-hier": "hierarchical"}[name]
        step = lambda: ccl.ccl_allreduce_algo(arena.ranks, op="avg", algo=algo, group_size=4, stream=stream)
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        kernel = "hier_order_kernel<bf16, AVG, L=4>" if algo == "hierarchical" else "tree_order_kernel<bf16, AVG, 8>"
        print(json.dumps(line("AllReduce (%s order) HBM GB/s, N=8 bf16 128 MB/rank, 1 GB300" % algo, 2 * N * K * 2,
                              per, launches, kernel, "bf16", {"nranks": N, "count": K, "algo": algo},
                              {"clocks": clk}, total_ms=tot)))
        return

    if name == "allreduce-premul":
        N, K = 8, 64 * 1024 * 1024
        arena = RankArena(N, K, torch.bfloat16, device=dev)
        for r in range(N):
            arena.ranks[r].copy_(randn_bf16(K))
        step = lambda: ccl.ccl_allreduce(arena.ranks, op="avg_premul", stream=stream)
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        print(json.dumps(line("AllReduce (pre-multiplied AVG) HBM GB/s, N=8 bf16 128 MB/rank, 1 GB300", 2 * N * K * 2,
                              per, launches, "fused_reduce_kernel<bf16, AVG_PREMUL, 8 ranks>", "bf16",
                              {"nranks": N, "count": K, "op": "avg_premul"}, {"clocks": clk}, total_ms=tot)))
        return

    if name == "overlap":
        N, TOK, H, F = 8, 4096, 4096, 11008
        numels = W.llama_layer_numels(4)
        shapes = [(H,), (H, H), (H, H), (H, H), (H, H), (H,), (F, H), (F, H), (H, F)] * 4  # (out, in) per tensor
        grads = [[torch.empty(n, dtype=torch.bfloat16, device=dev) for n in numels] for _ in range(N)]
        dYt = {H: torch.randn(H, TOK, generator=g, device=dev).to(torch.bfloat16),
               F: torch.randn(F, TOK, generator=g, device=dev).to(torch.bfloat16)}
        X = {H: torch.randn(TOK, H, generator=g, device=dev).to(torch.bfloat16),
             F: torch.randn(TOK, F, generator=g, device=dev).to(torch.bfloat16)}
        # the bucket kernels go on a high-priority stream: their CTAs are
        # scheduled as soon as the backward GEMMs' CTAs free SMs
        compute, comm = torch.cuda.Stream(dev), torch.cuda.Stream(dev, priority=-1)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        bk = None

        def backward(mark):
            # gradients in reverse registration order, each computed for every rank
            for t in range(len(numels) - 1, -1, -1):
                with torch.cuda.stream(compute):
                    for r in range(N):
                        if len(shapes[t]) == 1:
                            grads[r][t].fill_(1e-3)
                        else:
                            o, i = shapes[t]
                            torch.matmul(dYt[o], X[i], out=grads[r][t].view(o, i))
                    if mark:
                        ev = torch.cuda.Event()
                        ev.record(compute)
                if mark:
                    bk.mark_ready(t, ev, comm)

        def run(kind):
            comm.wait_stream(torch.cuda.current_stream(dev))
            compute.wait_stream(torch.cuda.current_stream(dev))
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record(compute)
            comm.wait_event(a)
            if kind == "backward":
                backward(False)
            elif kind == "allreduce":
                ccl.ccl_bucket_allreduce(grads, bucket_bytes=25 * W.MiB, op="sum", stream=comm)
            else:
                bk.reset()
                backward(True)
            # b: the last gradient is ready; c: the last bucket is reduced
            b.record(compute)
            c.record(comm)
            torch.cuda.synchronize(dev)
            tb_, tc_ = a.elapsed_time(b), a.elapsed_time(c)
            return max(tb_, tc_), max(0.0, tc_ - tb_)

        def timed(kind):
            for _ in range(2):
                run(kind)
            rs = [run(kind) for _ in range(max(3, min(args.steps, 10)))]
            return statistics.median(r[0] for r in rs), statistics.median(r[1] for r in rs)

        tb, tar = timed("backward")[0], timed("allreduce")[0]
        # bucket-size policies (Collective Communication, "Bucket fusion": 5-10 MB
        # start communicating earlier, 50-100 MB amortise the per-bucket cost, 25 MB
        # is PyTorch's reference point), each with the bucket kernels' CTA cap that
        # gives the shortest step
        policies = {}
        for mib in (5, 10, 25, 50, 100):
            res = {}
            for cap in (0, sms // 2, sms):  # CTAs a bucket kernel may hold (0: no cap)
                bk = ccl.CclBucketer(grads, bucket_bytes=mib * W.MiB, op="sum", max_ctas=cap)
                nb = bk.status()[0]
                res[cap] = timed("overlap")
                bk.close()
            best = min(res, key=lambda c_: res[c_][0])
            policies[mib] = {"buckets": nb, "bucket_kernel_max_ctas": best,
                             "overlapped_ms": round(res[best][0], 3), "exposed_tail_ms": round(res[best][1], 3),
                             "overlapped_ms_by_max_ctas": {str(k_): round(v[0], 3) for k_, v in res.items()}}
        to = policies[25]["overlapped_ms"]
        alg = 2 * N * sum(numels) * 2
        d = line("Bucket AllReduce overlapped with a synthetic backward, N=8 bf16 4 Llama layers, 1 GB300", alg,
                 [tar], 62, "bucket_reduce_kernel<bf16, SUM, 8> per bucket", "bf16",
                 {"nranks": N, "tokens": TOK, "buckets": 62},
                 {"overlap": {"backward_ms": round(tb, 3), "allreduce_ms": round(tar, 3), "overlapped_ms": to,
                              "exposed_comm_ms": round(max(to - tb, 0.0), 3),
                              "exposed_tail_ms": policies[25]["exposed_tail_ms"],
                              "hidden_fraction": round(min(1.0, max(0.0, (tb + tar - to) / tar)), 4),
                              "bucket_kernel_max_ctas": policies[25]["bucket_kernel_max_ctas"],
                              "exposed_tail": "time from the last gradient's ready event to the last bucket's "
                                              "completion (the optimizer's wait)",
                              "policies_by_bucket_mib": {str(k_): v for k_, v in policies.items()}}})
        print(json.dumps(d))
        return

    if name == "allreduce-int8":
        N, K = 8, args.count  # 64Mi per rank unless --count picks a profiling size
        grads = [randn_bf16(K) for _ in range(N)]
        res = [torch.zeros(K, dtype=torch.float32, device=dev) for _ in range(N)]
        step = lambda: ccl.ccl_allreduce_compressed(grads, res, op="avg", comp="int8_block", block=128,
                                                    stream=stream)
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        alg = N * K * (2 + 4 + 4 + 2)  # gradients read and written, residuals read and written
        print(json.dumps(line("Compressed AllReduce (INT8 blocks + error feedback) HBM GB/s, N=8 bf16 128 MB/rank, "
                              "1 GB300", alg, per, launches, "compressed_pipe_kernel<bf16, 4, INT8>", "bf16",
                              {"nranks": N, "count": K, "block": 128}, {"clocks": clk}, total_ms=tot)))
        return

    if name == "allreduce-topk":
        N, K = 8, args.count
        kk = K // 100
        grads = [randn_bf16(K) for _ in range(N)]
        res = [torch.zeros(K, dtype=torch.float32, device=dev) for _ in range(N)]
        work = torch.empty(ccl.ccl_plan_topk_work_bytes(N), dtype=torch.uint8, device=dev)
        step = lambda: ccl.ccl_allreduce_topk(grads, res, kk, op="avg", work=work, stream=stream)

        def fresh_inputs(calls=20):
            """Back to back, each step reduces the previous step's sparse output,
            so the residuals drift to bf16-valued numbers.  In training a step
            sees new gradients and fp32 residuals: restore those before every
            call (the copies outside the timed events) and time the call alone."""
            g0 = [randn_bf16(K) for _ in range(N)]
            e0 = [torch.randn(K, generator=g, device=dev) * 1e-3 for _ in range(N)]
            ts = []
            for i in range(calls + 3):
                for r in range(N):
                    grads[r].copy_(g0[r])
                    res[r].copy_(e0[r])
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step()
                b.record(stream)
                torch.cuda.synchronize(dev)
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            ms = statistics.median(ts)
            return {"ms_per_call": round(ms, 4), "GBs": round(alg / (ms / 1e3) / 1e9, 1),
                    "frac": round(alg / (ms / 1e3) / 1e9 / peak, 4), "calls": calls,
                    "inputs": "Normal(0, 1e-3) bf16 gradients and Normal(0, 1e-3) fp32 residuals, restored before "
                              "each call"}

        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        # the least any exact Top-k must move: g and e read once to find the
        # threshold, then gradients and residuals read and written once
        alg = N * K * (2 + 4) + N * K * (2 + 4 + 4 + 2)
        print(json.dumps(line("Top-k AllReduce (1%% kept + error feedback) HBM GB/s of the %d-byte minimum, N=8 bf16 "
                              "%d MB/rank, 1 GB300" % (alg, K * 2 // 2**20), alg, per, launches,
                              "whole step: topk_init, topk_sample, topk_window, topk_main, topk_top_scan, the "
                              "fallback clear and pass (they return at once after a window hit), topk_low_sum, "
                              "topk_low_scan, compressed_pipe_kernel<bf16, 4, TOPK>", "bf16",
                              {"nranks": N, "count": K, "k": kk},
                              {"clocks": clk, "fresh_inputs": fresh_inputs()}, total_ms=tot)))
        return

    if name in ("allreduce-step", "broadcast"):
        N, K = 8, 64 * 1024 * 1024
        arena = RankArena(N, K, torch.bfloat16, device=dev)
        for r in range(N):
            arena.ranks[r].copy_(randn_bf16(K))
        if name == "allreduce-step":
            step = lambda: ccl.ccl_allreduce(arena.ranks, op="avg", mode="step", stream=stream)
            alg, kernel = 2 * N * K * 2, "ring_step_kernel<bf16, AVG> x 14 + AVG scale"
            metric = "AllReduce (step mode) HBM GB/s of the algorithmic 2*N*M bytes, N=8 bf16 128 MB/rank, 1 GB300"
        else:
            step = lambda: ccl.ccl_broadcast(arena.ranks, arena.ranks, root=0, stream=stream)
            alg, kernel = N * K * 2, "fanout_kernel<bf16> (1 source, N-1 destinations)"
            metric = "Broadcast HBM GB/s, N=8 bf16 128 MB, in place, 1 GB300"
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        print(json.dumps(line(metric, alg, per, launches, kernel, "bf16", {"nranks": N, "count": K},
                              {"clocks": clk}, total_ms=tot)))
        return

    if name in ("reduce", "gather", "scatter"):
        # Reduce: 64Mi elements per rank.  Gather / Scatter: 64Mi elements in
        # total unless --count sets the total (e.g. 8x that, 128 MiB per rank)
        N, K = 8, 64 * 1024 * 1024
        if name != "reduce" and args.count != DEFAULT_COUNT:
            K = args.count
        if name == "reduce":
            send = [randn_bf16(K) for _ in range(N)]
            recv = [None] * N
            recv[0] = torch.empty(K, dtype=torch.bfloat16, device=dev)
            step = lambda: ccl.ccl_reduce(send, recv, root=0, op="sum", stream=stream)
            alg, kernel = N * K * 2 + K * 2, "fused_reduce_kernel<bf16, SUM, 8 ranks> (root only)"
            metric = "Reduce HBM GB/s, N=8 bf16 128 MB/rank to one root, 1 GB300"
        else:
            _, ln = ccl.ccl_plan_chunks(K, N)
            parts = [randn_bf16(ln[r]) for r in range(N)]
            full = [None] * N
            full[0] = randn_bf16(K)
            if name == "gather":
                step = lambda: ccl.ccl_gather(parts, full, root=0, stream=stream)
                kernel = "fanout_kernel<bf16> (N sources, 1 destination)"
            else:
                step = lambda: ccl.ccl_scatter(full, parts, root=0, stream=stream)
                kernel = "copy_segments_kernel (N segments)"
            alg = 2 * K * 2
            metric = "%s HBM GB/s, N=8 bf16 %d MB total, 1 GB300" % (name.capitalize(), K * 2 // 2**20)
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        extra = {"clocks": clk}
        if name != "reduce":
            # a short call pays a fixed ramp and drain: the runtime's own device
            # copy of the same bytes (cudaMemcpyAsync), timed the same way, is the
            # roofline a call of this size can reach
            src = torch.empty(K, dtype=torch.bfloat16, device=dev)
            dst = torch.empty(K, dtype=torch.bfloat16, device=dev)
            _, cper, _ = _timed(torch, ccl, lambda: dst.copy_(src), args.steps, args.warmup, stream, dev)
            cgbs = alg * len(cper) / (sum(cper) / 1e3) / 1e9
            ach = alg * len(per) / (sum(per) / 1e3) / 1e9
            extra["same_size_copy"] = {"GBs": round(cgbs, 1), "frac": round(ach / cgbs, 4),
                                       "what": "torch copy_ (cudaMemcpyAsync device to device) of the same %d bytes, "
                                               "per-launch CUDA-event time" % (K * 2)}
            del src, dst
        print(json.dumps(line(metric, alg, per, launches, kernel, "bf16", {"nranks": N, "count": K},
                              extra, total_ms=tot)))
        return

    if name in ("reduce-scatter", "allgather"):
        N, K = 16, 16_777_259
        off, ln = ccl.ccl_plan_chunks(K, N)
        full = [torch.empty(K, dtype=torch.float32, device=dev).uniform_(-1, 1, generator=g) for _ in range(N)]
        part = [torch.empty(ln[r], dtype=torch.float32, device=dev).uniform_(-1, 1, generator=g) for r in range(N)]
        if name == "reduce-scatter":
            step = lambda: ccl.ccl_reduce_scatter(full, part, op="sum", stream=stream)
            alg, kernel = N * K * 4 + K * 4, "fused_reduce_kernel<fp32, SUM, 16 ranks> (ReduceScatter)"
            metric = "ReduceScatter HBM GB/s, N=16 fp32 16,777,259/rank (ragged), 1 GB300"
        else:
            step = lambda: ccl.ccl_allgather(part, full, stream=stream)
            alg, kernel = K * 4 + N * K * 4, "fanout_kernel<fp32> (AllGather)"
            metric = "AllGather HBM GB/s, N=16 fp32 16,777,259 total (ragged), 1 GB300"
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        print(json.dumps(line(metric, alg, per, launches, kernel, "fp32", {"nranks": N, "count": K},
                              {"clocks": clk}, total_ms=tot)))
        return

    if name == "alltoallv":
        N, T, H = 8, 4096, 7168
        counts = W.zipf_expert_counts(N, T, 64, 1.2, 1000) * H
        send = [randn_bf16(T * H) for _ in range(N)]
        recv = [torch.empty(int(counts[:, j].sum()), dtype=torch.bfloat16, device=dev) for j in range(N)]
        cl = counts.tolist()
        step = lambda: ccl.ccl_alltoallv(send, recv, cl, stream=stream)
        alg = 2 * int(counts.sum()) * 2
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        print(json.dumps(line("AllToAllv HBM GB/s, N=8 MoE dispatch 4096x7168 bf16/rank, 1 GB300", alg, per,
                              launches, "copy_segments_kernel (64 blocks)", "bf16",
                              {"nranks": N, "tokens": T, "hidden": H, "max_recv_tokens": int(counts.sum(0).max() // H)},
                              {"clocks": clk}, total_ms=tot)))
        return

    if name == "bucket":
        N, L = 8, args.layers
        numels = W.llama_layer_numels(L)
        nbuckets = len(ccl.ccl_plan_buckets(numels, W.bucket_elems(25 * W.MiB, 2))) - 1
        grads = [[randn_bf16(n) for n in numels] for _ in range(N)]
        step = lambda: ccl.ccl_bucket_allreduce(grads, bucket_bytes=25 * W.MiB, op="sum", stream=stream)
        alg = 2 * N * sum(numels) * 2
        clocks.start()
        tot, per, launches = _timed(torch, ccl, step, args.steps, args.warmup, stream, dev)
        clk = clocks.stop()
        print(json.dumps(line("Bucket-fused AllReduce HBM GB/s, N=8 bf16 %d Llama layer%s (%.2f GB/rank), 25 MiB "
                              "buckets, 1 GB300" % (L, "s" if L != 1 else "", sum(numels) * 2 / 1e9), alg, per,
                              launches, "bucket_reduce_kernel<bf16, SUM, 8>", "bf16",
                              {"nranks": N, "layers": L, "tensors": len(numels), "buckets": nbuckets},
                              {"clocks": clk}, total_ms=tot)))
        return
    raise SystemExit("unknown workload %s" % name)


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=4,
                    help="bucket workload: Llama layers per rank (4 is the benchmark; 1 is a profiling size)")
    ap.add_argument("--count", type=int, default=COUNT,
                    help="elements per rank (default: the 64Mi-element workload; smaller values are for profiling)")
    ap.add_argument("--workload", default="allreduce", choices=["allreduce"] + sorted(ROWS),
                    help="allreduce (the headline) or another collective's workload, each printed as its own line")
    args = ap.parse_args()
    if args.count != COUNT:
        set_count(args.count)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return
    if args.workload != "allreduce":
        run_row(args, args.workload, local)
        return

    import torch

    import ring_allreduce_rank_gb300 as ccl
    from ring_allreduce_rank_gb300 import workloads as W
    from ring_allreduce_rank_gb300.arena import RankArena

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ccl.lib()

    x = W.normal_bf16(NRANKS, COUNT, std=1e-3, seed_base=0)
    arena = RankArena(NRANKS, COUNT, torch.bfloat16, device=dev)
    arena.load([r.view(np.int16) for r in x])
    stream = torch.cuda.current_stream(dev)

    def step():
        ccl.ccl_allreduce(arena.ranks, op="avg", mode="fused", stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = ccl.ccl_launch_count()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ccl.ccl_launch_count() - n0
    if dist:
        dist.barrier()
    clk = clocks.stop()

    total_ms = max_over_ranks(dist, t_all0.elapsed_time(t_all1), dev)
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step = total_ms / args.steps
    value = job_gbs(world, ALG_BYTES, args.steps, total_ms)

    avg_launch_s = statistics.mean(per_launch_ms) / 1e3
    achieved = ALG_BYTES / avg_launch_s / 1e9
    peak, peak_src = measured_peak()
    traffic, ncu_pct = recorded_ncu() if COUNT == DEFAULT_COUNT else (None, None)

    # end to end through the public API with host buffers: every step copies
    # each rank's input from pinned host memory, reduces, and copies each
    # rank's result back (ccl_allreduce_host pipelines the two directions)
    e2e = None
    if args.e2e_steps > 0:
        host_in = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        host_out = torch.empty((NRANKS, COUNT), dtype=torch.bfloat16).pin_memory()
        host_io = ([host_in[r] for r in range(NRANKS)], [host_out[r] for r in range(NRANKS)],
                   torch.empty(HOST_WORK_BYTES, dtype=torch.uint8, device=dev))
        for _ in range(2):
            e2e_step(ccl, host_io, stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step(ccl, host_io, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        direct = ccl.ccl_get_config()["host_path"] == "direct"
        e2e = {"value": round(job_gbs(world, ALG_BYTES, args.e2e_steps, e2e_ms), 2), "unit": UNIT,
               "h2d_bytes_per_step": NRANKS * COUNT * ELEM, "d2h_bytes_per_step": NRANKS * COUNT * ELEM,
               "steps": args.e2e_steps,
               "path": ("ccl_allreduce_host: pinned host rank buffers in and out, read and written in place over "
                        "the host link by the fused AllReduce kernel (both link directions at once)") if direct else
                       ("ccl_allreduce_host: pinned host rank buffers in and out, %d MiB of device stages; "
                        "copy-in, reduction and copy-out of slices overlapped" % (HOST_WORK_BYTES >> 20))}
        del host_io, host_in, host_out

    # alpha: device time of one tiny AllReduce (8 elements per rank), from a
    # CUDA graph of many such calls, so host call overhead is excluded
    tiny = [torch.zeros(8, dtype=torch.bfloat16, device=dev) for _ in range(NRANKS)]
    alpha_s = graph_call_seconds(torch, ccl, lambda st: ccl.ccl_allreduce(tiny, op="sum", stream=st), 16, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, dt, k = oracle_sample_gbs(target_s=12.0)
        nt = max(1, min(NRANKS, os.cpu_count() or 1))
        gbs_t, dt_t, k_t = oracle_sample_gbs(target_s=6.0, threads=nt)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "N=8 bf16 AVG, first %d of %d elements per rank (%.1f s), step-by-step ring "
                         "simulation in plain C, one thread" % (k, COUNT, dt),
               "threaded": {"value": round(gbs_t, 4), "unit": UNIT, "cores": nt,
                            "sample": "the same simulation with one thread per rank and a barrier per step, "
                                      "first %d elements per rank (%.1f s)" % (k_t, dt_t)},
               "cpu_model": cpu_model(), "host_cores": os.cpu_count()}

    if rank != 0:
        return
    M = COUNT * ELEM
    algbw = M / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(world),
        "method": "fused ring-order AllReduce, one launch per step (ReduceScatter fold, AVG scaling and AllGather "
                  "in one pass)",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "frac_of_spec": round(achieved / SPEC_HBM_GBS, 4), "spec_peak_GBs": SPEC_HBM_GBS,
                     "ncu_dram_pct": ncu_pct,
                     "ncu_source": "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed of one full-size launch "
                                   "(profiles/fused_allreduce_bf16_n8_128mib.traffic; null if the kernel sources "
                                   "changed since)",
                     "algorithmic_bytes_per_launch": ALG_BYTES, "peak_source": peak_src,
                     "kernel": "fused_reduce_kernel<bf16, AVG, 8 ranks>",
                     "achieved_median": round(ALG_BYTES / (statistics.median(per_launch_ms) / 1e3) / 1e9, 1),
                     "launch_us": {"mean": round(statistics.mean(per_launch_ms) * 1e3, 2),
                                   "median": round(statistics.median(per_launch_ms) * 1e3, 2),
                                   "min": round(min(per_launch_ms) * 1e3, 2),
                                   "max": round(max(per_launch_ms) * 1e3, 2)}},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "alpha_beta": {"algbw_GBs": round(algbw, 2), "busbw_GBs": round(algbw * 2 * (NRANKS - 1) / NRANKS, 2),
                       "alpha_us": round(alpha_s * 1e6, 3), "beta_GBs": peak,
                       "model_ms": round((2 * (NRANKS - 1) * alpha_s + 2 * (NRANKS - 1) / NRANKS * M /
                                          (peak * 1e9)) * 1e3, 4),
                       "formula": "algbw = M/t; busbw = algbw*2(N-1)/N; T = 2(N-1)alpha + 2(N-1)/N * M/beta, "
                                  "M = bytes per rank, alpha = device time of one 8-element AllReduce (CUDA graph replay), beta = HBM peak"},
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def headline_config(world: int) -> dict:
    """The headline workload, identical for the GPU arm and the reference arm."""
    return {"workload": WORKLOAD, "nranks": NRANKS, "count_per_rank": COUNT, "op": "avg",
            "order": "ring (chunk c folded from rank c, per-hop bf16 rounding)",
            "inputs": "Normal(0, 1e-3) bf16, per-rank seeds",
            "l2": "inputs larger than L2 (1 GiB read per step > 129 MB), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def e2e_step(ccl, host_io, stream):
    send, recv, work = host_io
    ccl.ccl_allreduce_host(send, recv, op="avg", work=work, stream=stream)


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one step-by-step ring
    AllReduce of a bounded sample of the workload on the host cores."""
    import oracle
    from ring_allreduce_rank_gb300 import workloads as W

    oracle.build()
    steps, warm = args.steps, max(args.warmup, 3)
    budget = 120.0  # seconds for the whole run
    _, dt, k = oracle_sample_gbs(target_s=budget / (steps + warm), max_count=COUNT)
    x = list(W.normal_bf16(NRANKS, k, std=1e-3, seed_base=0))
    for _ in range(warm):
        oracle.ring_allreduce(x, "avg")
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.ring_allreduce(x, "avg")
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    val = 2 * NRANKS * k * ELEM * steps / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": UNIT, "n_gpus": 1,
            "steps": steps, "warmup": warm, "ms_per_step": round(tot / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": headline_config(int(os.environ.get("WORLD_SIZE", "1"))),
            "method": "CPU oracle: step-by-step simulation of the ring schedule (2(N-1) steps, per-hop rounding), "
                      "bit-identical to the fused GPU result",
            "cpu_baseline": {"value": round(val, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "N=8 bf16 AVG, first %d of %d elements per rank per step, step-by-step "
                                       "ring simulation in plain C, one thread" % (k, COUNT)},
            "e2e": {"value": round(val, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
