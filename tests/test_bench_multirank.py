"""The benchmark's multi-replica harness on CPU: two gloo ranks agree on the
slowest replica's time, the whole-job throughput counts every replica's bytes,
and the reference arm under torchrun runs on rank 0 only."""
import datetime
import os
import socket
import subprocess
import sys
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    ms = [10.0, 12.5][rank]
    got = bench.max_over_ranks(dist, ms, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 12.5, 1: 12.5}


def test_job_gbs_counts_every_replica():
    one = bench.job_gbs(1, bench.ALG_BYTES, 10, 5.0)
    assert bench.job_gbs(4, bench.ALG_BYTES, 10, 5.0) == pytest.approx(4 * one)
    assert one == pytest.approx(bench.ALG_BYTES * 10 / 5e-3 / 1e9)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def _leaver(rank, world, port, q):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    dist.barrier()
    if rank == 1:
        q.put((rank, "left"))
        q.close()
        q.join_thread()
        os._exit(0)  # leaves between steps: nothing of it is in flight
    t0 = time.time()
    try:
        bench.max_over_ranks(dist, 1.0, "cpu")
        q.put((rank, "no error"))
    except Exception:
        q.put((rank, "error after %.1f s" % (time.time() - t0)))
    q.close()
    q.join_thread()
    os._exit(0)


def test_replica_that_leaves_is_detected_within_the_timeout():
    """A replica that exits between steps: the other one's next timing
    reduction ends with an error inside the process-group timeout instead of
    hanging (failure made on the host, no GPU involved)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaver, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode is not None
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[1] == "left"
    assert res[0].startswith("error after")
    assert float(res[0].split()[2]) < 60
