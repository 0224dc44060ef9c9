"""The multi-GPU bench path is replicas only (no collective on the data
path): its host logic, the maximum over ranks of the timed region, the
weak-scaling job rate and rank-0-only reporting, exercised with a two-rank
gloo process group on the CPU."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out_q.put((rank, bench.max_over_ranks(dist, values[rank])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [[1.5, 7.0, 0.25], [2.5, 3.0, 0.5]]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert got[r] == [2.5, 7.0, 0.5]


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3.0, 1.0]) == [3.0, 1.0]


def test_whole_job_rate_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    # each of 4 ranks moves 3.37e9 bytes; the slowest took 1.5 ms
    assert bench.whole_job_rate(3.37e9, 1.5e-3, 4) == pytest.approx(4 * 3.37e9 / 1.5e-3)
    assert bench.whole_job_rate(10.0, 2.0, 1) == 5.0


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_only_rank0_reports():
    other = _run_reference(1, 2)
    assert other.returncode == 0 and other.stdout.strip() == ""
    first = _run_reference(0, 2)
    assert first.returncode == 0
    line = json.loads(first.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
