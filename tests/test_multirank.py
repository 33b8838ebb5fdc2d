"""The multi-replica bench path on CPU with world_size 2 over gloo: the job's step time is the
max over ranks and its throughput counts every rank's tokens; under torchrun the reference
arm prints exactly one line (rank 0) and the other rank exits cleanly."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1.0 + rank * 0.5          # rank 1 is the slower replica
        ms = bench.job_step_ms(local_ms)
        results[rank] = (ms, bench.job_value(4096, world, ms))
    finally:
        dist.destroy_process_group()


def test_job_aggregation_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, value = results[r]
        assert ms == 1.5                     # max over ranks
        assert value == pytest.approx(2 * 4096 / 1.5e-3)


def test_job_aggregation_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_step_ms(2.5) == 2.5
    assert bench.job_value(100, 1, 2.0) == pytest.approx(50000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
