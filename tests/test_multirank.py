"""The benchmark's multi-rank path on CPU (gloo, world size 2): ranks run independent
replicas of the workload and only the timing is combined, as the slowest rank's time
over the work of all ranks; under torchrun the reference arm prints one line, on rank 0."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks(rank, world, port, out):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = [3.5, 5.25][rank]  # rank 1 is the slow one
        t = bench.max_over_ranks(ms, "cpu")
        out[rank] = (t, bench.job_rate(100.0, world, t * 1e-3))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:  # no fork: CUDA may be initialised
        out = m.dict()
        mp.spawn(_ranks, args=(world, free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, rate = res[rank]
        assert t == 5.25                    # every rank sees the slowest rank's time
        assert rate == 100.0 * 2 / 5.25e-3  # all ranks' units over that time


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
           "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
