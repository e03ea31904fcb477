"""Multi-rank host logic of the benchmark, on CPU with world-size-2 gloo
ranks: the max-over-ranks reduction of step times, the reference arm that
only rank 0 runs, and the bound on the reference arm's per-step sample.  The
library's data path has no collective (rows are independent; several GPUs
run replicas), so these are the only parts that see more than one rank."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    q.put((rank, bench.max_over_ranks(1.5 + 2.0 * rank, "cpu")))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 3.5), (1, 3.5)]


def test_max_over_ranks_without_group_is_identity():
    import bench

    assert bench.max_over_ranks(2.25, "cpu") == 2.25


def test_reference_rows_per_step_is_bounded():
    import bench

    # many steps: one row per core per step, whatever the budget
    assert bench.reference_rows_per_step(20000, 16, 0.01) == 16
    # few steps: the whole batch
    assert bench.reference_rows_per_step(10, 16, 0.01) == bench.B
    # in between: whole rounds of one row per core that fit the budget
    r = bench.reference_rows_per_step(500, 8, 0.01, budget_s=120.0)
    assert r % 8 == 0 and 500 * (r // 8) * 0.01 <= 120.0


def test_reference_arm_two_ranks_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
