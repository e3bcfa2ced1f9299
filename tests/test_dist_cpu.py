"""The multi-process (N > 1) path of bench.py, run as two CPU ranks over gloo.

Decode sequences are independent, so N GPUs run N replicas of the workload
and meet only at the timing barrier and a MAX reduction of the step time
(the slowest rank sets the job time) plus a SUM of the work done; these
tests run exactly those helpers with world_size 2 on the host, and the
reference arm under torchrun, where rank 0 alone prints the JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    bench.init_dist(world, "gloo")
    try:
        bench.barrier(world)
        step_s = [0.25, 0.75][rank]          # the second rank is slower
        tokens = [8, 8][rank]
        t_max = bench.max_over_ranks(step_s, world)
        t_sum = bench.sum_over_ranks(tokens, world)
        bench.barrier(world)
        out[rank] = (t_max, t_sum)
    finally:
        dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        # every rank sees the slowest rank's time and the work of both
        assert dict(out) == {0: (0.75, 16.0), 1: (0.75, 16.0)}


def test_reference_arm_two_ranks_prints_one_line():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-budget-s", "0.5"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
