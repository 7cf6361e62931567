"""The N > 1 path of bench.py on CPU: two gloo ranks, replicas only (no data-path collective).

Each rank reports its own step time; the job time is the maximum over ranks, and the throughput
counts the units every rank processed.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(w, "gloo")
    try:
        t = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        dist.barrier()
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0


def test_reference_arm_prints_once_under_two_ranks():
    # `bench.py --impl reference` launched as two ranks: rank 0 times the oracle and prints the one
    # JSON line, rank 1 exits 0 without work.
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
        p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                            "--ref-budget", "1"], cwd=root, env=env, capture_output=True, text=True, timeout=600)
        assert p.returncode == 0, p.stderr[-2000:]
        outs.append(p.stdout.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["gpu_launches"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
