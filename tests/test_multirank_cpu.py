"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank draws
its own batch, the timed region is the slowest rank's, the whole-job rate counts the
units of all ranks, and the reference arm runs on rank 0 alone.  No GPU is used."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, elapsed, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        t = bench.max_over_ranks(elapsed[rank], dist, torch.device("cpu"))
        wl = synth.WORKLOADS["c1"]
        inp = synth.make_inputs(wl, bench.rank_seed(wl.name, rank))
        # every rank sees the other's batch checksum: the batches differ
        mine = torch.tensor([float(np.asarray(inp["tgt"], np.float64).sum())], dtype=torch.float64)
        both = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(both, mine)
        dist.barrier()
        out[rank] = (t, [float(x.item()) for x in both])
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_distinct_batches():
    world = 2
    elapsed = [12.5, 17.25]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), elapsed, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r][0] == max(elapsed)
    sums = res[0][1]
    assert sums == res[1][1] and sums[0] != sums[1]


def test_job_rate_counts_every_rank():
    assert bench.job_rate(1000, 1, 500.0) == pytest.approx(2000.0)
    assert bench.job_rate(1000, 4, 500.0) == pytest.approx(8000.0)
    assert bench.max_over_ranks(3.0, None, None) == 3.0


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
