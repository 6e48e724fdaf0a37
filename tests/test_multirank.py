"""The multi-rank host logic of bench.py on CPU (gloo, world size 2).

The path has no exchange step: under torchrun every rank runs its own
replica on its own seed, and the only collective is the max over ranks of
the timings (the slowest rank sets the job time).  The reference arm runs
on rank 0 alone.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    got = bench.max_over_ranks([rank + 1.0, 10.0 - rank, 0.5 * rank], world, "cpu")
    world_seen, rank_seen, _ = bench._dist()
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr((got, world_seen, rank_seen)))


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for rank in range(world):
        got, world_seen, rank_seen = eval(open(tmp_path / f"r{rank}.txt").read())
        assert got == [2.0, 10.0, 0.5]           # every rank sees the slowest rank's figures
        assert (world_seen, rank_seen) == (world, rank)


def test_single_rank_returns_values_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2], 1, "cpu") == [1.5, 2.0]


def test_replicas_get_distinct_seeded_batches():
    from variable_length_flashattention_gb300 import workloads as W
    a, b = W.packed(0 + 0), W.packed(0 + 1)          # rank r runs seed + r
    assert a.lengths_q != b.lengths_q or not torch.equal(a.q, b.q)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
