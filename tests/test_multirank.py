"""The N > 1 path of the benchmark on CPU: two gloo ranks.

The step has no exchange in it, so N GPUs run N independent replicas; the only
collectives are the barrier around the timed region and the max over ranks of
the elapsed time.  These tests run those pieces with world_size 2 on the gloo
backend, check that replicas draw independent (seeded per rank) workloads of the
same size, and that the reference arm's non-zero ranks exit quietly."""
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


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from chunked_prefill_paged_cpa_gb300 import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank reports a different elapsed time; all must see the max
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")
        # replicas: the same workload shape, seeded per rank
        sc = workloads.scenario("tiny", seed=rank)
        ws = workloads.WorkloadState(sc, device="cpu")
        inp = ws.step(0)
        tokens = inp["meta"].num_tokens
        checksum = float(inp["q"].double().sum())
        got = [None] * world
        dist.all_gather_object(got, (t, tokens, checksum))
        torch.save(got, os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


def test_barrier_max_over_ranks_and_independent_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        got = torch.load(tmp_path / f"rank{rank}.pt")
        times = [g[0] for g in got]
        tokens = [g[1] for g in got]
        sums = [g[2] for g in got]
        assert times == [2.5, 2.5]               # max over ranks seen by every rank
        assert tokens[0] == tokens[1] > 0         # same step size on every replica
        assert sums[0] != sums[1]                 # but independent (seeded per rank) inputs


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
