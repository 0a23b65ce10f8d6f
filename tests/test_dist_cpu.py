"""The multi-rank host logic of bench.py on CPU with the gloo backend,
world_size 2: every rank runs its own batch (no data-path collective); the
only collective is the max of the per-rank time, and the reported rate is all
ranks' tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, w)
    rate = bench.aggregate_rate(4096 * 3, w, slowest * 3 / 1e3)
    q.put((r, w, lr, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_and_aggregation_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r, (rank, w, lr, slowest, rate) in enumerate(out):
        assert rank == r and w == world and lr == r
        assert slowest == 15.0                  # max over ranks
        assert rate == pytest.approx(4096 * 3 * 2 / (15.0 * 3 / 1e3))


def test_single_rank_defaults():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_rate(100, 1, 0.5) == 200.0


def test_reference_arm_only_on_rank0(monkeypatch):
    import bench
    from top_routing_grouped_bias_b300 import synth
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 0
    assert bench.bench_reference(A, synth.WORKLOADS["tiny_fp32"]) is None
