"""bench.py's multi-rank host logic on CPU: world-size-2 gloo process groups
(barrier, max over ranks of the step time, weak-scaling aggregation, and the
reference arm's rank-0-only output)."""

import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.reduce_max(1.5 * (rank + 1), world)
        env = bench.dist_env()
        args = bench.parse_args(["--impl", "reference", "--workload", "enc_self_f32", "--steps", "1",
                                 "--warmup", "0"])
        line = bench.run_reference(args, env[0], env[1])
        queue.put((rank, slowest, env, line is not None))
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_max_and_reference_rank0_only():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in results] == [3.0, 3.0]                  # max over ranks
    assert [r[2] for r in results] == [(0, 2, 0), (1, 2, 1)]      # RANK, WORLD_SIZE, LOCAL_RANK
    assert [r[3] for r in results] == [True, False]               # only rank 0 prints a line


def test_weak_scaling_aggregate():
    # Two ranks, 1 TFLOP each per step, slowest rank 2 ms per step -> 1000 TFLOP/s.
    assert bench.aggregate_tflops(1e12, 2, 2.0) == pytest.approx(1000.0)
    assert bench.aggregate_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
