"""The bench's multi-rank host logic on CPU: two gloo ranks (one process each, as torchrun
would start them) reduce their timings to the slowest rank's, and the whole-job µs per
token counts every rank's tokens. No GPU is used."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, times, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        total = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
        q.put((rank, total, bench.per_token_us(total, 10, 4, world)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, times = 2, [12.5, 17.0]            # ms for 10 steps on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, us in out:
        assert total == pytest.approx(17.0)
        # 10 steps of 4 tokens on each of 2 ranks in 17 ms: 17 ms / 80 tokens
        assert us == pytest.approx(17.0 * 1000.0 / 80)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, torch.device("cpu"), 1) == 3.25
    assert bench.per_token_us(20.0, 20, 1, 1) == pytest.approx(1000.0)
