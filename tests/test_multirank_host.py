"""The N>1 benchmark path on CPU: two gloo ranks agree on the slowest rank's time
and on the whole-job (weak-scaling) tokens/s.  Each GPU rank in a multi-GPU run
decodes its own batch with no collective in the data path; only these timing
reductions cross ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
        value = bench.whole_job_tokens_per_s(world, 32, slowest)
        out_q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    times = [0.31, 0.35]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == pytest.approx(0.35)
        assert value == pytest.approx(2 * 32 / 0.35e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, torch.device("cpu"), 1) == 1.5
    assert bench.whole_job_tokens_per_s(1, 16, 2.0) == pytest.approx(8000.0)
