"""The benchmark's multi-rank bookkeeping on CPU with the gloo backend.

bench.py runs one replica of the workload per GPU (weak scaling; the forward
shards by head and batch with no exchange).  Its only cross-rank steps are
the barrier and the max-over-ranks step time that turns into the whole-job
throughput; these are checked here with two gloo ranks on the CPU."""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.slowest_rank_ms(1.5 + rank)  # rank 1 is the slow one
        dist.barrier()
        q.put((rank, t, bench.job_tokens_per_s(8192, world, t)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [2.5, 2.5]        # both ranks see the slowest time
    assert got[0][2] == pytest.approx(2 * 8192 / 2.5e-3)  # all ranks' tokens / that time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(3.25) == 3.25
    assert bench.job_tokens_per_s(8192, 1, 0.1) == pytest.approx(8192 / 1e-4)


def test_local_attention_flop_count():
    # closed form vs a direct sum over positions (window below, at and above n)
    import bench
    for n, d, W in ((10, 4, 3), (37, 8, 37), (5, 2, 9), (8192, 128, 512)):
        keys = sum(min(t + 1, W) for t in range(n))
        assert bench.local_attention_flops(2, n, d, W) == 4.0 * d * keys * 2
