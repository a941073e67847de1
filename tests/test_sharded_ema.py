"""The batch-sharded centroid step, across two gloo ranks on the CPU.

sharded_centroid_ema splits the step into this rank's sums, one all-reduce and
the blend.  Its cross-rank logic -- which rows each rank sums, that the
all-reduce adds the shards, that every rank applies the same blend -- is run
here with two gloo processes.  The two device halves are replaced by the
oracle's restatement of the same halves (centroid_sums / centroid_apply, each
pinned in test_oracle_pins.py), since this machine has no GPU; the result must
equal the oracle's one-call step on the whole batch on both ranks.  The CUDA
halves themselves are compared with the oracle in test_gpu_parity.py.
"""

import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    rng = np.random.default_rng(3)
    B, H, n, d, k = 4, 2, 40, 8, 5
    x = rng.standard_normal((B, H, n, d))
    a = rng.integers(0, k, size=(B, H, n))
    a[:, 1, :] = np.where(a[:, 1, :] == 4, 0, a[:, 1, :])  # head 1: centroid 4 empty
    mu = rng.standard_normal((H, k, d))
    mu /= np.linalg.norm(mu, axis=-1, keepdims=True)
    return x, a, mu


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle.routing_oracle as orc
    from content_sparse_attention_shared_b300 import _binding, sharded

    # host stand-ins for the two device halves (same arguments, CPU tensors)
    def fake_sums(qk, assign, k, workspace=None, stream=None):
        return torch.from_numpy(orc.centroid_sums(qk.numpy(), assign.numpy(), k))

    def fake_apply(sums, centroids, decay, stream=None):
        centroids.copy_(torch.from_numpy(orc.centroid_apply(sums.numpy(), centroids.numpy(), decay)))
        return centroids

    _binding.rt_centroid_ema_sums = fake_sums
    _binding.rt_centroid_ema_apply = fake_apply
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, a, mu = _batch()
        per = x.shape[0] // world
        lo, hi = rank * per, (rank + 1) * per
        c = torch.from_numpy(mu.copy())
        sharded.sharded_centroid_ema(torch.from_numpy(x[lo:hi]), torch.from_numpy(a[lo:hi]), c, 0.6)
        q.put((rank, c.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_equal_the_whole_batch_step():
    sys.path.insert(0, ROOT)
    import oracle.routing_oracle as orc

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x, a, mu = _batch()
    want = orc.centroid_ema(x, a, mu, 0.6)
    for r in (0, 1):
        np.testing.assert_allclose(got[r], want, atol=1e-12)
    assert np.array_equal(got[0], got[1])            # replicas stay identical
    assert np.array_equal(got[0][1, 4], mu[1, 4])   # empty centroid untouched
