"""Centroid update for a batch sharded over GPUs (one process per GPU).

The forward pass shards by sequence with no exchange (each sequence is routed
and attended on its own), but the centroid step averages over every sequence
of the batch: centroids are shared across sequences ("Efficient
Content-Based Sparse Attention with Routing Transformers", §4 "Routing
attention with clustering"; §2, mini-batch spherical k-means).  So each rank
computes its shard's per-centroid sums and counts, one all-reduce (SUM) adds
them, and every rank applies the same blend, which keeps the replicas'
centroids identical.  torch.distributed carries the all-reduce (NCCL on GPU);
the sums and the blend run in the CUDA library.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import _binding


def sharded_centroid_ema(qk: torch.Tensor, assign: torch.Tensor, centroids: torch.Tensor,
                         decay: float, group=None, workspace=None, stream=None) -> torch.Tensor:
    """One centroid step over the union of every rank's shard, in place.

    qk [B_local, H, n, d] and assign [B_local, H, n] are this rank's
    sequences; centroids [H, k, d] must be identical on every rank (they stay
    so).  Without an initialised process group this is rt_centroid_ema split
    in its two halves.
    """
    import torch.distributed as dist

    H, k, d = centroids.shape
    sums = _binding.rt_centroid_ema_sums(qk, assign, k, workspace=workspace, stream=stream)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(sums, op=dist.ReduceOp.SUM, group=group)
    return _binding.rt_centroid_ema_apply(sums, centroids, decay, stream=stream)
