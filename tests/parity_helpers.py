"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (fixed here, used by every parity test):
  * index lists and argmax assignments: bit-exact, except that a mismatch is
    accepted where the fp64 scores of the swapped positions differ by less
    than 1e-5 (the fp32 score gap rule); in addition the GPU's lists must be
    exactly the top-w (and argmax) of the GPU's own fp32 scores.
  * attention output: 2e-2 max-abs for bf16 inputs with fp32 accumulation,
    1e-4 for fp32 inputs, against the oracle evaluated on the GPU's lists.
  * centroid update: 1e-5 max-abs, on the GPU's own assignment.
  * scores: 1e-5 max-abs against the fp64 scores.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.routing_oracle as orc

TIE_GAP = 1e-5
TOL_OUT = {"bf16": 2e-2, "f32": 1e-4}
TOL_EMA = 1e-5
TOL_SCORE = 1e-5


def to_device(wl, device="cuda"):
    if wl.dtype == "f32":
        q = torch.from_numpy(np.ascontiguousarray(wl.q)).to(device)
        v = torch.from_numpy(np.ascontiguousarray(wl.v)).to(device)
    else:
        q = torch.from_numpy(np.ascontiguousarray(wl.q).view(np.int16)).view(torch.bfloat16).to(device)
        v = torch.from_numpy(np.ascontiguousarray(wl.v).view(np.int16)).view(torch.bfloat16).to(device)
    mu = torch.from_numpy(np.ascontiguousarray(wl.centroids)).to(device)
    return q, v, mu


def out_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_index_lists(gpu_idx: np.ndarray, S64: np.ndarray, w: int, n: int):
    """gpu_idx [k, w] for one (b, h); S64 [k, n] fp64 scores."""
    k = S64.shape[0]
    assert gpu_idx.shape == (k, w)
    assert gpu_idx.min() >= 0 and gpu_idx.max() < n
    assert np.all(np.diff(gpu_idx, axis=1) > 0), "lists must be strictly ascending"
    want = orc.top_w_per_centroid(S64, w)
    mism = 0
    for c in range(k):
        G, O = set(gpu_idx[c].tolist()), set(want[c].tolist())
        if G == O:
            continue
        mism += 1
        for i in G - O:
            for j in O - G:
                gap = abs(S64[c, i] - S64[c, j])
                assert gap < TIE_GAP, (
                    f"centroid {c}: GPU kept {i}, oracle kept {j}, score gap {gap:.3g}")
    return mism


def check_assign(gpu_a: np.ndarray, S64: np.ndarray):
    want = orc.kmeans_assign(S64)
    bad = np.nonzero(gpu_a != want)[0]
    for t in bad:
        gap = abs(S64[gpu_a[t], t] - S64[want[t], t])
        assert gap < TIE_GAP, f"row {t}: GPU centroid {gpu_a[t]}, oracle {want[t]}, gap {gap:.3g}"
    return len(bad)


def check_self_consistent(gpu_idx: np.ndarray, gpu_a: np.ndarray, gpu_S: np.ndarray, w: int):
    """The GPU's lists are exactly the top-w / argmax of its own fp32 scores."""
    S = gpu_S.astype(np.float64)
    assert np.array_equal(gpu_idx, orc.top_w_per_centroid(S, w))
    if gpu_a is not None:
        assert np.array_equal(gpu_a, orc.kmeans_assign(S))


def oracle_scores(q64_head: np.ndarray, mu_head: np.ndarray) -> np.ndarray:
    return orc.centroid_scores(orc.normalise_rows(q64_head), mu_head.astype(np.float64))


def oracle_output_on(q64_head, v64_head, idx_head, causal, scale):
    n = q64_head.shape[0]
    Y = np.stack([orc.cluster_attention(q64_head, q64_head, v64_head, idx_head[c], causal, scale)
                  for c in range(idx_head.shape[0])])
    return orc.scatter_average(Y, idx_head, n)
