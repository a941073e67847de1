"""fp64 CPU oracle for routing attention -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow reference the CUDA library is checked against.
Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import it; the library itself never calls it and has no CPU fallback.
It shares no code with the CUDA path: it reads the same seeded inputs and
restates the method step by step in float64, one numpy library primitive
(matmul, sort, exp) per step, without blocking, fusion or reordering.

Method: "Efficient Content-Based Sparse Attention with Routing Transformers"
(Roy, Saffar, Vaswani, Grangier).  The pages available state the method only
in summary form (paperlayer.ai source-linked summary, §3 and §4; arXiv
abstract).  Where they leave a step open the plainest reading is taken and
named in the docstring of the step ("reading: ...").

Steps (per batch b and head h, with Q shared as K):
  a1 normalise   r_t = (x_t - mean x_t) / ||x_t - mean x_t||       (0 if norm 0)
  a2 score       S[c, t] = <r_t, mu_c>;  a_t = first argmax_c S[c, t]
  a3 select      T_c = the w tokens with largest S[c, .], ties -> lower t
  a4 sort        idx[c] = T_c in ascending position order
  a5 attention   inside each cluster: softmax(scale * Q_c K_c^T + causal mask) V_c
  a6 scatter     O[t] = mean of t's per-cluster outputs; 0 if t is in no cluster
  a7 update      mu_c <- normalise(decay * mu_c + (1 - decay) * mean of the r_t
                 with a_t = c, over every sequence of the batch); unchanged if none
  a7' variant    the same step with the tokens of c's own top-w lists in place of
                 the argmax assignment (centroid_ema_topw)
  a7 in halves   per-centroid sums and counts of a shard of the batch
                 (centroid_sums), added over shards, then the blend
                 (centroid_apply)
  local          the companion layer: causal attention of every position over the
                 `window` positions ending at it (local_attention)
  backward       gradients of a5..a6 with respect to the shared Q/K rows and V,
                 routing held fixed (routing_attention_head_backward)
  separate QK    queries and keys routed separately by the same centroids
                 (routing_attention_head_separate)

Parity status: every function below is pinned by tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force, library
routines); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "normalise_rows",
    "centroid_scores",
    "kmeans_assign",
    "top_w_per_centroid",
    "cluster_attention",
    "scatter_average",
    "membership_counts",
    "routing_attention_head",
    "routing_attention",
    "centroid_ema",
    "centroid_ema_topw",
    "centroid_sums",
    "centroid_apply",
    "local_attention",
    "routing_attention_head_backward",
    "routing_attention_head_separate",
]


def normalise_rows(x: np.ndarray) -> np.ndarray:
    """a1: project each row onto the unit sphere.

    Source: §4 "Routing attention with clustering" (unit-normalised queries and
    keys make nearest-centroid routing a maximum-inner-product search).
    Reading: "layer-normalised onto the unit sphere" = subtract the row mean
    (layer norm without affine; its variance scaling does not change the
    direction), then divide by the Euclidean norm.  A row whose centred norm is
    exactly 0 maps to the zero vector.
    """
    x = np.asarray(x, dtype=np.float64)
    u = x - x.mean(axis=-1, keepdims=True)
    nrm = np.sqrt((u * u).sum(axis=-1, keepdims=True))
    safe = np.where(nrm > 0.0, nrm, 1.0)
    return np.where(nrm > 0.0, u / safe, 0.0)


def centroid_scores(r: np.ndarray, mu: np.ndarray) -> np.ndarray:
    """a2: S[c, t] = <r_t, mu_c> for r [n, d] and mu [k, d]; returns [k, n].

    Source: §4 "Routing attention with clustering": routing compares every
    token with every centroid, O(nkd).  Reading: the nearest centroid is the
    one with the largest inner product (centroids are kept at unit norm, so
    this equals the smallest Euclidean distance).
    """
    r = np.asarray(r, dtype=np.float64)
    mu = np.asarray(mu, dtype=np.float64)
    return mu @ r.T


def kmeans_assign(S: np.ndarray) -> np.ndarray:
    """a2: a_t = the centroid with the largest score; ties go to the lower index.

    Source: §4 (nearest-centroid routing of the online k-means).  np.argmax
    returns the first maximum, which is the lower-index tie rule.
    """
    return np.argmax(np.asarray(S), axis=0).astype(np.int64)


def top_w_per_centroid(S: np.ndarray, w: int) -> np.ndarray:
    """a3 + a4: for every centroid the w tokens with the largest score, ties
    to the lower position, listed in ascending position order.  Returns [k, w].

    Source: §4 "Routing attention with clustering": balanced clusters, each
    query compares with about n/k keys, via a top-k assignment of cost
    O(n log n).  Reading: each centroid takes its own top-w tokens (so a token
    may sit in several clusters or in none), and the chosen tokens are put back
    in position order so the causal mask inside a cluster is the plain lower
    triangle.
    """
    S = np.asarray(S)
    k, n = S.shape
    if not (1 <= w <= n):
        raise ValueError("need 1 <= w <= n")
    pos = np.arange(n)
    out = np.empty((k, w), dtype=np.int64)
    for c in range(k):
        # primary key: score descending; secondary: position ascending
        order = np.lexsort((pos, -S[c]))
        out[c] = np.sort(order[:w])
    return out


def cluster_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, members: np.ndarray,
                      causal: bool, scale: float, return_probs: bool = False):
    """a5: dense softmax attention restricted to one cluster.

    q, k, v: [n, d] rows of one (batch, head); members: ascending positions of
    the cluster.  Returns Y [w, d] (and P [w, w] if asked).

    Source: §3 "Self-Attentive Auto-regressive Sequence Modeling" (an n-by-n
    attention matrix from queries and keys, rows normalised with softmax,
    output = attention times values; autoregressive queries see only earlier
    positions) and §4 (only query-key pairs of the same cluster are
    considered).  Readings: the attention uses the raw Q, K, V rows (the
    normalised vectors serve routing only); a position attends to itself; the
    causal mask compares original positions, i.e. key p_j is visible to query
    p_i iff p_j <= p_i.
    """
    members = np.asarray(members)
    qc = np.asarray(q, dtype=np.float64)[members]
    kc = np.asarray(k, dtype=np.float64)[members]
    vc = np.asarray(v, dtype=np.float64)[members]
    logits = scale * (qc @ kc.T)
    if causal:
        visible = members[None, :] <= members[:, None]
        logits = np.where(visible, logits, -np.inf)
    row_max = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - row_max)
    P = e / e.sum(axis=1, keepdims=True)
    Y = P @ vc
    if return_probs:
        return Y, P
    return Y


def membership_counts(idx: np.ndarray, n: int) -> np.ndarray:
    """m_t = number of clusters whose member list contains position t."""
    return np.bincount(np.asarray(idx).reshape(-1), minlength=n)[:n]


def scatter_average(Y: np.ndarray, idx: np.ndarray, n: int) -> np.ndarray:
    """a6: put every cluster's outputs back at their positions.

    Y [k, w, d], idx [k, w].  Reading: a position chosen by several clusters
    gets the plain arithmetic mean of its outputs; a position chosen by none
    gets a zero row (the pages leave the combination open).
    """
    Y = np.asarray(Y, dtype=np.float64)
    idx = np.asarray(idx)
    d = Y.shape[-1]
    acc = np.zeros((n, d), dtype=np.float64)
    np.add.at(acc, idx.reshape(-1), Y.reshape(-1, d))
    m = membership_counts(idx, n)
    out = np.zeros((n, d), dtype=np.float64)
    hit = m > 0
    out[hit] = acc[hit] / m[hit, None]
    return out


def routing_attention_head(q, k, v, mu, w: int, causal: bool = True, scale=None,
                           idx=None):
    """a1..a6 for one (batch, head): returns dict(O, idx, assign, S).

    Routing uses the normalised shared query/key rows; ``idx`` may be given to
    evaluate a5..a6 on externally chosen clusters (e.g. another
    implementation's index lists).
    """
    q = np.asarray(q, dtype=np.float64)
    n, d = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(d)
    r = normalise_rows(q)
    S = centroid_scores(r, mu)
    a = kmeans_assign(S)
    if idx is None:
        idx = top_w_per_centroid(S, w)
    idx = np.asarray(idx)
    Y = np.stack([cluster_attention(q, k, v, idx[c], causal, scale)
                  for c in range(idx.shape[0])])
    O = scatter_average(Y, idx, n)
    return {"O": O, "idx": idx, "assign": a, "S": S}


def routing_attention(q, k, v, mu, w: int, causal: bool = True, scale=None):
    """a1..a6 over [B, H, n, d] inputs with centroids [H, k, d] shared across
    the batch (§4: centroids are shared across sequences)."""
    q = np.asarray(q, dtype=np.float64)
    B, H, n, d = q.shape
    kc = mu.shape[1]
    O = np.zeros((B, H, n, d))
    idx = np.zeros((B, H, kc, w), dtype=np.int64)
    assign = np.zeros((B, H, n), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            res = routing_attention_head(q[b, h], k[b, h], v[b, h], mu[h], w, causal, scale)
            O[b, h], idx[b, h], assign[b, h] = res["O"], res["idx"], res["assign"]
    return O, idx, assign


def centroid_ema(qk: np.ndarray, assign: np.ndarray, mu: np.ndarray, decay: float) -> np.ndarray:
    """a7: one online spherical k-means step for every head's centroids.

    qk [B, H, n, d] (raw rows; normalised here exactly as in a1),
    assign [B, H, n], mu [H, k, d].  Returns the updated centroids (float64).

    Source: §2 "Attention with Content-Based Sparsity" (centroids learned with
    mini-batch spherical k-means), §4 (centroids shared across sequences,
    learned online), §6 "Local vs Global" (spherical k-means over the global
    token set).  Readings: each token counts toward its argmax centroid only;
    the batch mean over every sequence of the head is blended in with weight
    (1 - decay); the result is put back on the unit sphere; a centroid with no
    assigned token is left exactly as it was.
    """
    qk = np.asarray(qk, dtype=np.float64)
    B, H, n, d = qk.shape
    mu = np.asarray(mu, dtype=np.float64)
    out = mu.copy()
    r = normalise_rows(qk)
    for h in range(H):
        rh = r[:, h].reshape(B * n, d)
        ah = np.asarray(assign)[:, h].reshape(B * n)
        for c in range(mu.shape[1]):
            sel = ah == c
            cnt = int(sel.sum())
            if cnt == 0:
                continue
            mean = rh[sel].sum(axis=0) / cnt
            blended = decay * mu[h, c] + (1.0 - decay) * mean
            nrm = np.sqrt((blended * blended).sum())
            out[h, c] = blended / nrm if nrm > 0 else blended
    return out


def centroid_ema_topw(qk: np.ndarray, idx: np.ndarray, mu: np.ndarray, decay: float) -> np.ndarray:
    """a7 variant: the centroid step driven by the top-w membership.

    qk [B, H, n, d] (raw rows; normalised as in a1), idx [B, H, k, w] (each
    centroid's kept positions, as a3/a4 produce them; entries outside [0, n)
    are ignored), mu [H, k, d].  Returns the updated centroids (float64).

    Source: §4 "Routing attention with clustering" (balanced clusters through
    a top-k assignment; centroids shared across sequences and learned online),
    §2 (mini-batch spherical k-means).  Reading: the pages do not say which
    membership moves a centroid; centroid_ema takes the argmax assignment,
    this variant takes the tokens each centroid selected itself.  Centroid c of
    head h moves toward the mean of the normalised rows listed in idx[b, h, c]
    for every sequence b (a token listed by several centroids counts for each
    of them), blended with weight (1 - decay) and put back on the unit sphere;
    with no valid entry it is left exactly as it was.
    """
    qk = np.asarray(qk, dtype=np.float64)
    B, H, n, d = qk.shape
    idx = np.asarray(idx)
    mu = np.asarray(mu, dtype=np.float64)
    out = mu.copy()
    r = normalise_rows(qk)
    for h in range(H):
        for c in range(mu.shape[1]):
            rows = [r[b, h, t] for b in range(B) for t in idx[b, h, c] if 0 <= t < n]
            if not rows:
                continue
            mean = np.sum(rows, axis=0) / len(rows)
            blended = decay * mu[h, c] + (1.0 - decay) * mean
            nrm = np.sqrt((blended * blended).sum())
            out[h, c] = blended / nrm if nrm > 0 else blended
    return out


def centroid_sums(qk: np.ndarray, assign: np.ndarray, k: int) -> np.ndarray:
    """a7, first half: for every head h and centroid c, the sum of the
    normalised rows r_t assigned to c over the sequences given, and how many
    there are.  qk [B, H, n, d], assign [B, H, n] (entries outside [0, k) count
    for no centroid).  Returns [H, k, d + 1]: the sum in [..., :d], the count
    in [..., d].

    Source: §4 "Routing attention with clustering" (centroids shared across
    sequences), §2 (mini-batch k-means).  Reading: a batch split into shards
    (one per GPU) gives each shard a part of every centroid's sum and count;
    the parts add up to the whole batch's, so one all-reduce of these arrays
    followed by centroid_apply is the step centroid_ema takes on the batch.
    """
    qk = np.asarray(qk, dtype=np.float64)
    B, H, n, d = qk.shape
    r = normalise_rows(qk)
    a = np.asarray(assign)
    out = np.zeros((H, k, d + 1))
    for h in range(H):
        rh = r[:, h].reshape(B * n, d)
        ah = a[:, h].reshape(B * n)
        for c in range(k):
            sel = ah == c
            out[h, c, :d] = rh[sel].sum(axis=0)
            out[h, c, d] = sel.sum()
    return out


def centroid_apply(sums: np.ndarray, mu: np.ndarray, decay: float) -> np.ndarray:
    """a7, second half: blend each centroid toward the mean sum / count and put
    it back on the unit sphere; a centroid with count 0 is left as it was.
    sums [H, k, d + 1] (as centroid_sums returns, possibly added over shards),
    mu [H, k, d].  Returns the updated centroids (float64).

    Source and readings as centroid_ema (§2, §4, §6 "Local vs Global").
    """
    sums = np.asarray(sums, dtype=np.float64)
    mu = np.asarray(mu, dtype=np.float64)
    d = mu.shape[-1]
    out = mu.copy()
    for h in range(mu.shape[0]):
        for c in range(mu.shape[1]):
            cnt = sums[h, c, d]
            if cnt <= 0:
                continue
            blended = decay * mu[h, c] + (1.0 - decay) * sums[h, c, :d] / cnt
            nrm = np.sqrt((blended * blended).sum())
            out[h, c] = blended / nrm if nrm > 0 else blended
    return out


def local_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int,
                    scale: float) -> np.ndarray:
    """Local (sliding-window) causal attention of one (batch, head).

    q, k, v: [n, d].  Position t attends to the positions
    max(0, t - window + 1) .. t (itself included); returns O [n, d].

    Source: §3 (causal and local attention choose each query's key set from
    positions alone; softmax rows, autoregressive masking), §6 "Local vs
    Global" (local attention with windows of 512 and 1024 positions, combined
    with routing layers).  Readings: the window counts the position itself
    (window 1 returns V); the raw rows with the given scale, as in a5.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n = q.shape[0]
    t = np.arange(n)
    logits = scale * (q @ k.T)
    visible = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - window)
    logits = np.where(visible, logits, -np.inf)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)) @ v


def routing_attention_head_backward(q, v, idx, dO, causal: bool = True, scale=None):
    """Gradients of a5..a6 (shared Q/K) for one (batch, head).

    q, v [n, d]; idx [k, w] the clusters' ascending member lists (routing, a1..a4,
    is held fixed: it is piecewise constant in q, and the centroids learn by the
    k-means step a7, not by gradients -- §2, §4); dO [n, d] the gradient of the
    loss with respect to O.  Returns (dq, dv), each [n, d]; dq collects both the
    query and the key role of every shared row.

    Per cluster, with P = softmax(scale Q_c Q_c^T + causal mask), Y_c = P V_c and
    O = the mean of a position's Y rows (a6): dY_c[i] = dO[p_i] / m_{p_i};
    dV_c = P^T dY_c; dP = dY_c V_c^T; dS = P * (dP - rowsum(dP * P));
    dq[p_i] += scale (dS Q_c)_i (query role) + scale (dS^T Q_c)_i (key role).
    Source: §3 (softmax attention rows), §4 (only same-cluster pairs).
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    n, d = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(d)
    idx = np.asarray(idx)
    m = membership_counts(idx, n)
    dq = np.zeros_like(q)
    dv = np.zeros_like(v)
    for members in idx:
        qc, vc = q[members], v[members]
        _, P = cluster_attention(q, q, v, members, causal, scale, return_probs=True)
        dY = dO[members] / m[members][:, None]
        dVc = P.T @ dY
        dP = dY @ vc.T
        dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
        np.add.at(dq, members, scale * (dS @ qc) + scale * (dS.T @ qc))
        np.add.at(dv, members, dVc)
    return dq, dv


def routing_attention_head_separate(q, k, v, mu, w: int, causal: bool = True, scale=None,
                                    idx_q=None, idx_k=None):
    """Routing with separate queries and keys, for one (batch, head).

    Queries and keys are each normalised (a1), scored against the same
    centroids (a2) and each centroid keeps its w best queries and, separately,
    its w best keys (a3, a4).  Inside cluster c every listed query attends to
    the listed keys at positions not after its own (causal) with softmax
    (a5); a position's output is the mean over the clusters that listed it as
    a query and gave it at least one visible key, zero if none (a6).
    Returns dict(O, idx_q, idx_k).  ``idx_q`` / ``idx_k`` may be given to
    evaluate a5..a6 on externally chosen lists (e.g. another implementation's).

    Source: §4 "Routing attention with clustering" (queries and keys routed to
    the same clusters; only same-cluster query/key pairs attend), §3.
    Reading: a (query, cluster) pair with no visible key carries no output and
    is left out of that position's mean.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(d)
    if idx_q is None:
        idx_q = top_w_per_centroid(centroid_scores(normalise_rows(q), mu), w)
    if idx_k is None:
        idx_k = top_w_per_centroid(centroid_scores(normalise_rows(k), mu), w)
    idx_q, idx_k = np.asarray(idx_q), np.asarray(idx_k)
    acc = np.zeros((n, d))
    cnt = np.zeros(n, dtype=np.int64)
    for c in range(idx_q.shape[0]):
        pq, pk = idx_q[c], idx_k[c]
        logits = scale * (q[pq] @ k[pk].T)
        visible = (pk[None, :] <= pq[:, None]) if causal else np.ones((len(pq), len(pk)), bool)
        logits = np.where(visible, logits, -np.inf)
        has = visible.any(axis=1)
        e = np.exp(logits[has] - logits[has].max(axis=1, keepdims=True))
        Y = (e / e.sum(axis=1, keepdims=True)) @ v[pk]
        np.add.at(acc, pq[has], Y)
        np.add.at(cnt, pq[has], 1)
    O = np.zeros((n, d))
    hit = cnt > 0
    O[hit] = acc[hit] / cnt[hit, None]
    return {"O": O, "idx_q": idx_q, "idx_k": idx_k}
