"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here re-types an oracle formula: every expected value is a closed
form worked by hand (tests/golden), a textbook routine (torch's
scaled_dot_product_attention in float64 for full causal attention), brute
force over all subsets, or an invariant of the method.  The mutation tests at
the bottom plant plausible mistakes in the oracle (on the CPU) and check that
some pin fails for each.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle.routing_oracle as orc
from tests.conftest import eval_tree

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _sdpa(q, k, v, causal, scale):
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), is_causal=causal, scale=scale)
    return out[0, 0].numpy()


def _zero_mean_orthonormal(d, m, rng):
    """m orthonormal vectors in the zero-mean subspace of R^d."""
    a = rng.standard_normal((d, m))
    a -= a.mean(axis=0, keepdims=True)
    qmat, _ = np.linalg.qr(a)
    return qmat.T  # [m, d]


# ---------------------------------------------------------------------------
# pin checks (each raises AssertionError on a mismatch)
# ---------------------------------------------------------------------------

def check_golden(g):
    q = np.array(g["q"], dtype=np.float64)
    v = np.array(g["v"], dtype=np.float64)
    mu = np.array(eval_tree(g["centroids"]))
    scale = eval_tree(g["scale"])
    ex = g["expected"]
    res = orc.routing_attention_head(q, q, v, mu, g["w"], causal=True, scale=scale)
    np.testing.assert_allclose(res["S"], np.array(eval_tree(ex["S"])), atol=1e-12)
    assert res["assign"].tolist() == ex["assign"]
    assert res["idx"].tolist() == ex["idx"]
    assert orc.membership_counts(res["idx"], g["n"]).tolist() == ex["membership"]
    np.testing.assert_allclose(res["O"], np.array(ex["O_causal"], dtype=float), atol=1e-12)
    res_nc = orc.routing_attention_head(q, q, v, mu, g["w"], causal=False, scale=scale)
    np.testing.assert_allclose(res_nc["O"], np.array(ex["O_noncausal"], dtype=float), atol=1e-12)
    a = np.array(ex["assign"])[None, None]
    qq = q[None, None]
    np.testing.assert_allclose(orc.centroid_ema(qq, a, mu[None], 0.0)[0],
                               np.array(eval_tree(ex["centroids_decay0"])), atol=1e-12)
    np.testing.assert_allclose(orc.centroid_ema(qq, a, mu[None], 0.5)[0],
                               np.array(eval_tree(ex["centroids_decay_half"])), atol=1e-12)
    np.testing.assert_allclose(orc.centroid_ema(qq, a, mu[None], 1.0)[0], mu, atol=1e-15)


def check_normalise_closed_form():
    rng = np.random.default_rng(11)
    for d in (4, 64, 128):
        basis = _zero_mean_orthonormal(d, 1, rng)[0]
        for offset, s in ((0.0, 1.0), (3.5, 0.25), (-2.0, 7.0)):
            x = offset + s * basis
            np.testing.assert_allclose(orc.normalise_rows(x[None])[0], basis, atol=1e-12)
            np.testing.assert_allclose(orc.normalise_rows(-x[None])[0], -basis, atol=1e-12)
        const = np.full((1, d), 1.25)
        assert np.array_equal(orc.normalise_rows(const), np.zeros((1, d)))


def check_scores_cosine():
    rng = np.random.default_rng(12)
    d = 16
    e = _zero_mean_orthonormal(d, 3, rng)
    thetas = np.array([0.0, 0.3, 1.1, 2.0, math.pi])
    x = 5.0 + 2.0 * (np.cos(thetas)[:, None] * e[0] + np.sin(thetas)[:, None] * e[1])
    mu = np.stack([e[0], e[1], e[2]])
    S = orc.centroid_scores(orc.normalise_rows(x), mu)
    assert S.shape == (3, len(thetas))
    np.testing.assert_allclose(S[0], np.cos(thetas), atol=1e-12)
    np.testing.assert_allclose(S[1], np.sin(thetas), atol=1e-12)
    np.testing.assert_allclose(S[2], 0.0, atol=1e-12)


def check_assign_ties():
    S = np.array([[0.5, 0.2, 0.9], [0.5, 0.7, 0.9], [0.1, 0.7, 0.9]])
    assert orc.kmeans_assign(S).tolist() == [0, 1, 0]


def check_top_w_exhaustive():
    rng = np.random.default_rng(13)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 4))
        S = rng.integers(0, 3, size=(k, n)).astype(float) / 2.0  # many ties
        for w in range(1, n + 1):
            got = orc.top_w_per_centroid(S, w)
            for c in range(k):
                valid = []
                for T in itertools.combinations(range(n), w):
                    Ts = set(T)
                    ok = all((S[c, i] > S[c, j]) or (S[c, i] == S[c, j] and i < j)
                             for i in Ts for j in range(n) if j not in Ts)
                    if ok:
                        valid.append(list(T))
                assert len(valid) == 1
                assert got[c].tolist() == valid[0]


def check_top_w_invariants():
    rng = np.random.default_rng(14)
    for n, k, w in ((50, 5, 10), (37, 3, 37), (64, 8, 1), (100, 7, 13)):
        S = rng.standard_normal((k, n))
        idx = orc.top_w_per_centroid(S, w)
        assert idx.shape == (k, w)
        for c in range(k):
            assert np.all(np.diff(idx[c]) > 0)
            assert idx[c].min() >= 0 and idx[c].max() < n
        assert orc.membership_counts(idx, n).sum() == k * w


def check_full_attention_k1():
    rng = np.random.default_rng(15)
    for n, d, causal in ((33, 8, True), (64, 16, True), (20, 4, False)):
        q = rng.standard_normal((n, d))
        v = rng.standard_normal((n, d))
        mu = orc.normalise_rows(rng.standard_normal((1, d)))
        scale = 1.0 / math.sqrt(d)
        res = orc.routing_attention_head(q, q, v, mu, n, causal=causal, scale=scale)
        assert res["idx"].tolist() == [list(range(n))]
        np.testing.assert_allclose(res["O"], _sdpa(q, q, v, causal, scale), atol=1e-12)
        # default scale is 1/sqrt(d)
        res2 = orc.routing_attention_head(q, q, v, mu, n, causal=causal)
        np.testing.assert_allclose(res2["O"], res["O"], atol=0)


def check_k_copies_average():
    rng = np.random.default_rng(16)
    n, d, kc = 40, 8, 3
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    mu = np.repeat(orc.normalise_rows(rng.standard_normal((1, d))), kc, axis=0)
    res = orc.routing_attention_head(q, q, v, mu, n, causal=True)
    assert orc.membership_counts(res["idx"], n).tolist() == [kc] * n
    np.testing.assert_allclose(res["O"], _sdpa(q, q, v, True, 1 / math.sqrt(d)), atol=1e-12)


def check_rows_sum_to_one():
    rng = np.random.default_rng(17)
    n, d = 30, 8
    q = rng.standard_normal((n, d)) * 3
    members = np.sort(rng.choice(n, size=12, replace=False))
    for causal in (True, False):
        _, P = orc.cluster_attention(q, q, rng.standard_normal((n, d)), members, causal,
                                     0.4, return_probs=True)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(P >= 0)
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
            assert np.all(np.diag(P) > 0)


def check_v_ones_and_coverage():
    rng = np.random.default_rng(18)
    n, d, kc, w = 50, 8, 4, 9
    q = rng.standard_normal((n, d))
    mu = orc.normalise_rows(rng.standard_normal((kc, d)))
    res = orc.routing_attention_head(q, q, np.ones((n, d)), mu, w)
    m = orc.membership_counts(res["idx"], n)
    assert (m == 0).any() and (m > 0).any()
    np.testing.assert_allclose(res["O"], np.broadcast_to(np.where(m[:, None] > 0, 1.0, 0.0), (n, d)), atol=1e-12)
    assert np.all(res["O"][m == 0] == 0.0)


def check_w1_and_first_slot():
    rng = np.random.default_rng(19)
    n, d, kc = 30, 8, 5
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    mu = orc.normalise_rows(rng.standard_normal((kc, d)))
    res = orc.routing_attention_head(q, q, v, mu, 1)
    m = orc.membership_counts(res["idx"], n)
    sel = m > 0
    np.testing.assert_allclose(res["O"][sel], v[sel], atol=1e-12)
    idx = orc.top_w_per_centroid(orc.centroid_scores(orc.normalise_rows(q), mu), 7)
    for c in range(kc):
        Y = orc.cluster_attention(q, q, v, idx[c], True, 0.3)
        np.testing.assert_allclose(Y[0], v[idx[c][0]], atol=1e-12)


def check_ema_special_cases():
    rng = np.random.default_rng(20)
    d, kc = 8, 3
    e = _zero_mean_orthonormal(d, 3, rng)
    mu = np.stack([e[0], e[1], e[2]])
    # two sequences of one head: tokens of centroid 0 are +-rotations around e0
    # in the (e0, e1) plane (mean direction e0); centroid 2 gets no token.
    ang = 0.4
    t_plus = math.cos(ang) * e[0] + math.sin(ang) * e[1]
    t_minus = math.cos(ang) * e[0] - math.sin(ang) * e[1]
    x = np.zeros((2, 1, 3, d))
    x[0, 0, 0] = 3 + 2 * t_plus
    x[1, 0, 0] = -1 + 5 * t_minus
    x[0, 0, 1] = 2 * e[1]
    x[1, 0, 1] = 4 * e[1]
    x[0, 0, 2] = 7 * t_plus
    x[1, 0, 2] = 0.5 * t_minus
    a = np.array([[[0, 1, 0]], [[0, 1, 0]]])
    out0 = orc.centroid_ema(x, a, mu[None], 0.0)[0]
    np.testing.assert_allclose(out0[0], e[0], atol=1e-12)   # mean of +-ang rotations
    np.testing.assert_allclose(out0[1], e[1], atol=1e-12)
    assert np.array_equal(out0[2], mu[2])                    # empty: untouched
    # decay d: unit-norm blend of mu0 = e0 and mean = cos(ang) e0 -> still e0
    np.testing.assert_allclose(orc.centroid_ema(x, a, mu[None], 0.999)[0][0], e[0], atol=1e-12)
    # a centroid between two directions: mu = e2, mean = e0 at decay 1/2 ->
    # (e2/2 + cos(ang) e0 / 2) normalised
    mu2 = np.stack([e[2], e[1], e[0]])
    got = orc.centroid_ema(x, a, mu2[None], 0.5)[0][0]
    want = (e[2] + math.cos(ang) * e[0]) / math.sqrt(1 + math.cos(ang) ** 2)
    np.testing.assert_allclose(got, want, atol=1e-12)
    np.testing.assert_allclose(orc.centroid_ema(x, a, mu[None], 1.0)[0], mu, atol=1e-15)
    out = orc.centroid_ema(x, a, rng.standard_normal((1, kc, d)), 0.3)[0]
    np.testing.assert_allclose(np.linalg.norm(out[:2], axis=1), 1.0, atol=1e-12)


def check_ema_in_halves():
    """centroid_sums / centroid_apply: closed forms on the hand-built batch of
    check_ema_special_cases, additivity over a split of the batch, and the two
    halves together against the one-call step."""
    rng = np.random.default_rng(22)
    d, kc = 8, 3
    e = _zero_mean_orthonormal(d, 3, rng)
    mu = np.stack([e[0], e[1], e[2]])
    ang = 0.4
    t_plus = math.cos(ang) * e[0] + math.sin(ang) * e[1]
    t_minus = math.cos(ang) * e[0] - math.sin(ang) * e[1]
    x = np.zeros((2, 1, 3, d))
    x[0, 0, 0] = 3 + 2 * t_plus       # normalises to t_plus
    x[1, 0, 0] = -1 + 5 * t_minus     # t_minus
    x[0, 0, 1] = 2 * e[1]             # e1
    x[1, 0, 1] = 4 * e[1]             # e1
    x[0, 0, 2] = 7 * t_plus           # t_plus
    x[1, 0, 2] = 0.5 * t_minus        # t_minus
    a = np.array([[[0, 1, 0]], [[0, 1, 0]]])
    s_all = orc.centroid_sums(x, a, kc)
    # centroid 0: 2 t_plus + 2 t_minus = 4 cos(ang) e0 over 4 rows; centroid 1:
    # 2 e1 over 2 rows; centroid 2: nothing
    np.testing.assert_allclose(s_all[0, 0, :d], 4 * math.cos(ang) * e[0], atol=1e-12)
    np.testing.assert_allclose(s_all[0, 1, :d], 2 * e[1], atol=1e-12)
    assert s_all[0, 0, d] == 4 and s_all[0, 1, d] == 2 and s_all[0, 2, d] == 0
    assert np.all(s_all[0, 2, :d] == 0)
    # additive over the two sequences
    s0 = orc.centroid_sums(x[:1], a[:1], kc)
    s1 = orc.centroid_sums(x[1:], a[1:], kc)
    np.testing.assert_allclose(s0 + s1, s_all, atol=1e-12)
    # the blend: decay 0 -> the mean direction; decay 1/2 between e2 and
    # cos(ang) e0 (the mean, not the sum); an empty centroid untouched
    np.testing.assert_allclose(orc.centroid_apply(s_all, mu[None], 0.0)[0][0], e[0], atol=1e-12)
    mu2 = np.stack([e[2], e[1], e[0]])
    got = orc.centroid_apply(s_all, mu2[None], 0.5)[0]
    want = (e[2] + math.cos(ang) * e[0]) / math.sqrt(1 + math.cos(ang) ** 2)
    np.testing.assert_allclose(got[0], want, atol=1e-12)
    assert np.array_equal(got[2], mu2[2])
    # random batches: sums over shards, applied, equal the one-call step
    B, H, n = 4, 2, 9
    xr = rng.standard_normal((B, H, n, d))
    ar = rng.integers(0, kc, size=(B, H, n))
    mur = orc.normalise_rows(rng.standard_normal((H, kc, d)))
    parts = orc.centroid_sums(xr[:1], ar[:1], kc) + orc.centroid_sums(xr[1:], ar[1:], kc)
    np.testing.assert_allclose(orc.centroid_apply(parts, mur, 0.7),
                               orc.centroid_ema(xr, ar, mur, 0.7), atol=1e-12)


def check_ema_topw_special_cases():
    rng = np.random.default_rng(21)
    d, kc = 8, 3
    e = _zero_mean_orthonormal(d, 3, rng)
    mu = np.stack([e[0], e[1], e[2]])
    ang = 0.4
    t_plus = math.cos(ang) * e[0] + math.sin(ang) * e[1]
    t_minus = math.cos(ang) * e[0] - math.sin(ang) * e[1]
    x = np.zeros((2, 1, 3, d))
    x[0, 0, 0] = 3 + 2 * t_plus
    x[1, 0, 0] = -1 + 5 * t_minus
    x[0, 0, 1] = 2 * e[1]
    x[1, 0, 1] = 4 * e[1]
    x[0, 0, 2] = 7 * t_plus
    x[1, 0, 2] = 0.5 * t_minus
    # lists equal to the argmax partition (-1: no entry): the argmax step's
    # closed forms hold -- mean of the +-ang rotations is e0, an empty list
    # leaves its centroid bit-exact
    idx = np.array([[[[0, 2], [1, -1], [-1, -1]]], [[[0, 2], [1, -1], [-1, -1]]]])
    out0 = orc.centroid_ema_topw(x, idx, mu[None], 0.0)[0]
    np.testing.assert_allclose(out0[0], e[0], atol=1e-12)
    np.testing.assert_allclose(out0[1], e[1], atol=1e-12)
    assert np.array_equal(out0[2], mu[2])
    np.testing.assert_allclose(orc.centroid_ema_topw(x, idx, mu[None], 1.0)[0], mu, atol=1e-15)
    # a token listed by two centroids counts for both: centroid 2 lists tokens
    # 0 and 1 of sequence 0 -> normalise(t_plus + e1) at decay 0
    idx2 = idx.copy()
    idx2[0, 0, 2] = [0, 1]
    got = orc.centroid_ema_topw(x, idx2, mu[None], 0.0)[0]
    want = (t_plus + e[1]) / np.linalg.norm(t_plus + e[1])
    np.testing.assert_allclose(got[2], want, atol=1e-12)
    np.testing.assert_allclose(got[0], e[0], atol=1e-12)
    # the argmax step and this one agree when every centroid's list is exactly
    # its argmax class (random rows, w tokens per centroid and sequence)
    B, n, w = 2, 12, 4
    xr = rng.standard_normal((B, 1, n, d))
    a = np.stack([rng.permutation(np.repeat(np.arange(kc), w)) for _ in range(B)])[:, None]
    lists = np.stack([[np.sort(np.nonzero(a[b, 0] == c)[0]) for c in range(kc)]
                      for b in range(B)])[:, None]
    mur = rng.standard_normal((1, kc, d))
    np.testing.assert_allclose(orc.centroid_ema_topw(xr, lists, mur, 0.3),
                               orc.centroid_ema(xr, a, mur, 0.3), atol=1e-12)


def check_local_attention():
    rng = np.random.default_rng(22)
    n, d = 37, 8
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    scale = 1.0 / math.sqrt(d)
    # a window covering the sequence is full causal attention
    np.testing.assert_allclose(orc.local_attention(q, q, v, n, scale),
                               _sdpa(q, q, v, True, scale), atol=1e-12)
    np.testing.assert_allclose(orc.local_attention(q, q, v, 10 * n, scale),
                               _sdpa(q, q, v, True, scale), atol=1e-12)
    # window 1: every position sees itself only
    np.testing.assert_allclose(orc.local_attention(q, q, v, 1, scale), v, atol=1e-15)
    # row t is the last row of causal attention over the window's positions
    # (the pinned cluster step on a cluster of consecutive positions)
    for W in (2, 5, 16):
        got = orc.local_attention(q, q, v, W, scale)
        for t in (0, 1, W - 1, W, n - 1):
            members = np.arange(max(0, t - W + 1), t + 1)
            want = orc.cluster_attention(q, q, v, members, True, scale)[-1]
            np.testing.assert_allclose(got[t], want, atol=1e-12)
    # and SDPA with the band as an explicit mask
    import torch
    W = 6
    tt = torch.arange(n)
    band = (tt[None, :] <= tt[:, None]) & (tt[None, :] > tt[:, None] - W)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(q)[None], torch.from_numpy(v)[None],
        attn_mask=band[None], scale=scale)[0].numpy()
    np.testing.assert_allclose(orc.local_attention(q, q, v, W, scale), ref, atol=1e-12)


def _torch_forward_shared(q, v, idx, causal, scale):
    """a5..a6 written with torch ops (autograd builds the backward)."""
    import torch
    n, d = q.shape
    out = torch.zeros((n, d), dtype=torch.float64)
    counts = torch.zeros(n, dtype=torch.float64)
    for members in idx:
        p = torch.as_tensor(np.asarray(members), dtype=torch.long)
        qc = q[p]
        S = scale * (qc @ qc.T)
        if causal:
            keep = torch.tril(torch.ones_like(S, dtype=torch.bool))
            S = S.masked_fill(~keep, float("-inf"))
        Y = torch.softmax(S, dim=1) @ v[p]
        out = out.index_add(0, p, Y)
        counts = counts.index_add(0, p, torch.ones(len(p), dtype=torch.float64))
    return out / counts.clamp(min=1.0)[:, None]


def check_backward_autograd():
    import torch
    rng = np.random.default_rng(23)
    n, d, kc, w = 24, 6, 3, 10   # k*w > n: some positions sit in several clusters
    for causal in (True, False):
        q = rng.standard_normal((n, d))
        v = rng.standard_normal((n, d))
        mu = orc.normalise_rows(rng.standard_normal((kc, d)))
        dO = rng.standard_normal((n, d))
        scale = 1.0 / math.sqrt(d)
        res = orc.routing_attention_head(q, q, v, mu, w, causal=causal, scale=scale)
        assert orc.membership_counts(res["idx"], n).max() >= 2
        dq, dv = orc.routing_attention_head_backward(q, v, res["idx"], dO, causal, scale)
        qt = torch.tensor(q, requires_grad=True)
        vt = torch.tensor(v, requires_grad=True)
        out = _torch_forward_shared(qt, vt, res["idx"], causal, scale)
        np.testing.assert_allclose(out.detach().numpy(), res["O"], atol=1e-12)
        (out * torch.from_numpy(dO)).sum().backward()
        np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-10)
        np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-10)


def check_backward_finite_difference():
    rng = np.random.default_rng(24)
    n, d, kc, w = 8, 3, 2, 5
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    mu = orc.normalise_rows(rng.standard_normal((kc, d)))
    dO = rng.standard_normal((n, d))
    idx = orc.routing_attention_head(q, q, v, mu, w)["idx"]
    dq, dv = orc.routing_attention_head_backward(q, v, idx, dO)

    def loss(qq, vv):
        return float((orc.routing_attention_head(qq, qq, vv, mu, w, idx=idx)["O"] * dO).sum())

    eps = 1e-6
    for (i, j) in ((0, 0), (3, 1), (n - 1, d - 1)):
        e = np.zeros((n, d))
        e[i, j] = eps
        np.testing.assert_allclose((loss(q + e, v) - loss(q - e, v)) / (2 * eps), dq[i, j],
                                   atol=1e-6)
        np.testing.assert_allclose((loss(q, v + e) - loss(q, v - e)) / (2 * eps), dv[i, j],
                                   atol=1e-6)


def check_separate_routing():
    rng = np.random.default_rng(25)
    n, d, kc, w = 30, 8, 4, 9
    q = rng.standard_normal((n, d))
    kk = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    mu = orc.normalise_rows(rng.standard_normal((kc, d)))
    scale = 1.0 / math.sqrt(d)
    # keys equal to the queries: the shared-QK step
    shared = orc.routing_attention_head(q, q, v, mu, w, causal=True, scale=scale)
    sep = orc.routing_attention_head_separate(q, q, v, mu, w, causal=True, scale=scale)
    np.testing.assert_allclose(sep["O"], shared["O"], atol=1e-12)
    assert np.array_equal(sep["idx_q"], shared["idx"]) and np.array_equal(sep["idx_k"], shared["idx"])
    # one centroid taking every position: full attention with separate keys
    mu1 = orc.normalise_rows(rng.standard_normal((1, d)))
    for causal in (True, False):
        got = orc.routing_attention_head_separate(q, kk, v, mu1, n, causal=causal, scale=scale)["O"]
        np.testing.assert_allclose(got, _sdpa(q, kk, v, causal, scale), atol=1e-12)
    # a query whose cluster's only key comes later sees nothing (causal): zero
    # row; without the mask it returns that key's value row exactly
    e = _zero_mean_orthonormal(d, 2, rng)
    qq = np.stack([e[0], -e[0], e[1], -e[1]])
    kq = np.stack([-e[0], e[1], -e[1], e[0]])
    vv = rng.standard_normal((4, d))
    m1 = e[0][None]
    got = orc.routing_attention_head_separate(qq, kq, vv, m1, 1, causal=True, scale=scale)
    assert got["idx_q"].tolist() == [[0]] and got["idx_k"].tolist() == [[3]]
    assert np.all(got["O"] == 0.0)
    got = orc.routing_attention_head_separate(qq, kq, vv, m1, 1, causal=False, scale=scale)
    np.testing.assert_allclose(got["O"][0], vv[3], atol=1e-15)
    assert np.all(got["O"][1:] == 0.0)


ALL_CHECKS = [
    check_normalise_closed_form, check_scores_cosine, check_assign_ties,
    check_top_w_exhaustive, check_top_w_invariants, check_full_attention_k1,
    check_k_copies_average, check_rows_sum_to_one, check_v_ones_and_coverage,
    check_w1_and_first_slot, check_ema_special_cases, check_ema_topw_special_cases,
    check_ema_in_halves,
    check_local_attention, check_backward_autograd, check_backward_finite_difference,
    check_separate_routing,
]


def test_golden_hand_worked(hand_worked):
    check_golden(hand_worked)


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_batched_entry_matches_heads():
    rng = np.random.default_rng(21)
    B, H, n, d, kc, w = 2, 2, 24, 8, 3, 6
    q = rng.standard_normal((B, H, n, d))
    v = rng.standard_normal((B, H, n, d))
    mu = orc.normalise_rows(rng.standard_normal((H, kc, d)))
    O, idx, a = orc.routing_attention(q, q, v, mu, w)
    for b in range(B):
        for h in range(H):
            r = orc.routing_attention_head(q[b, h], q[b, h], v[b, h], mu[h], w)
            assert np.array_equal(O[b, h], r["O"]) and np.array_equal(idx[b, h], r["idx"])


# ---------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# ---------------------------------------------------------------------------

def _fails(checks, hand_worked):
    for chk in checks:
        try:
            chk(hand_worked) if chk is check_golden else chk()
        except AssertionError:
            return True
    return False


def _mut_no_centering(x):
    x = np.asarray(x, dtype=np.float64)
    nrm = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    return np.where(nrm > 0, x / np.where(nrm > 0, nrm, 1), 0.0)


def _mut_mask_flipped(q, k, v, members, causal, scale, return_probs=False):
    members = np.asarray(members)
    qc, kc, vc = (np.asarray(a, dtype=np.float64)[members] for a in (q, k, v))
    logits = scale * qc @ kc.T
    if causal:
        logits = np.where(members[None, :] >= members[:, None], logits, -np.inf)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    P = e / e.sum(axis=1, keepdims=True)
    return (P @ vc, P) if return_probs else P @ vc


def _mut_no_scale(q, k, v, members, causal, scale, return_probs=False):
    return _ORIG_ATT(q, k, v, members, causal, 1.0, return_probs)


def _mut_ties_high(S, w):
    S = np.asarray(S)
    k, n = S.shape
    out = np.empty((k, w), dtype=np.int64)
    for c in range(k):
        order = np.lexsort((-np.arange(n), -S[c]))
        out[c] = np.sort(order[:w])
    return out


def _mut_sum_scatter(Y, idx, n):
    Y = np.asarray(Y, dtype=np.float64)
    acc = np.zeros((n, Y.shape[-1]))
    np.add.at(acc, np.asarray(idx).reshape(-1), Y.reshape(-1, Y.shape[-1]))
    return acc


def _mut_ema_swapped(qk, assign, mu, decay):
    return _ORIG_EMA(qk, assign, mu, 1.0 - decay)


def _mut_argmax_last(S):
    S = np.asarray(S)
    return (S.shape[0] - 1 - np.argmax(S[::-1], axis=0)).astype(np.int64)


def _mut_scores_transposed(r, mu):
    return np.asarray(r, dtype=np.float64) @ np.asarray(mu, dtype=np.float64).T


_ORIG_ATT = orc.cluster_attention
_ORIG_EMA = orc.centroid_ema
_ORIG_EMA_TOPW = orc.centroid_ema_topw
_ORIG_LOCAL = orc.local_attention
_ORIG_BWD = orc.routing_attention_head_backward
_ORIG_SEP = orc.routing_attention_head_separate


def _mut_backward_no_key_role(q, v, idx, dO, causal=True, scale=None):
    # drops the key-role term of dq: recomputed as the query role alone
    q = np.asarray(q, dtype=np.float64)
    n, d = q.shape
    sc = scale if scale and scale > 0 else 1.0 / np.sqrt(d)
    dq, dv = _ORIG_BWD(q, v, idx, dO, causal, scale)
    m = orc.membership_counts(idx, n)
    dq2 = np.zeros_like(q)
    for members in np.asarray(idx):
        qc, vc = q[members], np.asarray(v, dtype=np.float64)[members]
        _, P = orc.cluster_attention(q, q, v, members, causal, sc, return_probs=True)
        dY = np.asarray(dO, dtype=np.float64)[members] / m[members][:, None]
        dP = dY @ vc.T
        dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
        np.add.at(dq2, members, sc * (dS @ qc))
    return dq2, dv


def _mut_separate_keys_follow_queries(q, k, v, mu, w, causal=True, scale=None):
    # the keys take the queries' member lists instead of their own
    res = _ORIG_SEP(q, k, v, mu, w, causal, scale)
    q64, k64, v64 = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    n, d = q64.shape
    sc = scale if scale and scale > 0 else 1.0 / np.sqrt(d)
    acc = np.zeros((n, d))
    cnt = np.zeros(n, dtype=np.int64)
    for pq in res["idx_q"]:
        logits = sc * (q64[pq] @ k64[pq].T)
        vis = (pq[None, :] <= pq[:, None]) if causal else np.ones((len(pq), len(pq)), bool)
        logits = np.where(vis, logits, -np.inf)
        ex = np.exp(logits - logits.max(axis=1, keepdims=True))
        np.add.at(acc, pq, (ex / ex.sum(axis=1, keepdims=True)) @ v64[pq])
        np.add.at(cnt, pq, 1)
    O = np.zeros((n, d))
    O[cnt > 0] = acc[cnt > 0] / cnt[cnt > 0, None]
    return {"O": O, "idx_q": res["idx_q"], "idx_k": res["idx_q"]}


def _mut_ema_topw_first_sequence(qk, idx, mu, decay):
    qk = np.asarray(qk)
    return _ORIG_EMA_TOPW(qk[:1], np.asarray(idx)[:1], mu, decay)


def _mut_local_window_off_by_one(q, k, v, window, scale):
    return _ORIG_LOCAL(q, k, v, window + 1, scale)


_ORIG_APPLY = orc.centroid_apply
_ORIG_SUMS = orc.centroid_sums


def _mut_apply_sum_not_mean(sums, mu, decay):
    sums = np.array(sums, dtype=np.float64)
    d = sums.shape[-1] - 1
    sums[..., d] = np.where(sums[..., d] > 0, 1.0, 0.0)  # forgets the count
    return _ORIG_APPLY(sums, mu, decay)


def _mut_sums_raw_rows(qk, assign, k):
    qk = np.asarray(qk, dtype=np.float64)
    B, H, n, d = qk.shape
    a = np.asarray(assign)
    out = np.zeros((H, k, d + 1))
    for h in range(H):
        for c in range(k):
            sel = a[:, h].reshape(-1) == c
            out[h, c, :d] = qk[:, h].reshape(-1, d)[sel].sum(axis=0)  # not normalised
            out[h, c, d] = sel.sum()
    return out


MUTANTS = [
    ("normalise_rows", _mut_no_centering),
    ("cluster_attention", _mut_mask_flipped),
    ("cluster_attention", _mut_no_scale),
    ("top_w_per_centroid", _mut_ties_high),
    ("scatter_average", _mut_sum_scatter),
    ("centroid_ema", _mut_ema_swapped),
    ("kmeans_assign", _mut_argmax_last),
    ("centroid_scores", _mut_scores_transposed),
    ("centroid_ema_topw", _mut_ema_topw_first_sequence),
    ("local_attention", _mut_local_window_off_by_one),
    ("routing_attention_head_backward", _mut_backward_no_key_role),
    ("routing_attention_head_separate", _mut_separate_keys_follow_queries),
    ("centroid_apply", _mut_apply_sum_not_mean),
    ("centroid_sums", _mut_sums_raw_rows),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[f"{a}:{b.__name__}" for a, b in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, hand_worked, name, mutant):
    monkeypatch.setattr(orc, name, mutant)
    caught = False
    try:
        caught = _fails([check_golden] + ALL_CHECKS, hand_worked)
    except Exception:
        caught = True  # a shape error is also a caught mistake
    assert caught, f"no pin catches the planted mistake in {name}"
