"""GPU-vs-oracle parity through the C ABI (needs a B300).

Every case draws seeded inputs, runs the CUDA library, and compares with the
fp64 oracle element by element (tolerances in tests/parity_helpers.py).  The
five measured configurations run at their full sizes, in the same launch
configuration the benchmark times; the sweep adds ragged and degenerate
shapes (n=1, odd w, w=1, w=n, k*w != n, non-causal, several sequences).
"""

import math

import numpy as np
import pytest
import torch

import oracle.routing_oracle as orc
from tests import parity_helpers as ph
from workloads import CONFIG_ORDER, make_random, make_workload

pytestmark = pytest.mark.gpu

rt = pytest.importorskip("content_sparse_attention_shared_b300")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from content_sparse_attention_shared_b300 import build
    build.build()


def run_gpu(wl, causal=True, scale=0.0):
    q, v, mu = ph.to_device(wl)
    B, H, n, d, k, w = wl.B, wl.H, wl.n, wl.d, wl.k, wl.w
    ws = rt.Workspace.for_shape(B, H, n, d, k, w, q.dtype)
    idx = torch.empty((B, H, k, w), dtype=torch.int32, device="cuda")
    a = torch.empty((B, H, n), dtype=torch.int32, device="cuda")
    out = rt.rt_routing_attention(q, q, v, mu, w, causal=causal, scale=scale, idx_out=idx,
                                  assign_out=a, workspace=ws)
    idx2, a2, S = rt.rt_route_assign(q, mu, w, want_scores=True, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    return dict(q=q, v=v, mu=mu, ws=ws, out=out, idx=idx.cpu().numpy(), a=a.cpu().numpy(),
                idx2=idx2.cpu().numpy(), a2=a2.cpu().numpy(), S=S.cpu().numpy())


def check_forward(wl, res, causal=True, scale=None):
    q64 = wl.q_f32().astype(np.float64)
    v64 = wl.v_f32().astype(np.float64)
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(wl.d)
    out = ph.out_to_f64(res["out"])
    assert np.array_equal(res["idx"], res["idx2"]), "route_assign and the forward disagree"
    assert np.array_equal(res["a"], res["a2"])
    worst = 0.0
    for b in range(wl.B):
        for h in range(wl.H):
            S64 = ph.oracle_scores(q64[b, h], wl.centroids[h])
            gS = res["S"][b, h]
            assert np.max(np.abs(gS - S64)) < ph.TOL_SCORE
            ph.check_self_consistent(res["idx"][b, h], res["a"][b, h], gS, wl.w)
            ph.check_index_lists(res["idx"][b, h], S64, wl.w, wl.n)
            ph.check_assign(res["a"][b, h], S64)
            want = ph.oracle_output_on(q64[b, h], v64[b, h], res["idx"][b, h], causal, scale)
            err = np.max(np.abs(out[b, h] - want))
            worst = max(worst, err)
            m = orc.membership_counts(res["idx"][b, h], wl.n)
            assert np.all(out[b, h][m == 0] == 0.0), "uncovered rows must be exactly zero"
    assert worst <= ph.TOL_OUT[wl.dtype], f"max abs error {worst:.3g}"
    return worst


def check_ema(wl, res, decay):
    mu_gpu = res["mu"].clone()
    a_t = torch.from_numpy(res["a"]).cuda()
    rt.rt_centroid_ema(res["q"], a_t, mu_gpu, decay, workspace=res["ws"])
    torch.cuda.synchronize()
    want = orc.centroid_ema(wl.q_f32().astype(np.float64), res["a"], wl.centroids, decay)
    got = mu_gpu.cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - want))
    assert err <= ph.TOL_EMA, f"centroid update error {err:.3g}"
    # centroids nobody chose stay bit-exact
    for h in range(wl.H):
        counts = np.bincount(res["a"][:, h].reshape(-1), minlength=wl.k)
        for c in np.nonzero(counts == 0)[0]:
            assert np.array_equal(got[h, c], wl.centroids[h, c].astype(np.float64))


def check_ema_topw(wl, res, decay):
    """The top-w centroid step on the GPU's own index lists vs the oracle."""
    mu_gpu = res["mu"].clone()
    idx_t = torch.from_numpy(res["idx"]).cuda()
    rt.rt_centroid_ema_topw(res["q"], idx_t, mu_gpu, decay, workspace=res["ws"])
    torch.cuda.synchronize()
    want = orc.centroid_ema_topw(wl.q_f32().astype(np.float64), res["idx"], wl.centroids, decay)
    got = mu_gpu.cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - want))
    assert err <= ph.TOL_EMA, f"top-w centroid update error {err:.3g}"


# ---------------------------------------------------------------------------
# the five measured configurations, full size
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def cfg_results():
    return {}


@pytest.mark.parametrize("cid", CONFIG_ORDER)
def test_config_full_size(cid, cfg_results):
    wl = make_workload(cid)
    res = run_gpu(wl)
    check_forward(wl, res)
    check_ema(wl, res, wl.decay)
    check_ema(wl, res, 0.0)


def test_hand_worked_example(hand_worked):
    from tests.conftest import eval_tree
    g = hand_worked
    for dt in (torch.float32, torch.bfloat16):
        # d=4 is below the supported head dimension: embed in d=64 with zeros
        # appended (zero-mean rows stay zero-mean; dot products unchanged).
        d = 64
        q = np.zeros((1, 1, 4, d)); q[0, 0, :, :4] = g["q"]
        v = np.zeros((1, 1, 4, d)); v[0, 0, :, :4] = g["v"]
        mu = np.zeros((1, 2, d)); mu[0, :, :4] = eval_tree(g["centroids"])
        qt = torch.tensor(q, dtype=dt, device="cuda")
        vt = torch.tensor(v, dtype=dt, device="cuda")
        mt = torch.tensor(mu, dtype=torch.float32, device="cuda")
        idx = torch.empty((1, 1, 2, 2), dtype=torch.int32, device="cuda")
        a = torch.empty((1, 1, 4), dtype=torch.int32, device="cuda")
        scale = eval_tree(g["scale"])
        for causal, key in ((True, "O_causal"), (False, "O_noncausal")):
            out = rt.rt_routing_attention(qt, qt, vt, mt, 2, causal=causal, scale=scale,
                                          idx_out=idx, assign_out=a)
            torch.cuda.synchronize()
            assert idx.cpu().numpy()[0, 0].tolist() == g["expected"]["idx"]
            assert a.cpu().numpy()[0, 0].tolist() == g["expected"]["assign"]
            got = out.float().cpu().numpy()[0, 0, :, :4]
            tol = 1e-5 if dt == torch.float32 else 2e-2
            np.testing.assert_allclose(got, np.array(g["expected"][key], float), atol=tol)
            assert np.all(out.float().cpu().numpy()[0, 0, :, 4:] == 0)
        for decay, key in ((0.0, "centroids_decay0"), (0.5, "centroids_decay_half")):
            m2 = mt.clone()
            rt.rt_centroid_ema(qt, a, m2, decay)
            torch.cuda.synchronize()
            np.testing.assert_allclose(m2.cpu().numpy()[0, :, :4],
                                       np.array(eval_tree(g["expected"][key])), atol=1e-6)


# ---------------------------------------------------------------------------
# shape sweep: ragged, degenerate and extreme cases
# ---------------------------------------------------------------------------

SWEEP = [
    # B, H, n, d, k, w, dtype, causal
    (1, 1, 1, 64, 1, 1, "bf16", True),
    (1, 1, 7, 64, 3, 5, "f32", True),
    (1, 2, 100, 64, 7, 13, "bf16", True),
    (2, 1, 300, 128, 5, 61, "bf16", True),
    (1, 1, 300, 128, 1, 300, "bf16", True),     # one cluster = full causal attention
    (1, 1, 257, 64, 4, 257, "f32", True),       # every centroid takes everything
    (1, 3, 515, 64, 9, 1, "bf16", True),        # w = 1
    (2, 2, 640, 128, 10, 64, "f32", False),     # non-causal
    (1, 1, 1000, 64, 33, 97, "bf16", True),     # k*w != n, odd w
    (3, 2, 777, 128, 24, 129, "bf16", True),    # w just above a tile
    (1, 1, 2048, 128, 300, 16, "bf16", True),   # k > 256
    (1, 1, 600, 64, 2, 300, "bf16", False),     # several key blocks, non-causal
    (1, 2, 1024, 128, 8, 128, "bf16", False),   # one cluster per tile, non-causal
    (2, 1, 1500, 64, 5, 384, "bf16", True),     # three key blocks, causal
    (1, 2, 700, 64, 5, 200, "bf16", False),     # two row tiles in one CTA, non-causal
    (2, 1, 500, 128, 3, 256, "bf16", True),     # two full row tiles
    (1, 1, 300, 64, 2, 150, "bf16", True),      # two row tiles, d = 64
    (1, 1, 33004, 64, 6, 256, "bf16", True),    # long rows: select from group bins, last group ragged
    (1, 2, 32772, 128, 3, 200, "f32", True),    # the same through the fp32 score kernel
    (1, 1, 32771, 64, 4, 100, "bf16", True),    # long rows with n % 4 != 0: no group bins
    (1, 8, 4096, 64, 64, 64, "f32", True),      # fp32 with enough clusters for 64-row query blocks
    (1, 2, 10004, 64, 7, 200, "bf16", True),    # select rows of 8192 < n <= 16384, ragged segments
    (1, 2, 2000, 128, 200, 16, "bf16", True),   # 128 < k <= 256: column halves, ragged upper half and tile
    (2, 1, 777, 64, 144, 8, "bf16", True),      # the same with d = 64, one 16-column upper half, two sequences
    (1, 8, 16384, 64, 256, 64, "bf16", True),   # k = 256 on rows past 8192 without group bins (134 MB of S)
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "b{}h{}n{}d{}k{}w{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "" if c[7] else "nc"))
def test_sweep(case):
    B, H, n, d, k, w, dt, causal = case
    wl = make_random(B, H, n, d, k, w, dtype=dt, seed=n + k + w,
                     centroid_init="tokens" if k <= n else "random")
    res = run_gpu(wl, causal=causal)
    check_forward(wl, res, causal=causal)
    check_ema(wl, res, 0.3)


def test_full_attention_matches_sdpa():
    wl = make_random(1, 2, 512, 64, 1, 512, dtype="f32", seed=5)
    res = run_gpu(wl)
    q = res["q"].double()
    ref = torch.nn.functional.scaled_dot_product_attention(q, q, res["v"].double(), is_causal=True)
    assert torch.max(torch.abs(res["out"].double() - ref)).item() < 1e-4


@pytest.mark.parametrize("n,w", [(200, 37), (5000, 300)])
def test_degenerate_ties(n, w):
    # constant rows normalise to zero: every score is 0, so every centroid
    # takes the first w positions and every row goes to centroid 0.  With
    # n = 5000 the equal scores overflow the candidate buffer of the select
    # kernel and its exact radix path runs.
    B, H, d, k = 1, 2, 64, 5
    q = torch.full((B, H, n, d), 0.75, dtype=torch.bfloat16, device="cuda")
    v = torch.randn((B, H, n, d), device="cuda").to(torch.bfloat16)
    mu = torch.nn.functional.normalize(torch.randn(H, k, d, device="cuda"), dim=-1)
    idx = torch.empty((B, H, k, w), dtype=torch.int32, device="cuda")
    a = torch.empty((B, H, n), dtype=torch.int32, device="cuda")
    out = rt.rt_routing_attention(q, q, v, mu, w, idx_out=idx, assign_out=a)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), torch.arange(w, dtype=torch.int32).expand(B, H, k, w))
    assert int(a.abs().sum()) == 0
    assert torch.all(out[:, :, w:] == 0)


def test_value_ones_property_full_size():
    wl = make_workload("c3")
    q, v, mu = ph.to_device(wl)
    ones = torch.ones_like(v)
    idx = torch.empty((wl.B, wl.H, wl.k, wl.w), dtype=torch.int32, device="cuda")
    out = rt.rt_routing_attention(q, q, ones, mu, wl.w, idx_out=idx)
    torch.cuda.synchronize()
    m = torch.zeros((wl.B * wl.H, wl.n), dtype=torch.int32, device="cuda")
    flat = idx.view(wl.B * wl.H, -1).long()
    m.scatter_add_(1, flat, torch.ones_like(flat, dtype=torch.int32))
    want = (m > 0).to(out.dtype).view(wl.B, wl.H, wl.n, 1).expand_as(out)
    assert torch.max(torch.abs(out.float() - want.float())).item() < 1e-2


def test_deterministic_repeat():
    wl = make_workload("c2")
    q, v, mu = ph.to_device(wl)
    ws = rt.Workspace.for_shape(wl.B, wl.H, wl.n, wl.d, wl.k, wl.w)
    o1 = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws).clone()
    o2 = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_bad_arguments_raise_on_gpu():
    q = torch.zeros((1, 1, 64, 96), dtype=torch.bfloat16, device="cuda")
    mu = torch.zeros((1, 4, 96), device="cuda")
    with pytest.raises(rt.RoutingAttentionError):
        rt.rt_routing_attention(q, q, q, mu, 16)
    q = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    mu = torch.zeros((1, 4, 64), device="cuda")
    with pytest.raises(rt.RoutingAttentionError):
        rt.rt_routing_attention(q, q, q, mu, 65)          # w > n
    with pytest.raises(rt.RoutingAttentionError):
        rt.rt_routing_attention_separate(q, q, q, mu, 16)  # keys must differ from queries


# ---------------------------------------------------------------------------
# the centroid step driven by the top-w lists
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    (1, 8, 8192, 128, 128, 64, "bf16"),   # the measured workload's shape
    (2, 2, 640, 64, 10, 64, "f32"),        # several sequences, fp32 rows
    (3, 1, 777, 128, 24, 129, "bf16"),     # odd n and w
], ids=lambda c: "b{}h{}n{}d{}k{}w{}{}".format(*c))
def test_topw_centroid_update(case):
    B, H, n, d, k, w, dt = case
    wl = make_random(B, H, n, d, k, w, dtype=dt, seed=n + 7 * k + w, centroid_init="tokens")
    res = run_gpu(wl)
    check_ema_topw(wl, res, 0.999)
    check_ema_topw(wl, res, 0.0)


def test_topw_centroid_update_skips_invalid_entries():
    # lists padded with -1 and n: those entries are skipped; a list with no
    # valid entry leaves its centroid bit-exact
    B, H, n, d, k, w = 1, 1, 64, 64, 3, 8
    wl = make_random(B, H, n, d, k, w, dtype="bf16", seed=11, centroid_init="tokens")
    q, v, mu = ph.to_device(wl)
    idx = np.full((B, H, k, w), -1, dtype=np.int32)
    idx[0, 0, 0, :4] = [1, 5, 9, 30]
    idx[0, 0, 1, :] = [2, 3, 4, 5, 6, 7, n, n + 5]
    mu_gpu = mu.clone()
    rt.rt_centroid_ema_topw(q, torch.from_numpy(idx).cuda(), mu_gpu, 0.0)
    torch.cuda.synchronize()
    want = orc.centroid_ema_topw(wl.q_f32().astype(np.float64), idx, wl.centroids, 0.0)
    got = mu_gpu.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - want)) <= ph.TOL_EMA
    assert np.array_equal(got[0, 2], wl.centroids[0, 2].astype(np.float64))


# ---------------------------------------------------------------------------
# local (sliding-window) causal attention
# ---------------------------------------------------------------------------

LOCAL_CASES = [
    # B, H, n, d, window
    (1, 2, 1000, 128, 256),
    (2, 1, 777, 64, 100),
    (1, 1, 300, 128, 1000),   # window >= n: full causal attention
    (1, 1, 200, 64, 1),       # window 1: every position returns its own V row
    (1, 1, 513, 128, 129),    # window one past a key block, ragged last tile
]


@pytest.mark.parametrize("case", LOCAL_CASES, ids=lambda c: "b{}h{}n{}d{}win{}".format(*c))
def test_local_attention(case):
    B, H, n, d, W = case
    wl = make_random(B, H, n, d, 1, 1, dtype="bf16", seed=n + W)
    q, v, _ = ph.to_device(wl)
    out = rt.rt_local_attention(q, q, v, W)
    torch.cuda.synchronize()
    q64, v64 = wl.q_f32().astype(np.float64), wl.v_f32().astype(np.float64)
    got = ph.out_to_f64(out)
    for b in range(B):
        for h in range(H):
            want = orc.local_attention(q64[b, h], q64[b, h], v64[b, h], W, 1 / math.sqrt(d))
            assert np.max(np.abs(got[b, h] - want)) <= ph.TOL_OUT["bf16"]
    if W == 1:
        assert torch.equal(out, v)


def test_local_attention_full_size_sampled():
    # the measured shape with the pages' window of 512, checked on blocks of
    # rows: rows t0..t0+63 need only positions t0-511 .. t0+63
    B, H, n, d, W = 1, 8, 8192, 128, 512
    wl = make_random(B, H, n, d, 1, 1, dtype="bf16", seed=5)
    q, v, _ = ph.to_device(wl)
    out = rt.rt_local_attention(q, q, v, W)
    torch.cuda.synchronize()
    q64, v64 = wl.q_f32().astype(np.float64), wl.v_f32().astype(np.float64)
    got = ph.out_to_f64(out)
    for h in range(H):
        for t0 in (0, 448, 4000, n - 64):
            lo = max(0, t0 - W + 1)
            want = orc.local_attention(q64[0, h, lo:t0 + 64], q64[0, h, lo:t0 + 64],
                                       v64[0, h, lo:t0 + 64], W, 1 / math.sqrt(d))[t0 - lo:]
            assert np.max(np.abs(got[0, h, t0:t0 + 64] - want)) <= ph.TOL_OUT["bf16"]


# ---------------------------------------------------------------------------
# the centroid step on assignments given directly (chunking edge cases)
# ---------------------------------------------------------------------------

EMA_CASES = [
    # B, H, n, d, k, dtype, pattern
    (2, 3, 3000, 64, 40, "bf16", "random"),     # several chunks per sequence, ragged tail
    (1, 2, 2500, 128, 1500, "f32", "random"),   # k > 1024: 2048-position chunks, empty centroids
    (3, 1, 5000, 128, 8, "bf16", "one"),        # one centroid takes all 15000 rows
    (1, 1, 1, 64, 3, "bf16", "random"),         # a single row
    (2, 2, 1100, 64, 16, "bf16", "invalid"),    # entries outside [0, k) are skipped
]


@pytest.mark.parametrize("case", EMA_CASES, ids=lambda c: "b{}h{}n{}d{}k{}{}{}".format(*c))
def test_centroid_update_given_assignments(case):
    B, H, n, d, k, dt, pattern = case
    wl = make_random(B, H, n, d, min(k, n), 1, dtype=dt, seed=n + k)
    q, _, _ = ph.to_device(wl)
    rng = np.random.default_rng(n * 7 + k)
    mu0 = rng.standard_normal((H, k, d))
    mu0 = (mu0 / np.linalg.norm(mu0, axis=-1, keepdims=True)).astype(np.float32)
    if pattern == "one":
        a = np.zeros((B, H, n), dtype=np.int32)
    else:
        a = rng.integers(0, k, size=(B, H, n)).astype(np.int32)
    if pattern == "invalid":
        a[rng.random((B, H, n)) < 0.2] = -1
        a[rng.random((B, H, n)) < 0.1] = k + 3
    a_ref = np.where((a >= 0) & (a < k), a, -1)  # the oracle never matches -1
    for decay in (0.0, 0.999):
        mu = torch.from_numpy(mu0).cuda()
        ws = rt.Workspace.for_shape(B, H, n, d, k, 1, q.dtype)
        rt.rt_centroid_ema(q, torch.from_numpy(a).cuda(), mu, decay, workspace=ws)
        torch.cuda.synchronize()
        ws.check()
        want = orc.centroid_ema(wl.q_f32().astype(np.float64), a_ref, mu0, decay)
        got = mu.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got - want)) <= ph.TOL_EMA
        for h in range(H):
            hit = np.zeros(k, bool)
            hit[np.unique(a_ref[:, h][a_ref[:, h] >= 0])] = True
            assert np.array_equal(got[h, ~hit], mu0[h, ~hit].astype(np.float64))


# ---------------------------------------------------------------------------
# the centroid step in halves (per-shard sums, all-reduce, blend)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    (2, 8, 4096, 128, 128, "bf16"),
    (2, 2, 1500, 64, 700, "f32"),
], ids=lambda c: "b{}h{}n{}d{}k{}{}".format(*c))
def test_centroid_sums_and_apply(case):
    from content_sparse_attention_shared_b300 import sharded
    B, H, n, d, k, dt = case
    wl = make_random(B, H, n, d, k, 1, dtype=dt, seed=n + k)
    q, _, mu = ph.to_device(wl)
    a = rt.rt_route_assign(q, mu, 1)[1]
    torch.cuda.synchronize()
    a_np = a.cpu().numpy()
    q64 = wl.q_f32().astype(np.float64)
    # each sequence as a shard: sums against the oracle's
    shard_sums = []
    for b in range(B):
        s = rt.rt_centroid_ema_sums(q[b:b + 1].contiguous(), a[b:b + 1].contiguous(), k)
        torch.cuda.synchronize()
        want = orc.centroid_sums(q64[b:b + 1], a_np[b:b + 1], k)
        got = s.cpu().numpy().astype(np.float64)
        assert np.array_equal(got[..., d], want[..., d])          # counts exact
        cnt = np.maximum(want[..., d:], 1.0)
        assert np.max(np.abs(got[..., :d] - want[..., :d]) / cnt) <= ph.TOL_EMA
        shard_sums.append(s)
    # "all-reduce" of the shards (elementwise sum), then the blend
    for decay in (0.0, 0.999):
        c = mu.clone()
        rt.rt_centroid_ema_apply(shard_sums[0] + shard_sums[1], c, decay)
        torch.cuda.synchronize()
        want = orc.centroid_ema(q64, a_np, wl.centroids, decay)
        assert np.max(np.abs(c.cpu().numpy() - want)) <= ph.TOL_EMA
    # one shard holding the whole batch: the same bits as the one-call step
    c1, c2 = mu.clone(), mu.clone()
    rt.rt_centroid_ema(q, a, c1, 0.999)
    sharded.sharded_centroid_ema(q, a, c2, 0.999)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


# ---------------------------------------------------------------------------
# separate queries and keys
# ---------------------------------------------------------------------------

def _run_separate(q, k, v, mu, w, causal=True):
    B, H, n, d = q.shape
    kc = mu.shape[1]
    iq = torch.empty((B, H, kc, w), dtype=torch.int32, device="cuda")
    ik = torch.empty((B, H, kc, w), dtype=torch.int32, device="cuda")
    ws = rt.Workspace.for_shape(B, H, n, d, kc, w, q.dtype)
    out = rt.rt_routing_attention_separate(q, k, v, mu, w, causal=causal, idx_q_out=iq,
                                           idx_k_out=ik, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    return out, iq.cpu().numpy(), ik.cpu().numpy()


def _check_separate(q64, k64, v64, mu, out, iq, ik, w, causal, dtype):
    B, H, n, d = q64.shape
    got = ph.out_to_f64(out)
    for b in range(B):
        for h in range(H):
            Sq = ph.oracle_scores(q64[b, h], mu[h])
            Sk = ph.oracle_scores(k64[b, h], mu[h])
            ph.check_index_lists(iq[b, h], Sq, w, n)
            ph.check_index_lists(ik[b, h], Sk, w, n)
            want = orc.routing_attention_head_separate(
                q64[b, h], k64[b, h], v64[b, h], mu[h], w, causal=causal,
                idx_q=iq[b, h], idx_k=ik[b, h])["O"]
            assert np.max(np.abs(got[b, h] - want)) <= ph.TOL_OUT[dtype]
            # positions with no membership that sees a key are exactly zero
            assert np.all(got[b, h][np.all(want == 0.0, axis=1)] == 0.0)


SEP_CASES = [
    # B, H, n, d, k, w, dtype, causal
    (1, 8, 4096, 64, 64, 64, "bf16", True),     # the n=4096 configuration's shape
    (1, 8, 8192, 128, 128, 64, "bf16", True),   # the n=8192 configuration's shape
    (2, 2, 777, 128, 24, 129, "bf16", True),    # ragged, two key blocks
    (1, 2, 1000, 64, 9, 300, "bf16", False),    # three key blocks, non-causal
    (1, 2, 300, 64, 5, 61, "f32", True),        # fp32 path
    (2, 1, 200, 128, 4, 33, "f32", False),
]


@pytest.mark.parametrize("case", SEP_CASES, ids=lambda c: "b{}h{}n{}d{}k{}w{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "" if c[7] else "nc"))
def test_separate_qk(case):
    B, H, n, d, k, w, dt, causal = case
    wq = make_random(B, H, n, d, k, w, dtype=dt, seed=n + 3 * k)
    wk = make_random(B, H, n, d, k, w, dtype=dt, seed=n + 3 * k + 1)
    q, v, mu = ph.to_device(wq)
    kk, _, _ = ph.to_device(wk)
    out, iq, ik = _run_separate(q, kk, v, mu, w, causal)
    _check_separate(wq.q_f32().astype(np.float64), wk.q_f32().astype(np.float64),
                    wq.v_f32().astype(np.float64), wq.centroids, out, iq, ik, w, causal, dt)


@pytest.mark.parametrize("w", [8, 40])
def test_separate_qk_queries_without_visible_keys(w):
    # one centroid e: queries score high early, keys score high late.  With
    # w = 8 every listed query (positions 0..7) precedes every listed key
    # (32..39): all rows are zero.  With w = 40 the lists overlap and some
    # queries see keys, others none.
    n, d = 64, 64
    rng = np.random.default_rng(5)
    e = rng.standard_normal(d)
    e -= e.mean()
    e /= np.linalg.norm(e)
    sign = np.where(np.arange(n) < 32, 1.0, -1.0)[:, None]
    q = (sign * e)[None, None]
    k = (-sign * e)[None, None]
    v = rng.standard_normal((1, 1, n, d))
    mu = e[None, None].astype(np.float32)
    for dt, tdt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
        qt = torch.tensor(q, dtype=tdt, device="cuda")
        kt = torch.tensor(k, dtype=tdt, device="cuda")
        vt = torch.tensor(v, dtype=tdt, device="cuda")
        out, iq, ik = _run_separate(qt, kt, vt, torch.tensor(mu, device="cuda"), w)
        q64 = qt.double().cpu().numpy()
        k64 = kt.double().cpu().numpy()
        v64 = vt.double().cpu().numpy()
        _check_separate(q64, k64, v64, mu, out, iq, ik, w, True, dt)
        if w == 8:
            assert iq[0, 0, 0].tolist() == list(range(8))
            assert ik[0, 0, 0].tolist() == list(range(32, 40))
            assert torch.all(out == 0)


def test_separate_qk_with_equal_keys_matches_shared():
    # keys equal to the queries (another tensor): the lists and the output of
    # the shared-QK pass
    wl = make_random(1, 2, 1000, 128, 12, 100, dtype="bf16", seed=9)
    q, v, mu = ph.to_device(wl)
    out, iq, ik = _run_separate(q, q.clone(), v, mu, wl.w)
    idx = torch.empty((1, 2, 12, 100), dtype=torch.int32, device="cuda")
    ref = rt.rt_routing_attention(q, q, v, mu, wl.w, idx_out=idx)
    torch.cuda.synchronize()
    assert np.array_equal(iq, idx.cpu().numpy()) and np.array_equal(ik, iq)
    assert torch.max(torch.abs(out.float() - ref.float())).item() <= 2 * ph.TOL_OUT["bf16"]


# ---------------------------------------------------------------------------
# mixed local and routing heads in one call
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    (2, 4, 1000, 64, 2, 128, 8, 100),      # two sequences, half the heads local
    (1, 8, 8192, 128, 4, 512, 128, 64),    # the n=8192 shape, window 512
    (1, 3, 700, 128, 3, 1024, 4, 50),      # every head local
    (2, 2, 500, 64, 0, 64, 5, 100),        # every head routed
], ids=lambda c: "b{}h{}n{}d{}local{}win{}k{}w{}".format(*c))
def test_mixed_local_and_routing_heads(case):
    B, H, n, d, nl, W, k, w = case
    wl = make_random(B, H, n, d, k, w, dtype="bf16", seed=n + nl + W)
    q, v, mu_all = ph.to_device(wl)
    Hr = H - nl
    mu = mu_all[nl:].contiguous() if Hr > 0 else None
    idx = torch.empty((B, Hr, k, w), dtype=torch.int32, device="cuda") if Hr > 0 else None
    out = rt.rt_mixed_attention(q, v, mu, nl, W, w, idx_out=idx)
    torch.cuda.synchronize()
    q64, v64 = wl.q_f32().astype(np.float64), wl.v_f32().astype(np.float64)
    got = ph.out_to_f64(out)
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        for h in range(H):
            if h < nl:
                # local heads: sampled row blocks at the long shape
                spans = [(0, n)] if n <= 1000 else [(0, 64), (4000, 4064), (n - 64, n)]
                for t0, t1 in spans:
                    lo = max(0, t0 - W + 1)
                    want = orc.local_attention(q64[b, h, lo:t1], q64[b, h, lo:t1],
                                               v64[b, h, lo:t1], W, scale)[t0 - lo:]
                    assert np.max(np.abs(got[b, h, t0:t1] - want)) <= ph.TOL_OUT["bf16"]
            else:
                gidx = idx[b, h - nl].cpu().numpy()
                S64 = ph.oracle_scores(q64[b, h], wl.centroids[h])
                ph.check_index_lists(gidx, S64, w, n)
                want = ph.oracle_output_on(q64[b, h], v64[b, h], gidx, True, scale)
                assert np.max(np.abs(got[b, h] - want)) <= ph.TOL_OUT["bf16"]


# ---------------------------------------------------------------------------
# backward pass (routing held fixed)
# ---------------------------------------------------------------------------

BWD_CASES = [
    # B, H, n, d, k, w, dtype, causal
    (1, 8, 4096, 64, 64, 64, "bf16", True),     # the n=4096 configuration's shape
    (2, 2, 777, 128, 24, 129, "bf16", True),    # three 64-slot blocks, ragged
    (1, 2, 640, 64, 10, 64, "f32", False),      # fp32, non-causal
    (1, 1, 300, 128, 1, 300, "f32", True),      # one cluster: full causal attention
    (1, 2, 515, 64, 9, 1, "bf16", True),        # w = 1
    (1, 1, 256, 128, 6, 200, "bf16", True),     # positions in several clusters
]


def _bwd_tol(ref):
    return 2e-4 * (1.0 + float(np.max(np.abs(ref))))


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "b{}h{}n{}d{}k{}w{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "" if c[7] else "nc"))
def test_backward(case):
    B, H, n, d, k, w, dt, causal = case
    wl = make_random(B, H, n, d, k, w, dtype=dt, seed=n + 5 * k + w)
    q, v, mu = ph.to_device(wl)
    idx = torch.empty((B, H, k, w), dtype=torch.int32, device="cuda")
    rt.rt_routing_attention(q, q, v, mu, w, causal=causal, idx_out=idx)
    g = torch.Generator(device="cpu").manual_seed(n + k)
    dout = torch.randn((B, H, n, d), generator=g, dtype=torch.float32).cuda()
    ws = rt.Workspace.for_shape(B, H, n, d, k, w, q.dtype)
    dq, dv = rt.rt_routing_attention_backward(q, v, idx, dout, causal=causal, workspace=ws)
    dq2, dv2 = rt.rt_routing_attention_backward(q, v, idx, dout, causal=causal, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(dq, dq2) and torch.equal(dv, dv2)  # deterministic
    q64, v64 = wl.q_f32().astype(np.float64), wl.v_f32().astype(np.float64)
    gidx, do64 = idx.cpu().numpy(), dout.cpu().numpy().astype(np.float64)
    gq, gv = dq.cpu().numpy().astype(np.float64), dv.cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(H):
            wq, wv = orc.routing_attention_head_backward(q64[b, h], v64[b, h], gidx[b, h],
                                                         do64[b, h], causal=causal)
            assert np.max(np.abs(gq[b, h] - wq)) <= _bwd_tol(wq)
            assert np.max(np.abs(gv[b, h] - wv)) <= _bwd_tol(wv)
            m = orc.membership_counts(gidx[b, h], n)
            assert np.all(gq[b, h][m == 0] == 0) and np.all(gv[b, h][m == 0] == 0)


def test_backward_full_attention_matches_autograd():
    # one cluster taking every position: the gradient of full causal attention
    n, d = 384, 64
    wl = make_random(1, 1, n, d, 1, n, dtype="f32", seed=12)
    q, v, mu = ph.to_device(wl)
    idx = torch.empty((1, 1, 1, n), dtype=torch.int32, device="cuda")
    rt.rt_routing_attention(q, q, v, mu, n, idx_out=idx)
    dout = torch.randn((1, 1, n, d), device="cuda")
    dq, dv = rt.rt_routing_attention_backward(q, v, idx, dout)
    torch.cuda.synchronize()
    q64 = q.double().cpu().requires_grad_(True)
    v64 = v.double().cpu().requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(q64, q64, v64, is_causal=True)
    o.backward(dout.double().cpu())
    assert torch.max(torch.abs(dq.double().cpu() - q64.grad)).item() <= _bwd_tol(q64.grad.numpy())
    assert torch.max(torch.abs(dv.double().cpu() - v64.grad)).item() <= _bwd_tol(v64.grad.numpy())


# ---------------------------------------------------------------------------
# the training-step call (forward, then the centroid step on a forked stream)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cid", ["c1", "c3", "c5"])
def test_training_step_equals_two_calls(cid):
    wl = make_workload(cid)
    q, v, mu = ph.to_device(wl)
    B, H, n, d, k, w = wl.B, wl.H, wl.n, wl.d, wl.k, wl.w
    ws = rt.Workspace.for_shape(B, H, n, d, k, w, q.dtype)
    idx1 = torch.empty((B, H, k, w), dtype=torch.int32, device="cuda")
    a1 = torch.empty((B, H, n), dtype=torch.int32, device="cuda")
    mu1 = mu.clone()
    out1 = rt.rt_routing_attention(q, q, v, mu1, w, idx_out=idx1, assign_out=a1, workspace=ws)
    rt.rt_centroid_ema(q, a1, mu1, wl.decay, workspace=ws)
    idx2 = torch.empty_like(idx1)
    a2 = torch.empty_like(a1)
    mu2 = mu.clone()
    out2 = rt.rt_routing_attention_step(q, v, mu2, w, wl.decay, idx_out=idx2, assign_out=a2,
                                        workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(out1, out2) and torch.equal(idx1, idx2) and torch.equal(a1, a2)
    assert torch.equal(mu1, mu2)
    # and inside a captured graph, replayed twice (the centroids move each time)
    mu3 = mu.clone()
    out3 = torch.empty_like(out1)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        rt.rt_routing_attention_step(q, v, mu3.clone(), w, wl.decay, out=out3, workspace=ws)
    side.synchronize()
    with torch.cuda.graph(g, stream=side):
        rt.rt_routing_attention_step(q, v, mu3, w, wl.decay, out=out3, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out3, out1) and torch.equal(mu3, mu1)
    g.replay()
    torch.cuda.synchronize()
    mu4 = mu1.clone()
    out4 = rt.rt_routing_attention(q, q, v, mu1, w, assign_out=a1, workspace=ws)
    rt.rt_centroid_ema(q, a1, mu4, wl.decay, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out3, out4) and torch.equal(mu3, mu4)
