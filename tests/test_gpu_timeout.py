"""The device-side timeout path, exercised without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded; when one runs out
the kernel sets the device status word, gives back what it holds and returns,
and every later kernel finds the word set and returns too.  This test makes a
wait run out on purpose with the library's test aid
(rt_debug_inject_wait_timeout): the selected kernels begin with a bounded
wait (1 ms) on a barrier that nothing arrives on, before they issue any copy
or tensor-core operation, so nothing is in flight when they give up.  It then
checks that the call returned, that rt_check_device_status reports
RT_ERR_TIMEOUT (and clears the word), that the outputs of the failed call were
left alone where the fail-stop rule says so, and that the next call is
correct again.
"""

import ctypes

import pytest
import torch

from tests import parity_helpers as ph
from workloads import make_random, make_workload

pytestmark = pytest.mark.gpu

rt = pytest.importorskip("content_sparse_attention_shared_b300")
from content_sparse_attention_shared_b300 import _binding as bnd  # noqa: E402

LIMIT_NS = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from content_sparse_attention_shared_b300 import build
    build.build()


def _expect_timeout(ws):
    with pytest.raises(rt.RoutingAttentionError) as ei:
        ws.check()
    assert ei.value.status == bnd.RT_ERR_TIMEOUT
    ws.check()  # the word was cleared


@pytest.mark.parametrize("kernels", [bnd.RT_DEBUG_SCORE, bnd.RT_DEBUG_ATTENTION],
                         ids=["score", "attention"])
@pytest.mark.parametrize("cid", ["c2", "c5"])
def test_forward_timeout_reported_and_recoverable(kernels, cid):
    wl = make_workload(cid)
    q, v, mu = ph.to_device(wl)
    ws = rt.Workspace.for_shape(wl.B, wl.H, wl.n, wl.d, wl.k, wl.w, q.dtype)
    idx = torch.empty((wl.B, wl.H, wl.k, wl.w), dtype=torch.int32, device="cuda")
    ref = rt.rt_routing_attention(q, q, v, mu, wl.w, idx_out=idx, workspace=ws).clone()
    ref_idx = idx.clone()
    torch.cuda.synchronize()
    ws.check()
    out = torch.full_like(v, 7.0)
    idx.fill_(-5)
    rt.rt_debug_inject_wait_timeout(kernels, LIMIT_NS)
    try:
        rt.rt_routing_attention(q, q, v, mu, wl.w, out=out, idx_out=idx, workspace=ws)
        torch.cuda.synchronize()
    finally:
        rt.rt_debug_inject_wait_timeout(0, 0)
    _expect_timeout(ws)
    if kernels == bnd.RT_DEBUG_SCORE:
        # nothing after the score kernel ran: lists and output untouched
        assert torch.all(idx == -5) and torch.all(out == 7.0)
    else:
        # routing ran; the attention gave up and the scatter did nothing
        assert torch.equal(idx, ref_idx)
    # fail-stop holds until the word is checked: nothing ran in between, and
    # the next call computes the same result as before the failure
    out2 = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(out2, ref)


def test_failed_pass_stops_later_calls_until_checked():
    wl = make_random(1, 2, 1000, 128, 8, 100, dtype="bf16", seed=3)
    q, v, mu = ph.to_device(wl)
    ws = rt.Workspace.for_shape(wl.B, wl.H, wl.n, wl.d, wl.k, wl.w, q.dtype)
    rt.rt_debug_inject_wait_timeout(bnd.RT_DEBUG_SCORE, LIMIT_NS)
    try:
        rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    finally:
        rt.rt_debug_inject_wait_timeout(0, 0)
    # a second call on the same workspace before the check: every kernel
    # finds the word set and writes nothing
    out = torch.full_like(v, 3.0)
    mu2 = mu.clone()
    a = torch.zeros((1, 2, 1000), dtype=torch.int32, device="cuda")
    rt.rt_routing_attention(q, q, v, mu, wl.w, out=out, workspace=ws)
    rt.rt_centroid_ema(q, a, mu2, 0.0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.equal(mu2, mu)
    _expect_timeout(ws)
    rt.rt_routing_attention(q, q, v, mu, wl.w, out=out, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert not torch.all(out == 3.0)


def test_local_attention_timeout():
    wl = make_random(1, 2, 600, 64, 1, 1, dtype="bf16", seed=4)
    q, v, _ = ph.to_device(wl)
    ws = rt.Workspace(256)
    ref = rt.rt_local_attention(q, q, v, 128, workspace=ws).clone()
    out = torch.full_like(v, 7.0)
    rt.rt_debug_inject_wait_timeout(bnd.RT_DEBUG_LOCAL_ATTENTION, LIMIT_NS)
    try:
        rt.rt_local_attention(q, q, v, 128, out=out, workspace=ws)
        torch.cuda.synchronize()
    finally:
        rt.rt_debug_inject_wait_timeout(0, 0)
    _expect_timeout(ws)
    assert torch.all(out == 7.0)
    out2 = rt.rt_local_attention(q, q, v, 128, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(out2, ref)


def test_injection_arguments_checked():
    lib = bnd.load_library()
    assert lib.rt_debug_inject_wait_timeout(8, LIMIT_NS) == bnd.RT_ERR_INVALID_ARG
    assert lib.rt_debug_inject_wait_timeout(1, 0) == bnd.RT_ERR_INVALID_ARG
    assert lib.rt_debug_inject_wait_timeout(1, 2_000_000_000) == bnd.RT_ERR_INVALID_ARG
    assert lib.rt_debug_inject_wait_timeout(0, 0) == 0
