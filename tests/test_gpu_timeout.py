"""The device-side timeout path, exercised without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded; when one runs out
the kernel sets the device status word, gives back what it holds and returns.
The later kernels of the call still run on what they find (every index they
follow is bounds-checked), so the call's outputs are undefined but no access
leaves its buffer.  This test makes a wait run out on purpose with the
library's test aid (rt_debug_inject_wait_timeout): the selected kernels begin
with a bounded wait (1 ms) on a barrier that nothing arrives on, before they
issue any copy or tensor-core operation, so nothing is in flight when they
give up.  It then checks that the call returned, that rt_check_device_status
reports RT_ERR_TIMEOUT (and clears the word; it stays set until then), and
that the next call is correct again.
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
    if kernels == bnd.RT_DEBUG_ATTENTION:
        assert torch.equal(idx, ref_idx)  # routing ran before the attention gave up
    # the next call computes the same result as before the failure
    out2 = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(out2, ref)


def test_status_word_stays_set_until_checked():
    # calls after a failure, before the check, return normally; the word stays
    # set, and every later call's result is right again once it is cleared
    wl = make_random(1, 2, 1000, 128, 8, 100, dtype="bf16", seed=3)
    q, v, mu = ph.to_device(wl)
    ws = rt.Workspace.for_shape(wl.B, wl.H, wl.n, wl.d, wl.k, wl.w, q.dtype)
    ref = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws).clone()
    rt.rt_debug_inject_wait_timeout(bnd.RT_DEBUG_SCORE, LIMIT_NS)
    try:
        rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    finally:
        rt.rt_debug_inject_wait_timeout(0, 0)
    out = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)  # this call itself ran normally
    _expect_timeout(ws)           # ... but the earlier failure is still reported
    out = rt.rt_routing_attention(q, q, v, mu, wl.w, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(out, ref)


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
