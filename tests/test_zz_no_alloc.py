"""rt_route_assign_noalloc: routing for callers that cannot allocate.

Some callers cannot call cudaMalloc where they route (they run inside a host
framework whose device allocator they do not own, or keep a device footprint
fixed at start-up), so they cannot hand rt_route_assign a workspace.  This
entry point takes its score scratch from a fixed array the library owns.  The
test calls it through the C ABI, twice in a row (the array keeps the previous
call's contents), and checks that its index lists and assignments equal those
of rt_route_assign with a caller workspace -- bit-exact, the tolerance every
index test here uses.  The first case's lists are also checked against the
fp64 oracle with the same rule the parity tests use, and after the calls the
entry point's own device status word (read with rt_check_device_status(NULL,
0, stream)) must be clear.  It also checks the size limit.  This file is
collected last so that a failure here cannot hide another test's result.
"""

import ctypes

import numpy as np
import pytest
import torch


from tests import parity_helpers as ph
from workloads import make_random, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from content_sparse_attention_shared_b300 import build, load_library
    build.build()
    return load_library()


def _noalloc(lib, q, mu, w, idx, a):
    B, H, n, d = q.shape
    dt = 1 if q.dtype == torch.bfloat16 else 0
    return lib.rt_route_assign_noalloc(
        ctypes.c_void_p(q.data_ptr()), dt, B, H, n, d, ctypes.c_void_p(mu.data_ptr()),
        mu.shape[1], w, ctypes.c_void_p(idx.data_ptr()),
        ctypes.c_void_p(a.data_ptr()) if a is not None else None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    ("c2", None),                                    # n=4096, k=64, w=64
    ("c3", None),                                    # n=8192, k=128: exactly the array size
    ("ragged", (2, 3, 1000, 128, 33, 97, "bf16")),
    ("f32", (1, 1, 257, 64, 4, 64, "f32")),
]


@pytest.mark.parametrize("name,shape", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_path(lib, name, shape):
    import content_sparse_attention_shared_b300 as rt
    if shape is None:
        wl = make_workload(name)
    else:
        B, H, n, d, k, w, dt = shape
        wl = make_random(B, H, n, d, k, w, dtype=dt, seed=11)
    q, _, mu = ph.to_device(wl)
    idx_ref, a_ref, _ = rt.rt_route_assign(q, mu, wl.w)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row on the shared scratch array
        idx = torch.full((wl.B, wl.H, wl.k, wl.w), -1, dtype=torch.int32, device="cuda")
        a = torch.full((wl.B, wl.H, wl.n), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, q, mu, wl.w, idx, a) == 0, lib.rt_last_error_detail()
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref)
        assert torch.equal(a, a_ref)
    # without the assignment output
    idx = torch.full((wl.B, wl.H, wl.k, wl.w), -1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, q, mu, wl.w, idx, None) == 0
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref)
    # the entry point's own device status word: no wait ran out
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.rt_check_device_status(None, 0, stream) == 0, lib.rt_last_error_detail()
    if name == "c2":
        # and the lists agree with the fp64 oracle (score-gap rule for swaps)
        q64 = wl.q_f32().astype(np.float64)
        got_idx, got_a = idx_ref.cpu().numpy(), a_ref.cpu().numpy()
        for b in range(wl.B):
            for h in range(wl.H):
                S64 = ph.oracle_scores(q64[b, h], wl.centroids[h])
                ph.check_index_lists(got_idx[b, h], S64, wl.w, wl.n)
                ph.check_assign(got_a[b, h], S64)


def test_noalloc_rejects_sizes_beyond_the_array(lib):
    # B*H*k*n above RT_NOALLOC_MAX_SCORES: refused before any launch
    q = torch.zeros((1, 8, 8192, 128), dtype=torch.bfloat16, device="cuda")
    mu = torch.zeros((8, 129, 128), device="cuda")
    idx = torch.zeros((1, 8, 129, 64), dtype=torch.int32, device="cuda")
    st = _noalloc(lib, q, mu, 64, idx, None)
    assert st == 2  # RT_ERR_UNSUPPORTED
    assert b"exceed" in lib.rt_last_error_detail()
    assert torch.all(idx == 0)


def test_noalloc_timeout_reported_on_its_own_status_word(lib):
    # a bounded wait that runs out inside the entry point's score kernel (made
    # to run out with the library's test aid, before the kernel issues any
    # copy) is reported through the entry point's own status word, which
    # rt_check_device_status(NULL, 0, stream) reads and clears; the next call
    # is correct again
    import content_sparse_attention_shared_b300 as rt
    wl = make_workload("c2")
    q, _, mu = ph.to_device(wl)
    idx_ref, a_ref, _ = rt.rt_route_assign(q, mu, wl.w)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    idx = torch.full((wl.B, wl.H, wl.k, wl.w), -1, dtype=torch.int32, device="cuda")
    assert lib.rt_debug_inject_wait_timeout(1, 1_000_000) == 0
    try:
        assert _noalloc(lib, q, mu, wl.w, idx, None) == 0
        torch.cuda.synchronize()
    finally:
        lib.rt_debug_inject_wait_timeout(0, 0)
    assert lib.rt_check_device_status(None, 0, stream) == 5  # RT_ERR_TIMEOUT
    assert lib.rt_check_device_status(None, 0, stream) == 0  # cleared
    a = torch.full((wl.B, wl.H, wl.n), -1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, q, mu, wl.w, idx, a) == 0
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref) and torch.equal(a, a_ref)
