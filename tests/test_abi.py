"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re

import pytest

from content_sparse_attention_shared_b300 import build as rt_build
from content_sparse_attention_shared_b300 import _binding as bnd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    rt_build.build()
    return bnd.load_library()


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(rt_\w+)\s*\(", text, re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("rt_route_assign", "rt_routing_attention", "rt_centroid_ema",
                     "rt_workspace_bytes", "rt_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in bnd.SIGNATURES, f"{name} has no binding signature"


def test_workspace_bytes(lib):
    ws = bnd.rt_workspace_bytes(1, 8, 8192, 128, 128, 64)
    # scores [BH,k,n] fp32 alone are 32 MiB
    assert ws >= 8 * 128 * 8192 * 4
    assert ws % 256 == 0
    assert bnd.rt_workspace_bytes(1, 8, 8192, 96, 128, 64) == 0      # d unsupported
    assert bnd.rt_workspace_bytes(1, 8, 100, 64, 4, 101) == 0        # w > n


def test_status_strings(lib):
    assert lib.rt_status_string(0) == b"RT_OK"
    assert lib.rt_status_string(3) == b"RT_ERR_WORKSPACE"
    assert lib.rt_kernel_name(2) == b"select_topw"


FAKE = 0x10000  # never dereferenced: every case below fails host validation


def _attn(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=1, B=1, H=1, n=128, d=64, mu=FAKE, kc=2, w=64, causal=1,
             scale=0.0, out=FAKE, idx=None, assign=None, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.rt_routing_attention(a["q"], a["k"], a["v"], a["dt"], a["B"], a["H"], a["n"], a["d"],
                                    a["mu"], a["kc"], a["w"], a["causal"], a["scale"], a["out"],
                                    a["idx"], a["assign"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), bnd.RT_ERR_INVALID_ARG),
    (dict(k=None), bnd.RT_ERR_INVALID_ARG),
    (dict(k=FAKE + 4096, d=96), bnd.RT_ERR_UNSUPPORTED),   # separate keys, bad d
    (dict(k=FAKE + 8), bnd.RT_ERR_INVALID_ARG),             # separate keys, misaligned
    (dict(d=96), bnd.RT_ERR_UNSUPPORTED),
    (dict(w=129), bnd.RT_ERR_INVALID_ARG),                   # w > n
    (dict(w=0), bnd.RT_ERR_INVALID_ARG),
    (dict(causal=2), bnd.RT_ERR_INVALID_ARG),
    (dict(dt=7), bnd.RT_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), bnd.RT_ERR_INVALID_ARG),            # misaligned
    (dict(wsb=100), bnd.RT_ERR_WORKSPACE),
    (dict(ws=None), bnd.RT_ERR_WORKSPACE),
    (dict(ws=FAKE + 16), bnd.RT_ERR_INVALID_ARG),            # workspace not 256-aligned
    (dict(scale=float("nan")), bnd.RT_ERR_INVALID_ARG),
])
def test_host_validation(lib, kw, status):
    assert _attn(lib, **kw) == status
    assert lib.rt_last_error_detail() != b""


def test_ema_validation(lib):
    r = lib.rt_centroid_ema(FAKE, 1, 1, 1, 64, 64, FAKE, FAKE, 4, ctypes.c_float(1.5), FAKE,
                            1 << 30, None)
    assert r == bnd.RT_ERR_INVALID_ARG  # decay outside [0, 1]
    r = lib.rt_centroid_ema(FAKE, 1, 1, 1, 64, 64, FAKE, FAKE, 4, ctypes.c_float(0.5), FAKE, 8,
                            None)
    assert r == bnd.RT_ERR_WORKSPACE


def test_ema_topw_validation(lib):
    def call(qk=FAKE, d=64, n=64, idx=FAKE, w=4, k=4, decay=0.5, wsb=1 << 30):
        return lib.rt_centroid_ema_topw(qk, 1, 1, 1, n, d, idx, w, FAKE, k, ctypes.c_float(decay),
                                        FAKE, wsb, None)
    assert call(decay=1.5) == bnd.RT_ERR_INVALID_ARG
    assert call(idx=None) == bnd.RT_ERR_INVALID_ARG
    assert call(idx=FAKE + 4) == bnd.RT_ERR_INVALID_ARG   # misaligned
    assert call(d=96) == bnd.RT_ERR_UNSUPPORTED
    assert call(w=65) == bnd.RT_ERR_INVALID_ARG           # w > n
    assert call(wsb=8) == bnd.RT_ERR_WORKSPACE
    assert lib.rt_last_error_detail() != b""


def test_local_attention_validation(lib):
    def call(q=FAKE, k=FAKE, dt=1, n=256, d=64, window=64, ws=FAKE, wsb=1 << 20):
        return lib.rt_local_attention(q, k, FAKE, dt, 1, 1, n, d, window, ctypes.c_float(0.0),
                                      FAKE, ws, wsb, None)
    assert call(dt=0) == bnd.RT_ERR_UNSUPPORTED          # fp32 rows
    assert call(window=0) == bnd.RT_ERR_INVALID_ARG
    assert call(k=FAKE + 4096) == bnd.RT_ERR_UNSUPPORTED  # separate keys
    assert call(d=96) == bnd.RT_ERR_UNSUPPORTED
    assert call(q=None, k=None) == bnd.RT_ERR_INVALID_ARG
    assert call(wsb=8) == bnd.RT_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == bnd.RT_ERR_INVALID_ARG   # workspace not 256-aligned
    assert lib.rt_last_error_detail() != b""


def test_separate_validation(lib):
    def call(q=FAKE, k=FAKE + 4096, d=64, w=64, wsb=1 << 30, ws=FAKE):
        return lib.rt_routing_attention_separate(q, k, FAKE, 1, 1, 1, 128, d, FAKE, 2, w, 1,
                                                 ctypes.c_float(0.0), FAKE, None, None, None, ws,
                                                 wsb, None)
    assert call(k=FAKE) == bnd.RT_ERR_INVALID_ARG          # the same tensor: shared QK
    assert call(d=96) == bnd.RT_ERR_UNSUPPORTED
    assert call(w=129) == bnd.RT_ERR_INVALID_ARG
    assert call(wsb=100) == bnd.RT_ERR_WORKSPACE
    assert call(k=FAKE + 4100) == bnd.RT_ERR_INVALID_ARG   # misaligned keys
    assert lib.rt_last_error_detail() != b""


def test_mixed_validation(lib):
    def call(dt=1, H=4, n=256, d=64, n_local=2, window=64, mu=FAKE, kc=4, w=64, causal=1,
             ws=FAKE, wsb=1 << 30, out=FAKE):
        return lib.rt_mixed_attention(FAKE, FAKE, dt, 1, H, n, d, n_local, window, mu, kc, w,
                                      causal, ctypes.c_float(0.0), out, None, None, ws, wsb, None)
    assert call(n_local=5) == bnd.RT_ERR_INVALID_ARG        # more local heads than heads
    assert call(n_local=-1) == bnd.RT_ERR_INVALID_ARG
    assert call(dt=0) == bnd.RT_ERR_UNSUPPORTED             # local heads need bf16
    assert call(window=0) == bnd.RT_ERR_INVALID_ARG
    assert call(mu=None) == bnd.RT_ERR_INVALID_ARG          # routing heads need centroids
    assert call(w=300) == bnd.RT_ERR_INVALID_ARG            # w > n (routing half)
    assert call(d=96) == bnd.RT_ERR_UNSUPPORTED
    assert call(causal=3) == bnd.RT_ERR_INVALID_ARG
    assert call(out=FAKE + 8) == bnd.RT_ERR_INVALID_ARG
    assert call(wsb=512) == bnd.RT_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == bnd.RT_ERR_INVALID_ARG
    assert lib.rt_last_error_detail() != b""


def test_step_validation(lib):
    def call(decay=0.5, kc=4, w=64, mu=FAKE, wsb=1 << 30):
        return lib.rt_routing_attention_step(FAKE, FAKE, 1, 1, 1, 128, 64, mu, kc, w, 1,
                                             ctypes.c_float(0.0), ctypes.c_float(decay), FAKE,
                                             None, None, FAKE, wsb, None)
    assert call(decay=1.5) == bnd.RT_ERR_INVALID_ARG
    assert call(mu=None) == bnd.RT_ERR_INVALID_ARG
    assert call(kc=5000) == bnd.RT_ERR_UNSUPPORTED
    assert call(w=129) == bnd.RT_ERR_INVALID_ARG
    assert call(wsb=100) == bnd.RT_ERR_WORKSPACE
    assert lib.rt_last_error_detail() != b""


def test_route_validation(lib):
    r = lib.rt_route_assign(FAKE, 1, 1, 1, 64, 64, FAKE, 4, 16, None, None, None, FAKE, 1 << 30,
                            None)
    assert r == bnd.RT_ERR_INVALID_ARG  # idx output missing


def test_no_cpu_fallback_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    q = torch.zeros(1, 1, 64, 64)
    with pytest.raises(Exception):
        bnd.rt_routing_attention(q, q, q, torch.zeros(1, 2, 64), 32)
