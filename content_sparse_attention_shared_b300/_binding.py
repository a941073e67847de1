"""Thin Python binding of the routing-attention C ABI (ctypes).

Argument marshalling only: torch supplies device memory and the stream; every
step of the computation runs in the CUDA library.  There is no fallback: if
the library is missing or no GPU is present the calls raise.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librouting_attention.so")

RT_OK, RT_ERR_INVALID_ARG, RT_ERR_UNSUPPORTED, RT_ERR_WORKSPACE, RT_ERR_CUDA, RT_ERR_TIMEOUT = range(6)
RT_F32, RT_BF16 = 0, 1

# name -> (restype, argtypes) for every symbol of include/routing_attention.h
_c_int, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
SIGNATURES = {
    "rt_workspace_bytes": (_c_size, [_c_int] * 6 + [_c_int]),
    "rt_route_assign": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _c_int,
                                 _vp, _vp, _vp, _vp, _c_size, _vp]),
    "rt_routing_attention": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                      _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp, _c_size,
                                      _vp]),
    "rt_routing_attention_step": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                           _c_int, _c_int, _c_int, _c_float, _c_float, _vp, _vp, _vp,
                                           _vp, _c_size, _vp]),
    "rt_routing_attention_separate": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                               _vp, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp,
                                               _vp, _vp, _c_size, _vp]),
    "rt_routing_attention_backward": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                               _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp,
                                               _c_size, _vp]),
    "rt_centroid_ema": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_int,
                                 _c_float, _vp, _c_size, _vp]),
    "rt_centroid_ema_topw": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp,
                                      _c_int, _c_float, _vp, _c_size, _vp]),
    "rt_centroid_ema_sums": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp,
                                      _vp, _c_size, _vp]),
    "rt_centroid_ema_apply": (_c_int, [_vp, _c_int, _c_int, _vp, _c_int, _c_float, _vp]),
    "rt_local_attention": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_float, _vp, _vp, _c_size, _vp]),
    "rt_mixed_attention": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _vp, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp,
                                    _c_size, _vp]),
    "rt_route_assign_noalloc": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int,
                                         _c_int, _vp, _vp, _vp]),
    "rt_workspace_init": (_c_int, [_vp, _c_size, _vp]),
    "rt_check_device_status": (_c_int, [_vp, _c_size, _vp]),
    "rt_debug_inject_wait_timeout": (_c_int, [ctypes.c_uint, ctypes.c_ulonglong]),
    "rt_status_string": (ctypes.c_char_p, [_c_int]),
    "rt_last_error_detail": (ctypes.c_char_p, []),
    "rt_launch_count": (ctypes.c_int64, []),
    "rt_profile_set": (_c_int, [ctypes.POINTER(_vp), _c_int]),
    "rt_profile_kernel_id": (_c_int, [_c_int]),
    "rt_kernel_name": (ctypes.c_char_p, [_c_int]),
}

_lib: Optional[ctypes.CDLL] = None


class RoutingAttentionError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_status_name(status)}: {detail}")


def _status_name(s: int) -> str:
    names = ["RT_OK", "RT_ERR_INVALID_ARG", "RT_ERR_UNSUPPORTED", "RT_ERR_WORKSPACE",
             "RT_ERR_CUDA", "RT_ERR_TIMEOUT"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"routing-attention CUDA library not built ({path} missing); run "
            "python -m content_sparse_attention_shared_b300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != RT_OK:
        detail = load_library().rt_last_error_detail().decode()
        raise RoutingAttentionError(status, detail)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return RT_F32
    if t.dtype == torch.bfloat16:
        return RT_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# C-named entry points
# ---------------------------------------------------------------------------

def rt_workspace_bytes(B: int, H: int, n: int, d: int, k: int, w: int, dtype=torch.bfloat16) -> int:
    code = dtype if isinstance(dtype, int) else (RT_F32 if dtype == torch.float32 else RT_BF16)
    return int(load_library().rt_workspace_bytes(B, H, n, d, k, w, code))


class Workspace:
    """A device scratch buffer sized by rt_workspace_bytes (torch-allocated)."""

    def __init__(self, nbytes: int, device=None, stream=None):
        if nbytes <= 0:
            detail = load_library().rt_last_error_detail().decode() or "invalid shape"
            raise RoutingAttentionError(RT_ERR_INVALID_ARG, "no workspace size: " + detail)
        self.nbytes = int(nbytes)
        # torch's caching allocator returns 512-byte aligned blocks
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check(load_library().rt_workspace_init(self.buf.data_ptr(), self.nbytes, _stream(stream)))

    @classmethod
    def for_shape(cls, B, H, n, d, k, w, dtype=torch.bfloat16, device=None):
        return cls(rt_workspace_bytes(B, H, n, d, k, w, dtype), device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def check(self, stream=None):
        _check(load_library().rt_check_device_status(self.ptr, self.nbytes, _stream(stream)))


def _ws(ws: Optional[Workspace], B, H, n, d, k, w, dtype, device) -> Workspace:
    return ws if ws is not None else Workspace.for_shape(B, H, n, d, k, w, dtype, device)


def rt_route_assign(qk: torch.Tensor, centroids: torch.Tensor, w: int,
                    idx: Optional[torch.Tensor] = None, assign: Optional[torch.Tensor] = None,
                    scores: Optional[torch.Tensor] = None, want_assign: bool = True,
                    want_scores: bool = False, workspace: Optional[Workspace] = None,
                    stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]:
    B, H, n, d = qk.shape
    k = centroids.shape[1]
    dev = qk.device
    if idx is None:
        idx = torch.empty((B, H, k, w), dtype=torch.int32, device=dev)
    if assign is None and want_assign:
        assign = torch.empty((B, H, n), dtype=torch.int32, device=dev)
    if scores is None and want_scores:
        scores = torch.empty((B, H, k, n), dtype=torch.float32, device=dev)
    ws = _ws(workspace, B, H, n, d, k, w, qk.dtype, dev)
    _check(load_library().rt_route_assign(
        _ptr(qk), _dtype_code(qk), B, H, n, d, _ptr(centroids), k, w, _ptr(idx), _ptr(assign),
        _ptr(scores), ws.ptr, ws.nbytes, _stream(stream)))
    return idx, assign, scores


def rt_routing_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         centroids: torch.Tensor, w: int, causal: bool = True, scale: float = 0.0,
                         out: Optional[torch.Tensor] = None, idx_out: Optional[torch.Tensor] = None,
                         assign_out: Optional[torch.Tensor] = None,
                         workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    B, H, n, d = q.shape
    kc = centroids.shape[1]
    if out is None:
        out = torch.empty_like(v)
    ws = _ws(workspace, B, H, n, d, kc, w, q.dtype, q.device)
    _check(load_library().rt_routing_attention(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, H, n, d, _ptr(centroids), kc, w,
        1 if causal else 0, float(scale), _ptr(out), _ptr(idx_out), _ptr(assign_out), ws.ptr,
        ws.nbytes, _stream(stream)))
    return out


def rt_routing_attention_step(q: torch.Tensor, v: torch.Tensor, centroids: torch.Tensor, w: int,
                              decay: float, causal: bool = True, scale: float = 0.0,
                              out: Optional[torch.Tensor] = None,
                              idx_out: Optional[torch.Tensor] = None,
                              assign_out: Optional[torch.Tensor] = None,
                              workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """Forward pass, then the centroid step on the same rows (centroids in place)."""
    B, H, n, d = q.shape
    kc = centroids.shape[1]
    if out is None:
        out = torch.empty_like(v)
    ws = _ws(workspace, B, H, n, d, kc, w, q.dtype, q.device)
    _check(load_library().rt_routing_attention_step(
        _ptr(q), _ptr(v), _dtype_code(q), B, H, n, d, _ptr(centroids), kc, w, 1 if causal else 0,
        float(scale), float(decay), _ptr(out), _ptr(idx_out), _ptr(assign_out), ws.ptr, ws.nbytes,
        _stream(stream)))
    return out


def rt_routing_attention_separate(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                  centroids: torch.Tensor, w: int, causal: bool = True,
                                  scale: float = 0.0, out: Optional[torch.Tensor] = None,
                                  idx_q_out: Optional[torch.Tensor] = None,
                                  idx_k_out: Optional[torch.Tensor] = None,
                                  assign_out: Optional[torch.Tensor] = None,
                                  workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """Routing attention with queries and keys routed separately."""
    B, H, n, d = q.shape
    kc = centroids.shape[1]
    if out is None:
        out = torch.empty_like(v)
    ws = _ws(workspace, B, H, n, d, kc, w, q.dtype, q.device)
    _check(load_library().rt_routing_attention_separate(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, H, n, d, _ptr(centroids), kc, w,
        1 if causal else 0, float(scale), _ptr(out), _ptr(idx_q_out), _ptr(idx_k_out),
        _ptr(assign_out), ws.ptr, ws.nbytes, _stream(stream)))
    return out


def rt_routing_attention_backward(q: torch.Tensor, v: torch.Tensor, idx: torch.Tensor,
                                  dout: torch.Tensor, causal: bool = True, scale: float = 0.0,
                                  dq: Optional[torch.Tensor] = None,
                                  dv: Optional[torch.Tensor] = None,
                                  workspace: Optional[Workspace] = None, stream=None):
    """Gradients (dq, dv), fp32, of the forward with routing held fixed."""
    B, H, n, d = q.shape
    kc, w = idx.shape[2], idx.shape[3]
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    ws = _ws(workspace, B, H, n, d, kc, w, q.dtype, q.device)
    _check(load_library().rt_routing_attention_backward(
        _ptr(q), _ptr(v), _dtype_code(q), B, H, n, d, _ptr(idx), kc, w, 1 if causal else 0,
        float(scale), _ptr(dout), _ptr(dq), _ptr(dv), ws.ptr, ws.nbytes, _stream(stream)))
    return dq, dv


def rt_centroid_ema(qk: torch.Tensor, assign: torch.Tensor, centroids: torch.Tensor, decay: float,
                    workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    B, H, n, d = qk.shape
    k = centroids.shape[1]
    ws = _ws(workspace, B, H, n, d, k, 1, qk.dtype, qk.device)
    _check(load_library().rt_centroid_ema(
        _ptr(qk), _dtype_code(qk), B, H, n, d, _ptr(assign), _ptr(centroids), k, float(decay),
        ws.ptr, ws.nbytes, _stream(stream)))
    return centroids


def rt_centroid_ema_topw(qk: torch.Tensor, idx: torch.Tensor, centroids: torch.Tensor,
                         decay: float, workspace: Optional[Workspace] = None,
                         stream=None) -> torch.Tensor:
    """The centroid step driven by the top-w lists idx [B,H,k,w] (in place)."""
    B, H, n, d = qk.shape
    k, w = centroids.shape[1], idx.shape[-1]
    ws = _ws(workspace, B, H, n, d, k, 1, qk.dtype, qk.device)
    _check(load_library().rt_centroid_ema_topw(
        _ptr(qk), _dtype_code(qk), B, H, n, d, _ptr(idx), w, _ptr(centroids), k, float(decay),
        ws.ptr, ws.nbytes, _stream(stream)))
    return centroids


def rt_centroid_ema_sums(qk: torch.Tensor, assign: torch.Tensor, k: int,
                         sums: Optional[torch.Tensor] = None,
                         workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """This shard's per-centroid sums of normalised rows and counts, [H,k,d+1]."""
    B, H, n, d = qk.shape
    if sums is None:
        sums = torch.empty((H, k, d + 1), dtype=torch.float32, device=qk.device)
    ws = _ws(workspace, B, H, n, d, k, 1, qk.dtype, qk.device)
    _check(load_library().rt_centroid_ema_sums(
        _ptr(qk), _dtype_code(qk), B, H, n, d, _ptr(assign), k, _ptr(sums), ws.ptr, ws.nbytes,
        _stream(stream)))
    return sums


def rt_centroid_ema_apply(sums: torch.Tensor, centroids: torch.Tensor, decay: float,
                          stream=None) -> torch.Tensor:
    """The centroid step from (all-reduced) sums [H,k,d+1], in place."""
    H, k, d = centroids.shape
    _check(load_library().rt_centroid_ema_apply(
        _ptr(sums), H, d, _ptr(centroids), k, float(decay), _stream(stream)))
    return centroids


def rt_local_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int,
                       scale: float = 0.0, out: Optional[torch.Tensor] = None,
                       workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """Local causal attention over the `window` positions ending at each one."""
    B, H, n, d = q.shape
    if out is None:
        out = torch.empty_like(v)
    ws = workspace if workspace is not None else Workspace(256, q.device)
    _check(load_library().rt_local_attention(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, H, n, d, int(window), float(scale),
        _ptr(out), ws.ptr, ws.nbytes, _stream(stream)))
    return out


RT_DEBUG_SCORE, RT_DEBUG_ATTENTION, RT_DEBUG_LOCAL_ATTENTION = 1, 2, 4


def rt_debug_inject_wait_timeout(kernels: int, limit_ns: int) -> None:
    """Test aid: the selected kernels start with a bounded wait that runs out
    (0, 0 turns it off)."""
    _check(load_library().rt_debug_inject_wait_timeout(int(kernels), int(limit_ns)))


def rt_mixed_attention(q: torch.Tensor, v: torch.Tensor, centroids: Optional[torch.Tensor],
                       n_local: int, window: int, w: int, causal: bool = True,
                       scale: float = 0.0, out: Optional[torch.Tensor] = None,
                       idx_out: Optional[torch.Tensor] = None,
                       assign_out: Optional[torch.Tensor] = None,
                       workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """Local attention on heads [0, n_local), routing attention on the rest."""
    B, H, n, d = q.shape
    Hr = H - n_local
    kc = centroids.shape[1] if centroids is not None else 1
    if out is None:
        out = torch.empty_like(v)
    if workspace is None:
        nbytes = rt_workspace_bytes(1, Hr, n, d, kc, w, q.dtype) if Hr > 0 else 256
        workspace = Workspace(nbytes, q.device)
    _check(load_library().rt_mixed_attention(
        _ptr(q), _ptr(v), _dtype_code(q), B, H, n, d, int(n_local), int(window), _ptr(centroids),
        kc, w, 1 if causal else 0, float(scale), _ptr(out), _ptr(idx_out), _ptr(assign_out),
        workspace.ptr, workspace.nbytes, _stream(stream)))
    return out


def rt_launch_count() -> int:
    return int(load_library().rt_launch_count())


def rt_profile_set(events) -> None:
    """events: list of (start, stop) torch.cuda.Event pairs (timing enabled)."""
    lib = load_library()
    flat = []
    for a, b in events:
        for e in (a, b):
            if not e.cuda_event:  # torch creates the handle on first record
                e.record()
        flat += [a.cuda_event, b.cuda_event]
    if events:
        torch.cuda.synchronize()
    arr = (ctypes.c_void_p * max(1, len(flat)))(*flat)
    _check(lib.rt_profile_set(arr, len(events)))


def rt_profile_kernel_name(i: int) -> str:
    lib = load_library()
    return lib.rt_kernel_name(lib.rt_profile_kernel_id(i)).decode()


def rt_route_assign_noalloc(qk: torch.Tensor, centroids: torch.Tensor, w: int, idx: torch.Tensor,
                            assign: Optional[torch.Tensor] = None, stream=None) -> None:
    """Routing with the library's fixed scratch array; outputs are caller-owned
    (no allocation on either side of the call)."""
    B, H, n, d = qk.shape
    k = centroids.shape[1]
    _check(load_library().rt_route_assign_noalloc(
        _ptr(qk), _dtype_code(qk), B, H, n, d, _ptr(centroids), k, w, _ptr(idx), _ptr(assign),
        _stream(stream)))
