"""Seeded generators for the routing-attention workloads.

Every workload is drawn with numpy's PCG64 ``default_rng(seed)`` in a fixed
order: mixture centres -> mixture labels -> noise -> (positional drift /
uniform-noise tokens) -> V -> centroid picks.  Token vectors for the mixture
workloads are layer-normalised (zero mean, unit variance over the head
dimension, eps 1e-5, no affine), then stored as bf16 with round-to-nearest-even
from their fp32 values.  Queries double as keys (shared QK).

The value structure follows the workloads the Routing Transformer paper trains
on ("Efficient Content-Based Sparse Attention with Routing Transformers",
§5 Experiments): PG-19 uses sequences of length 8192, ImageNet-64 is a
64x64x3 raster of 12288 positions.  No dataset is read; these synthetic
stand-ins only reproduce shapes and clustered structure.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# ---------------------------------------------------------------------------
# bf16 storage format (round to nearest even from fp32, exact decode)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = (bits + 0x7FFF + lsb) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32, exact."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str  # "f32" or "bf16": storage and arithmetic type of Q/K/V
    B: int
    H: int
    n: int
    d: int
    k: int
    w: int
    causal: bool
    ema: bool  # whether one centroid update follows the forward pass
    decay: float
    q: np.ndarray  # [B,H,n,d]; float32, or uint16 bf16 bits
    v: np.ndarray  # [B,H,n,d]; same storage as q
    centroids: np.ndarray  # [H,k,d] float32, unit norm

    def q_f32(self) -> np.ndarray:
        return self.q if self.dtype == "f32" else bf16_bits_to_f32(self.q)

    def v_f32(self) -> np.ndarray:
        return self.v if self.dtype == "f32" else bf16_bits_to_f32(self.v)

    @property
    def tokens(self) -> int:
        return self.B * self.n

    def nominal_flops(self) -> float:
        """4*k*w^2*d per head: the full w-by-w block for QK^T and PV."""
        return 4.0 * self.k * self.w * self.w * self.d * self.B * self.H


# The five configurations the library is measured on.  Seeds: 0 for the small
# fp32 case, then 1..4 in order.
CONFIGS = {
    "c1": dict(dtype="f32", B=1, H=1, n=256, d=64, k=4, w=64, seed=0, kind="gauss", ema=True),
    "c2": dict(dtype="bf16", B=1, H=8, n=4096, d=64, k=64, w=64, seed=1, kind="mixture",
               centres=32, sigma=0.3, ema=False),
    "c3": dict(dtype="bf16", B=1, H=8, n=8192, d=128, k=128, w=64, seed=2, kind="mixture",
               centres=128, sigma=0.3, ema=True),
    "c4": dict(dtype="bf16", B=2, H=16, n=12288, d=64, k=96, w=128, seed=3, kind="raster",
               centres=64, sigma=0.3, ema=False),
    "c5": dict(dtype="bf16", B=1, H=8, n=65536, d=128, k=256, w=256, seed=4, kind="mixture",
               centres=512, sigma=0.5, noise_frac=0.1, ema=True),
}
CONFIG_ORDER = ["c1", "c2", "c3", "c4", "c5"]


def workload_name(cfg_id: str) -> str:
    c = CONFIGS[cfg_id]
    kind = {
        "gauss": "gauss",
        "mixture": f"mix{c.get('centres', 0)}" + ("noise" if c.get("noise_frac") else ""),
        "raster": "raster64x64x3",
    }[c["kind"]]
    return (f"{kind}_{c['dtype']}_b{c['B']}h{c['H']}_n{c['n']}_d{c['d']}"
            f"_k{c['k']}_w{c['w']}")


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _layer_norm(x: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Input recipe: LN without affine over the last axis, in float64."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    return x32 if dtype == "f32" else f32_to_bf16_bits(x32)


def _raster_drift(rng: np.random.Generator, H: int, n: int, d: int) -> np.ndarray:
    """Smooth positional drift over a 64x64x3 raster, one set of axes per head.

    position t = (row*64 + col)*3 + ch;
    drift(t) = 0.5*(sin(2*pi*row/64) u1 + cos(2*pi*col/64) u2 + (ch/2) u3)
    """
    assert n == 64 * 64 * 3
    u = _unit_rows(rng.standard_normal((H, 3, d)))
    t = np.arange(n)
    ch = t % 3
    pix = t // 3
    row, col = pix // 64, pix % 64
    a = np.sin(2 * np.pi * row / 64.0)
    b = np.cos(2 * np.pi * col / 64.0)
    c = ch / 2.0
    drift = 0.5 * (a[None, :, None] * u[:, None, 0, :]
                   + b[None, :, None] * u[:, None, 1, :]
                   + c[None, :, None] * u[:, None, 2, :])
    return drift  # [H, n, d]


def _mixture_tokens(rng, B, H, n, d, centres, sigma, kind, noise_frac):
    cen = _unit_rows(rng.standard_normal((H, centres, d)))
    labels = rng.integers(0, centres, size=(B, H, n))
    x = rng.standard_normal((B, H, n, d), dtype=np.float32).astype(np.float64) * sigma
    x += cen[np.arange(H)[None, :, None], labels]
    if kind == "raster":
        x += _raster_drift(rng, H, n, d)[None]
    if noise_frac:
        mask = rng.random((B, H, n)) < noise_frac
        cnt = int(mask.sum())
        lim = math.sqrt(3.0)
        x[mask] = rng.uniform(-lim, lim, size=(cnt, d))
    return _layer_norm(x)


def make_workload(cfg_id: str, B: Optional[int] = None, H: Optional[int] = None,
                  n: Optional[int] = None) -> Workload:
    """Draw one of the five configurations (optionally with B/H/n overridden
    for reduced-size parity cases of the same recipe)."""
    c = dict(CONFIGS[cfg_id])
    if B is not None:
        c["B"] = B
    if H is not None:
        c["H"] = H
    if n is not None:
        c["n"] = n
    rng = np.random.default_rng(c["seed"])
    Bc, Hc, nc, d, k = c["B"], c["H"], c["n"], c["d"], c["k"]
    if c["kind"] == "gauss":
        q = rng.standard_normal((Bc, Hc, nc, d), dtype=np.float32)
        v = rng.standard_normal((Bc, Hc, nc, d), dtype=np.float32)
        mu = _unit_rows(rng.standard_normal((Hc, k, d))).astype(np.float32)
        qs, vs = _store(q, c["dtype"]), _store(v, c["dtype"])
    else:
        x = _mixture_tokens(rng, Bc, Hc, nc, d, c["centres"], c["sigma"], c["kind"],
                            c.get("noise_frac", 0.0))
        qs = _store(x, c["dtype"])
        del x
        v = rng.standard_normal((Bc, Hc, nc, d), dtype=np.float32)
        vs = _store(v, c["dtype"])
        del v
        qf = qs if c["dtype"] == "f32" else bf16_bits_to_f32(qs)
        mu = np.empty((Hc, k, d), dtype=np.float32)
        for h in range(Hc):
            picks = rng.choice(nc, size=k, replace=False)
            mu[h] = _unit_rows(qf[0, h, picks]).astype(np.float32)
    name = workload_name(cfg_id)
    if (B, H, n) != (None, None, None):
        name += f"_sub_b{Bc}h{Hc}n{nc}"
    return Workload(name=name, dtype=c["dtype"], B=Bc, H=Hc, n=nc, d=d, k=k, w=c["w"],
                    causal=True, ema=c["ema"], decay=0.999, q=qs, v=vs, centroids=mu)


def make_random(B: int, H: int, n: int, d: int, k: int, w: int, dtype: str = "bf16",
                seed: int = 0, kind: str = "mixture", centres: int = 16,
                sigma: float = 0.3, causal: bool = True, decay: float = 0.999,
                centroid_init: str = "tokens") -> Workload:
    """A free-shape workload for parity sweeps (ragged n, odd w, k*w != n)."""
    rng = np.random.default_rng(seed)
    if kind == "gauss":
        x = rng.standard_normal((B, H, n, d), dtype=np.float32).astype(np.float64)
    else:
        x = _mixture_tokens(rng, B, H, n, d, centres, sigma, "mixture", 0.0)
    qs = _store(x, dtype)
    v = rng.standard_normal((B, H, n, d), dtype=np.float32)
    vs = _store(v, dtype)
    qf = qs if dtype == "f32" else bf16_bits_to_f32(qs)
    if centroid_init == "tokens" and k <= n:
        mu = np.empty((H, k, d), dtype=np.float32)
        for h in range(H):
            picks = rng.choice(n, size=k, replace=False)
            mu[h] = _unit_rows(qf[0, h, picks]).astype(np.float32)
    else:
        mu = _unit_rows(rng.standard_normal((H, k, d))).astype(np.float32)
    return Workload(name=f"random_{kind}_{dtype}_b{B}h{H}_n{n}_d{d}_k{k}_w{w}_s{seed}",
                    dtype=dtype, B=B, H=H, n=n, d=d, k=k, w=w, causal=causal, ema=True,
                    decay=decay, q=qs, v=vs, centroids=mu)
