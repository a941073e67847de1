"""Routing-attention benchmark (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c3] [--no-configs] [--no-cpu-baseline] [--sequential-step]

A step is one pass of the whole hot path over one batch of synthetic input:
routing (normalise, score, argmax, top-w per centroid, position sort),
in-cluster causal attention, the averaging scatter and, where the workload
has one, the centroid update.  The headline workload is the n=8192, H=8,
d=128 configuration (mix128_bf16_b1h8_n8192_d128_k128_w64).

ours:       CUDA library; the step is one rt_routing_attention_step call (the
            forward, with the centroid update on a side stream from the end
            of the score kernel; --sequential-step: rt_routing_attention then
            rt_centroid_ema); device time with CUDA events per step (K replays
            of the step captured as one CUDA graph), L2 flushed (256 MiB write)
            before every timed step; e2e = the same step through the public
            API with pinned-host inputs copied in and the output copied out
            inside the timed region (copies in, compute and copies out
            overlapped across consecutive steps, as a serving loop runs them,
            with double-buffered device inputs and outputs); per-kernel times
            from the library's launch hook.  At one GPU the line also carries
            `configs`: the same measurements (fewer steps) on every one of the
            five workloads, each with the oracle timed on one core and on all
            host cores.
reference:  the fp64 CPU oracle on the host cores: every step runs all heads
            of the workload, one head per worker process (spawned, one BLAS
            thread each, as many workers as heads or cores), and is timed as
            a whole.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed-attention tokens/s and TFLOPS (% bf16 peak) at n=8192, H=8, d=128, 1 B300"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max_mhz=d.get("sm_max_mhz", 2032.0), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                sm_max_mhz=2032.0, source="fallback")


# ---------------------------------------------------------------------------
# algorithmic work per launch, by kernel kind (bytes moved that the method
# must move, or flops it must do): rows read and written once, scores written
# and read once, index lists, per-slot output rows.
# ---------------------------------------------------------------------------

def select_uses_group_bins(wl):
    """Whether the score kernel writes group bins and the select reads those
    instead of whole score rows (rows of n >= 32768, n a multiple of 4)."""
    return 32768 <= wl.n <= 262144 and wl.n % 4 == 0


def kernel_work(name, wl):
    s = 2 if wl.dtype == "bf16" else 4
    BH, n, d, k, w = wl.B * wl.H, wl.n, wl.d, wl.k, wl.w
    gbins = BH * k * ((n + 7) // 8) * 2 if select_uses_group_bins(wl) else 0
    if name in ("score_simt", "score_tc"):
        byts = BH * n * d * s + BH * k * n * 4 + BH * n * 4 * 2 + gbins
        return dict(bytes=byts, flops=2.0 * BH * n * k * d)
    if name == "select_topw":
        if gbins:
            # the group bins, the w groups (8 scores each) that must be read
            # again at least, index lists and membership counts
            return dict(bytes=gbins + BH * k * w * 8 * 4 + BH * k * w * 4 * 2, flops=0.0)
        return dict(bytes=BH * k * n * 4 + BH * k * w * 4 * 2, flops=0.0)
    if name in ("attention_simt", "attention_tc"):
        # gathered Q(=K) and V rows, per-slot output rows, index lists
        byts = 2 * BH * k * w * d * s + BH * k * w * d * s + BH * k * w * 4
        return dict(bytes=byts, flops=4.0 * BH * k * w * w * d)
    if name == "scatter_average":
        return dict(bytes=BH * n * 4 + BH * n * d * s, flops=0.0)
    if name == "ema_bucket":
        # the assignments, read once (the row ids it writes are scratch)
        return dict(bytes=BH * n * 4, flops=0.0)
    if name == "ema_update":
        # rows read once, centroids read and written
        return dict(bytes=BH * n * d * s + wl.H * k * d * 8, flops=3.0 * BH * n * d)
    if name == "centroid_prep":
        kpad = (k + 15) // 16 * 16
        return dict(bytes=wl.H * k * d * 4 + wl.H * (3 * kpad * d * 2 + kpad * 4), flops=0.0)
    return dict(bytes=0, flops=0.0)


LOCAL_WINDOW = 512  # the pages' local-attention window (§6 "Local vs Global")


def local_attention_flops(BH, n, d, window):
    """Useful flops of causal local attention: QK^T and PV over the
    min(t + 1, window) keys of every position t (2 d each, twice)."""
    W = min(window, n)
    keys = W * (W + 1) // 2 + (n - W) * W  # sum over t of min(t + 1, W)
    return 4.0 * d * keys * BH


def local_attention_timing(wl, q, v, flush, stream, steps):
    """Device time of the companion layer, rt_local_attention (shared QK,
    causal window of LOCAL_WINDOW positions), on the workload's own rows: CUDA
    events around each call on the launching stream, L2 flushed before each."""
    import torch
    import content_sparse_attention_shared_b300 as rt

    if wl.dtype != "bf16" or wl.d not in (64, 128):
        return None
    W = min(LOCAL_WINDOW, wl.n)
    out = torch.empty_like(v)
    ws = rt.Workspace(256, q.device)
    for _ in range(3):
        rt.rt_local_attention(q, q, v, W, out=out, workspace=ws)
    torch.cuda.synchronize()
    reps = max(10, min(steps, 50))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i in range(reps):
        flush.zero_()
        ev[i][0].record(stream)
        rt.rt_local_attention(q, q, v, W, out=out, workspace=ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ws.check()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flops = local_attention_flops(wl.B * wl.H, wl.n, wl.d, W)
    return {"window": W, "ms": ms, "tokens_per_s": wl.tokens / (ms * 1e-3),
            "tflops": flops / (ms * 1e-3) / 1e12,
            "timing": "CUDA events around each call, L2 flushed before each (256 MiB write)"}


def alu_peak_tflops(sm_mhz):
    # fp32 FMA: 148 SMs x 128 lanes x 2 flop per cycle
    return 148 * 128 * 2 * sm_mhz * 1e6 / 1e12


KERNEL_BOUND = {
    "score_simt": "alu", "attention_simt": "alu", "score_tc": "hbm", "attention_tc": "hbm",
    "select_topw": "hbm", "scatter_average": "hbm", "ema_update": "hbm",
    "ema_bucket": "hbm", "centroid_prep": "hbm",
}

KERNEL_SOURCES = {
    "score_simt": ["k_score_simt.cu"], "score_tc": ["k_score_tc.cu", "tc_ptx.cuh"],
    "centroid_prep": ["k_score_tc.cu"], "select_topw": ["k_select.cu"],
    "attention_simt": ["k_attention_simt.cu"],
    "attention_tc": ["k_attention_tc.cu", "k_attention_pipe.cu", "k_attention_pair.cu",
                     "attn_common.cuh", "tc_ptx.cuh"],
    "scatter_average": ["k_scatter.cu"], "ema_update": ["k_ema.cu"], "ema_bucket": ["k_ema.cu"],
}


def kernel_source_hash(name):
    """Hash of the source files a kernel kind is built from (so a stored ncu
    traffic figure is only used while those sources are unchanged)."""
    files = KERNEL_SOURCES.get(name)
    if not files:
        return None
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, "content_sparse_attention_shared_b300", "csrc", f)
        if not os.path.isfile(p):
            return None
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(name, wl_name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    e = rec.get(name)
    if not e or e.get("source_sha") != kernel_source_hash(name):
        return None
    if e.get("workload") != wl_name:
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock, power and clock-event reasons while the timed region
    runs: NVML from a polling thread (every ~2 ms, so even a region of a few
    tens of milliseconds gets samples), else ``nvidia-smi -lms``.  Read-only:
    nothing about the GPU's settings is changed."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, pci_bus_id=None):
        self.dev = device_index
        self.pci = pci_bus_id
        self.rows = []
        self.source = None
        self._stop = None
        self._thread = None
        self.proc = None
        self.path = None
        self.nvml_error = None

    class _Nvml:
        """Minimal read-only NVML access through ctypes (libnvidia-ml ships with
        the driver; no Python package needed)."""
        CLOCK_SM = 1
        REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

        def __init__(self, index, pci):
            import ctypes
            self.ct = ctypes
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            self.h = ctypes.c_void_p()
            rc = 1
            if pci:
                rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index),
                                                            ctypes.byref(self.h))
            if rc != 0:
                raise RuntimeError(f"no NVML handle (rc {rc})")
            fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

        def _u32(self, fn, *args):
            v = self.ct.c_uint()
            if fn(self.h, *args, self.ct.byref(v)) != 0:
                raise RuntimeError("NVML query failed")
            return v.value

        def sample(self):
            sm = self._u32(self.lib.nvmlDeviceGetClockInfo, self.CLOCK_SM)
            smax = self._u32(self.lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM)
            pw = self._u32(self.lib.nvmlDeviceGetPowerUsage) / 1000.0
            r = self.ct.c_ulonglong()
            if self.reasons_fn(self.h, self.ct.byref(r)) != 0:
                raise RuntimeError("NVML query failed")
            return dict(sm=float(sm), smax=float(smax), power=pw,
                        reasons=[k for k, b in self.REASONS.items() if r.value & b])

    def _poll(self, nv):
        while not self._stop.is_set():
            try:
                self.rows.append(nv.sample())
            except RuntimeError:
                break
            time.sleep(0.002)

    def __enter__(self):
        import threading
        try:
            nv = self._Nvml(self.dev, self.pci)
            nv.sample()
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, args=(nv,), daemon=True)
            self._thread.start()
            self.source = "nvml"
            return self
        except Exception as e:  # no NVML: fall back to nvidia-smi
            self._thread = None
            self.nvml_error = f"{type(e).__name__}: {e}"[:120]
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._read_smi()

    def _read_smi(self):
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                         "sw_power_cap")
                self.rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                      power=float(parts[3]),
                                      reasons=[nm for nm, v in zip(names, parts[5:9])
                                               if v.lower() == "active"]))
            except ValueError:
                continue
        os.unlink(self.path)

    def summary(self):
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "source": self.source}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = sorted({nm for r in rows for nm in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows), "source": self.source,
                **({"nvml_error": self.nvml_error} if self.nvml_error else {})}


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
_WORKER = {}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or "unknown"


def _oracle_worker_init(wl_id):
    """Spawned worker: one BLAS thread, its own copy of the workload (drawn
    from the same seed, so nothing large crosses the process boundary)."""
    os.environ.update(ONE_THREAD_ENV)
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from workloads import make_workload
    _WORKER["wl"] = make_workload(wl_id)


def _oracle_head(h):
    """The oracle's step on head h: a1..a6 on every sequence of the head, then
    a7 on the head's centroids (when the workload has it).  Returns the
    seconds spent in the oracle (input decoding excluded)."""
    import numpy as np

    import oracle.routing_oracle as orc

    wl = _WORKER["wl"]
    q64 = wl.q_f32()[:, h:h + 1].astype(np.float64)
    v64 = wl.v_f32()[:, h:h + 1].astype(np.float64)
    mu = wl.centroids[h:h + 1]
    t0 = time.perf_counter()
    _, _, a = orc.routing_attention(q64, q64, v64, mu, wl.w, causal=True)
    if wl.ema:
        orc.centroid_ema(q64, a, mu, wl.decay)
    return time.perf_counter() - t0


class OraclePool:
    """Spawned worker processes running the oracle head by head.  Spawned, not
    forked: the parent may hold a CUDA context."""

    def __init__(self, wl_id, workers):
        self.workers = workers
        self.pool = mp.get_context("spawn").Pool(workers, initializer=_oracle_worker_init,
                                                 initargs=(wl_id,))

    def one_head(self, h=0):
        return self.pool.apply(_oracle_head, (h,))

    def step(self, H):
        """Wall time of one whole step: every head, one per worker at a time."""
        t0 = time.perf_counter()
        self.pool.map(_oracle_head, range(H), chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_baseline(wl_id, wl):
    """The oracle as it stands on this host: one head on one core (scaled to
    the step by the head count), and one whole step with the heads spread over
    min(H, cores) worker processes."""
    nproc = os.cpu_count() or 1
    workers = max(1, min(wl.H, nproc))
    pool = OraclePool(wl_id, workers)
    try:
        one = pool.one_head(0)
        allc = pool.step(wl.H)
    finally:
        pool.close()
    one_step = one * wl.H
    return {
        "value": wl.tokens / allc, "unit": UNIT, "cores": workers, "kind": "oracle",
        "sample": f"one whole step of {wl.name} (every head; forward"
                  f"{' + centroid update' if wl.ema else ''}), fp64 numpy oracle, heads spread "
                  f"over {workers} spawned worker processes with one BLAS thread each; "
                  f"{allc:.2f} s for the step",
        "single_core": {"value": wl.tokens / one_step, "unit": UNIT, "cores": 1,
                        "sample": f"head 0 alone on one thread ({one:.2f} s) x {wl.H} heads"},
        "nproc": nproc, "cpu_model": cpu_model(),
    }


def base_config(wl):
    """The `config` object both arms print (same keys)."""
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "n": wl.n, "d": wl.d, "k": wl.k,
            "w": wl.w, "causal": True,
            "step": "forward + centroid update" if wl.ema else "forward"}


def run_reference(args, wl_id, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    nproc = os.cpu_count() or 1
    workers = max(1, min(wl.H, nproc))
    pool = OraclePool(wl_id, workers)
    t_start = time.perf_counter()
    try:
        for _ in range(args.warmup):
            pool.step(wl.H)
        times = [pool.step(wl.H) for _ in range(args.steps)]
    finally:
        pool.close()
    step_s = statistics.mean(times)
    value = wl.tokens / step_s
    sample = (f"each step: every head of {wl.name} through the fp64 oracle, heads spread over "
              f"{workers} spawned worker processes (one BLAS thread each)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": base_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle",
                             "sample": sample, "nproc": nproc, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_start}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# multi-rank bookkeeping (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------

def slowest_rank_ms(t_ms, device=None):
    """The step time of the slowest rank (all-reduce MAX); t_ms itself when
    running alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(t_ms)
    tt = torch.tensor([float(t_ms)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tokens_per_s(tokens_per_rank, world, t_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (t_ms * 1e-3)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def step_bytes(wl):
    """Algorithmic bytes of one whole step (sum over the kernels' rows)."""
    names = ["score_tc", "select_topw", "attention_tc", "scatter_average"]
    if wl.ema:
        names += ["ema_bucket", "ema_update"]
    return sum(kernel_work(nm, wl)["bytes"] for nm in names)


def causal_flops(wl):
    """Flops of the causal products inside the clusters: row i of a cluster
    meets i + 1 keys, for QK^T and PV (2 d flops each)."""
    return 4.0 * wl.d * (wl.w * (wl.w + 1) / 2) * wl.k * wl.B * wl.H


class Measured:
    """Device measurements of one workload (the library's tensors stay on the
    GPU until close())."""

    def __init__(self, wl, dev, fused=False):
        import numpy as np
        import torch

        import content_sparse_attention_shared_b300 as rt

        self.wl, self.dev = wl, dev
        if wl.dtype == "f32":
            q_h, v_h = torch.from_numpy(wl.q), torch.from_numpy(wl.v)
        else:
            q_h = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16)
            v_h = torch.from_numpy(wl.v.view(np.int16)).view(torch.bfloat16)
        self.q_h, self.v_h = q_h.pin_memory(), v_h.pin_memory()
        self.q, self.v = self.q_h.to(dev), self.v_h.to(dev)
        self.mu = torch.from_numpy(wl.centroids).to(dev)
        self.out = torch.empty_like(self.v)
        self.idx = torch.empty((wl.B, wl.H, wl.k, wl.w), dtype=torch.int32, device=dev)
        self.assign = torch.empty((wl.B, wl.H, wl.n), dtype=torch.int32, device=dev)
        self.ws = rt.Workspace.for_shape(wl.B, wl.H, wl.n, wl.d, wl.k, wl.w, self.q.dtype, dev)
        self.rt = rt
        self.fused = fused

    def step(self, qq=None, vv=None, oo=None):
        # launches go to torch's current stream (the capture stream while a
        # CUDA graph is being recorded)
        rt, wl = self.rt, self.wl
        qq = self.q if qq is None else qq
        vv = self.v if vv is None else vv
        oo = self.out if oo is None else oo
        if wl.ema and self.fused:
            # the training-step call: the centroid update overlaps the forward's tail
            rt.rt_routing_attention_step(qq, vv, self.mu, wl.w, wl.decay, causal=True,
                                         out=oo, idx_out=self.idx, assign_out=self.assign,
                                         workspace=self.ws)
            return
        rt.rt_routing_attention(qq, qq, vv, self.mu, wl.w, causal=True, out=oo,
                                idx_out=self.idx, assign_out=self.assign, workspace=self.ws)
        if wl.ema:
            rt.rt_centroid_ema(qq, self.assign, self.mu, wl.decay, workspace=self.ws)

    def capture(self, warmup):
        import torch
        for _ in range(max(3, warmup)):
            self.step()
        torch.cuda.synchronize()
        self.ws.check()
        n0 = self.rt.rt_launch_count()
        self.step()
        torch.cuda.synchronize()
        self.launches_per_step = self.rt.rt_launch_count() - n0
        self.graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(cap):
            self.step()  # warm-up on the capture stream
        cap.synchronize()
        with torch.cuda.graph(self.graph, stream=cap):
            self.step()
        torch.cuda.synchronize()
        for _ in range(max(3, warmup)):
            self.graph.replay()
        torch.cuda.synchronize()

    def timed(self, steps, flush, stream, world, clocks=None, soak_ms=0.0):
        """K graph replays, L2 flushed (outside the events) before each.
        With `clocks` (a ClockSampler), the sampler runs over `soak_ms` of
        untimed replays immediately before the timed region and over the
        region itself."""
        import torch
        import torch.distributed as dist
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

        def region():
            if soak_ms > 0:
                t_end = time.perf_counter() + soak_ms * 1e-3
                while time.perf_counter() < t_end:
                    for _ in range(20):
                        flush.zero_()
                        self.graph.replay()
                    torch.cuda.synchronize()
            for i in range(steps):
                flush.zero_()
                ev[i][0].record(stream)
                self.graph.replay()
                ev[i][1].record(stream)
            torch.cuda.synchronize()

        if clocks is not None:
            with clocks:
                region()
        else:
            region()
        t_ms = slowest_rank_ms(statistics.mean(a.elapsed_time(b) for a, b in ev), self.dev)
        if world > 1:
            dist.barrier()
        self.ws.check()
        return t_ms

    def kernel_times(self, steps, flush):
        """Per-kernel device times: one step in its sequential form (forward,
        then the centroid update on the same stream, so no kernel's bracket
        includes time spent waiting for SMs that another stream holds) is
        captured as a CUDA graph with the library's launch hook on, which puts
        a CUDA-event record node just before and just after every kernel; the
        graph is replayed, L2 flushed before each replay, and each kernel's
        time is the mean over the replays of its event pair's elapsed time."""
        rt = self.rt
        fused, self.fused = self.fused, False
        try:
            return self._kernel_times(steps, flush)
        finally:
            self.fused = fused

    def _kernel_times(self, steps, flush):
        import torch
        rt = self.rt
        prof_steps = min(steps, 50)
        self.step()  # the sequential form once, eagerly, before its capture
        torch.cuda.synchronize()
        n0 = rt.rt_launch_count()
        self.step()
        torch.cuda.synchronize()
        per_step = rt.rt_launch_count() - n0
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(per_step)]
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(torch.cuda.current_stream(self.dev))
        rt.rt_profile_set(pairs)
        try:
            with torch.cuda.graph(graph, stream=cap):
                self.step()
            names = [rt.rt_profile_kernel_name(i) for i in range(len(pairs))]
        finally:
            rt.rt_profile_set([])
        torch.cuda.synchronize()
        per_kind = {}
        for _ in range(prof_steps):
            flush.zero_()
            graph.replay()
            torch.cuda.synchronize()
            for i, (a, b) in enumerate(pairs):
                per_kind.setdefault(names[i], []).append(a.elapsed_time(b))
        del graph
        kern = {k2: {"launches": len(v2), "avg_us": 1e3 * statistics.mean(v2),
                     "total_ms": sum(v2)} for k2, v2 in per_kind.items()}
        total = sum(x["total_ms"] for x in kern.values())
        peaks = _peaks()
        for name, x in kern.items():
            x["share"] = x["total_ms"] / total if total else None
            wk = kernel_work(name, self.wl)
            x["hbm_gbs"] = wk["bytes"] / (x["avg_us"] * 1e-6) / 1e9 if x["avg_us"] else None
            x["hbm_frac"] = x["hbm_gbs"] / peaks["hbm_gbs"] if x["hbm_gbs"] else None
        return kern

    def e2e(self, steps, flush, stream, world):
        """The same step through the public API from pinned host buffers, run
        the way a serving loop runs it: every step's Q and V are copied in on
        a copy stream, the step (L2 flush, then the library call) runs on the
        compute stream once they have landed, and its output is copied out on
        a second copy stream.  Two sets of device buffers let the next step's
        inputs come in while this step computes and the previous output goes
        out (host-to-device and device-to-host copies use separate copy
        engines and PCIe directions).  The timed region runs from the first
        step's first copy in to the last step's copy out, so it holds every
        step's copies; the time per step is that span / steps."""
        import torch
        import torch.distributed as dist
        dev = self.dev
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        qb = [self.q, torch.empty_like(self.q)]
        vb = [self.v, torch.empty_like(self.v)]
        ob = [self.out, torch.empty_like(self.out)]
        out_h = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory() for _ in range(2)]
        ev = lambda: torch.cuda.Event(enable_timing=False)
        landed = [ev() for _ in range(steps)]
        computed = [ev() for _ in range(steps)]
        drained = [ev() for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        h2d_s.wait_stream(stream)
        for i in range(steps):
            j = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(computed[i - 2])  # the step that read this buffer is done
                qb[j].copy_(self.q_h, non_blocking=True)
                vb[j].copy_(self.v_h, non_blocking=True)
                landed[i].record(h2d_s)
            stream.wait_event(landed[i])
            if i >= 2:
                stream.wait_event(drained[i - 2])  # this output buffer has been read out
            flush.zero_()
            self.step(qb[j], vb[j], ob[j])
            computed[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(computed[i])
                out_h[j].copy_(ob[j], non_blocking=True)
                drained[i].record(d2h_s)
        stream.wait_event(drained[steps - 1])
        t1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = slowest_rank_ms(t0.elapsed_time(t1) / steps, dev)
        h2d = (self.q_h.numel() * self.q_h.element_size() + self.v_h.numel() * self.v_h.element_size())
        d2h = out_h[0].numel() * out_h[0].element_size()
        return e2e_ms, h2d, d2h

    def close(self):
        import torch
        for name in ("graph", "q", "v", "mu", "out", "idx", "assign", "ws", "q_h", "v_h"):
            if hasattr(self, name):
                delattr(self, name)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def roofline_for(kern, wl, peaks):
    dname, dstat = max(kern.items(), key=lambda kv: kv[1]["total_ms"])
    work = kernel_work(dname, wl)
    bound = KERNEL_BOUND.get(dname, "hbm")
    avg_s = dstat["avg_us"] * 1e-6
    if bound == "hbm":
        achieved, peak, unit = work["bytes"] / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        achieved, peak, unit = work["flops"] / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = (work["flops"] / avg_s / 1e12, alu_peak_tflops(peaks["sm_max_mhz"]),
                                "TFLOP/s")
    return {"kernel": dname, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic_for(dname, wl.name),
            "peak_source": (peaks["source"] if bound != "alu"
                            else "derived: 148 SMs x 128 fp32 lanes x 2 flop x max SM clock"),
            "algorithmic_per_launch": work["bytes"] if bound == "hbm" else work["flops"]}


def config_entry(wl, t_ms, kern, peaks, cpu):
    """The per-workload record of the `configs` map."""
    s = t_ms * 1e-3
    entry = {"workload": wl.name, "ms_per_step": t_ms, "tokens_per_s": wl.tokens / s,
             "tflops_nominal": wl.nominal_flops() / s / 1e12,
             "tflops_causal": causal_flops(wl) / s / 1e12,
             "tflops_frac_bf16": wl.nominal_flops() / s / 1e12 / peaks["bf16_tflops"],
             "step_hbm_frac": step_bytes(wl) / s / 1e9 / peaks["hbm_gbs"],
             "step": "forward + centroid update" if wl.ema else "forward",
             "kernels": {k2: {"avg_us": v2["avg_us"], "share": v2["share"],
                              "hbm_frac": v2["hbm_frac"]} for k2, v2 in kern.items()}}
    if cpu is not None:
        entry["cpu_oracle"] = cpu
    return entry


def run_ours(args, wl_id, wl):
    import torch
    import torch.distributed as dist

    import content_sparse_attention_shared_b300 as rt
    from content_sparse_attention_shared_b300 import build as rt_build
    from workloads import CONFIG_ORDER, make_workload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rt_build.build()
    rt.load_library()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()

    props = torch.cuda.get_device_properties(dev)
    pci = None
    if hasattr(props, "pci_bus_id"):
        pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                     getattr(props, "pci_device_id", 0))

    # ---- the headline workload ------------------------------------------
    m = Measured(wl, dev, fused=not args.sequential_step)
    m.capture(args.warmup)
    clk = ClockSampler(local, pci)
    t_ms = m.timed(args.steps, flush, stream, world, clocks=clk, soak_ms=args.soak_ms)
    gpu_launches = m.launches_per_step * args.steps  # kernels the timed replays ran
    kern = m.kernel_times(args.steps, flush)
    e2e_ms, h2d, d2h = m.e2e(args.steps, flush, stream, world)
    local_attn = local_attention_timing(wl, m.q, m.v, flush, stream, args.steps)
    launches_per_step = m.launches_per_step
    m.close()

    # ---- every workload, at one GPU --------------------------------------
    configs = None
    if world == 1 and not args.no_configs:
        configs = {}
        csteps = max(10, min(args.steps, 50))
        for cid in CONFIG_ORDER:
            cw = wl if cid == wl_id else make_workload(cid)
            if cid == wl_id:
                ct, ck = t_ms, kern
            else:
                cm = Measured(cw, dev, fused=not args.sequential_step)
                cm.capture(args.warmup)
                ct = cm.timed(csteps, flush, stream, world)
                ck = cm.kernel_times(csteps, flush)
                cm.close()
            cpu = None if args.no_cpu_baseline else oracle_baseline(cid, cw)
            configs[cid] = config_entry(cw, ct, ck, peaks, cpu)
            configs[cid]["steps"] = args.steps if cid == wl_id else csteps

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    value = job_tokens_per_s(wl.tokens, world, t_ms)
    tflops = wl.nominal_flops() * world / (t_ms * 1e-3) / 1e12
    clocks = clk.summary()
    clocks["window"] = (f"{args.soak_ms:.0f} ms of untimed replays immediately before the timed "
                        f"region, then the timed region")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": base_config(wl),
        "timing": {"step_call": ("rt_routing_attention + rt_centroid_ema, one stream"
                                 if args.sequential_step or not wl.ema else
                                 "rt_routing_attention_step (centroid update on a side stream)"),
                   "l2": "flushed before every timed step (256 MiB write)",
                   "graph": "the step captured once as a CUDA graph, replayed per step",
                   "kernel_times": "one step captured as a CUDA graph with a CUDA-event "
                                   "record node before and after every kernel, replayed with "
                                   "L2 flushed before each replay (a kernel's bracket includes "
                                   "its launch latency inside the graph); the centroid update "
                                   "runs after the forward on one stream, so each kernel is "
                                   "timed alone"},
        "e2e_schedule": ("copies in, compute and copies out overlapped across consecutive steps "
                         "(double-buffered device inputs and outputs); the timed span runs "
                         "from the first step's first copy in to the last step's copy out"),
        "tflops": tflops, "tflops_causal": causal_flops(wl) * world / (t_ms * 1e-3) / 1e12,
        "tflops_frac_bf16": tflops / peaks["bf16_tflops"],
        "roofline": roofline_for(kern, wl, peaks),
        "e2e": {"value": job_tokens_per_s(wl.tokens, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches, "launches_per_step": launches_per_step,
        "clocks": clocks, "kernels": kern,
        "local_attention": local_attn,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = (configs[wl_id]["cpu_oracle"] if configs
                                else oracle_baseline(wl_id, wl))
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3", help="c1..c5 (default: the n=8192 configuration)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only (no `configs` map)")
    ap.add_argument("--sequential-step", action="store_true",
                    help="time the step as rt_routing_attention then rt_centroid_ema on one "
                         "stream (default: one rt_routing_attention_step call, which runs the "
                         "centroid update on a side stream beside the forward's tail)")
    ap.add_argument("--soak-ms", type=float, default=300.0,
                    help="untimed replays right before the timed region, for the clock record")
    args = ap.parse_args()
    if args.impl == "reference":
        os.environ.update(ONE_THREAD_ENV)  # before numpy is imported
    from workloads import make_workload
    wl = make_workload(args.workload)
    if args.impl == "reference":
        run_reference(args, args.workload, wl)
    else:
        run_ours(args, args.workload, wl)


if __name__ == "__main__":
    main()
