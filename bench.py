"""Benchmark of the sliding-window-attention-with-sinks library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--primary-only]

Prints ONE JSON line. The primary metric is prefill banded TFLOP/s on the Llama-2-7B head shape
(B=1, H=32, L=8192, d=128, w=1024, s=4, bf16): banded FLOPs = 4 * B * H * d * sum_t min(t+1, w).
A step is one swa_sink_prefill call over that batch; inputs (256 MiB per step) are larger than L2.
Secondary entries: prefill at the Mistral-7B window shape (s=0 and s=4), streaming decode
(tokens/s, B=64, H=40, 4 sink + 1020 recent slots, 20480 steps) and chunked prefill
(L=131072 in 4096-token chunks). Under torchrun each rank runs the same per-GPU workload on its own
GPU (weak scaling; no collective on the data path) and the aggregate divides all ranks' work by the
slowest rank's time.

--impl reference times the oracle (fp64 C on the host cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PRIMARY = "prefill_llama7b_L8192_w1024_s4"
METRIC = "prefill banded TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------------------------------ accounting
def banded_pairs(L: int, w: int, pos0: int = 0) -> int:
    """sum over positions t in [pos0, pos0 + L) of min(t + 1, w): (query, key) pairs of the band."""
    lo, hi = pos0, pos0 + L
    ramp = min(hi, w)
    total = (ramp * (ramp + 1) - lo * (lo + 1)) // 2 if ramp > lo else 0
    return total + max(0, hi - max(lo, w)) * w


def banded_flops(B, H, L, d, w) -> int:
    return 4 * B * H * d * banded_pairs(L, w)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, files, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or taken on other code."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_hash") != kernel_source_hash(files) or d.get("workload") != workload:
        return None
    return d.get("bytes_per_launch")


# ------------------------------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    """Max of a float over ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_rate(units_per_rank: float, world: int, t_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / t_max


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms in the background; windows mark the timed regions."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.windows = []
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(prefix="clocks", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.out.name)
        inside = [r for r in rows if any(a - 0.25 <= r[0] <= b + 0.25 for a, b in self.windows)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


class NvmlWindowSampler:
    """Reads the SM clock and the active clock-event reasons of one GPU through NVML (read only; nothing is
    set) every ~0.5 ms from a background thread while a timed region runs, so that even a region of a few
    milliseconds gets its own clock samples.  NVML is reached through ctypes (libnvidia-ml.so.1)."""
    # clock-event reason bits of NVML
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None):
        self.ok = False
        self.samples = []
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if uuid:
                rc = self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
            else:
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if rc != 0:
                return
            self.reasons_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) != 0:  # 1 = NVML_CLOCK_SM
            return None
        self.reasons_fn(self.h, ctypes.byref(rs))
        return clk.value, rs.value

    def __enter__(self):
        self._stop = threading.Event()
        self.samples = []

        def loop():
            while not self._stop.is_set():
                r = self._read()
                if r is not None:
                    self.samples.append(r)
                time.sleep(0.0005)

        if self.ok:
            self._thr = threading.Thread(target=loop, daemon=True)
            self._thr.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._thr.join()

    def summary(self):
        if not self.samples:
            return {"samples": 0}
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"samples": len(self.samples), "sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_mhz_min": min(c for c, _ in self.samples),
                "reasons": sorted(v for k, v in self.REASONS.items() if bits & k)}


# ------------------------------------------------------------------------------------------ GPU legs
def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def _check_status(swa):
    rc = swa.swa_device_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {swa.last_error()}")


def time_loop(step, steps, warmup, world, clocks, window=None):
    """W untimed calls, then K calls bracketed by barrier + synchronize; returns max-over-ranks seconds.
    ``window``: an NvmlWindowSampler that samples the clocks inside the timed region itself."""
    import contextlib
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = _events()
    with (window if window is not None else contextlib.nullcontext()):
        t0 = time.time()
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        t1 = time.time()
    barrier(world)
    if clocks is not None:
        clocks.mark(t0, t1)
    return reduce_max(e0.elapsed_time(e1) / 1e3, world)


def dilated_flops(B, H, L, d, w, s, r):
    """4 d per (query, key) pair of the dilated key sets: sinks i < min(s, t + 1) plus min(m, t // r + 1)
    window keys, less the sinks that are also window keys."""
    m = w - s
    pairs = 0
    for t in range(L):
        both = sum(1 for i in range(min(s, t + 1)) if (t - i) % r == 0 and (t - i) // r < m)
        pairs += min(s, t + 1) + min(m, t // r + 1) - both
    return 4.0 * B * H * d * pairs


def blocksparse_pairs(L, w, s, globals_, block, rand) -> int:
    """Sum over the rows t of |K(t)| for the block-sparse key sets (causal union of sinks, window, global
    tokens, the random key blocks of t's query block; a global row sees all t + 1 earlier keys), counted as a
    union of position intervals per row."""
    m = w - s
    g = sorted(int(x) for x in globals_)
    runs = []  # global tokens as runs of consecutive positions
    for x in g:
        if runs and runs[-1][1] == x - 1:
            runs[-1][1] = x
        else:
            runs.append([x, x])
    gset = set(g)
    total = 0
    for t in range(L):
        if t in gset:
            total += t + 1
            continue
        iv = [(0, min(s, t + 1) - 1), (max(0, t - m + 1), t)]
        iv += [(a, min(b, t)) for a, b in runs if a <= t]
        if rand is not None:
            iv += [(kb * block, min(kb * block + block - 1, t)) for kb in rand[t // block] if 0 <= kb * block <= t]
        iv.sort()
        hi = -1
        for a, b in iv:
            if b < a:
                continue
            if a > hi:
                total += b - a + 1
                hi = b
            elif b > hi:
                total += b - hi
                hi = b
    return total


def hybrid_flops(B, H, L, d, w, s) -> float:
    """The banded SWA FLOPs plus the linear branch in its recurrent form: for each key that leaves the window
    (L - m - s of them) its feature map (2 d * d/2 * 2) and the rank-1 fold of phi(k)^T v (2 d^2); for each
    row with a non-empty state (also L - m - s rows) the query's feature map (2 d^2) and phi(q) S (2 d^2)."""
    n = max(0, L - (w - s) - s)
    return banded_flops(B, H, L, d, w) + B * H * n * 8.0 * d * d


def prefill_leg(swa, wl, steps, warmup, world, rank, clocks, e2e=False, rope=False, dilation=0, window=None,
                blocksparse=None, hybrid=False):
    """Prefill steps; with ``rope`` the RoPE prefill at the positions inside the cache (base 10000): a
    rotation pass over q and k, then the tensor-core prefill on the rotated rows (2 launches a step);
    ``blocksparse`` = (globals, block, rand): the block-sparse prefill with that pattern."""
    import numpy as np
    import torch
    import swa_inputs
    B, H, L, d, w, s = wl.B, wl.H, wl.L, wl.d, wl.w, wl.s
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, wl.seed + 7919 * rank, wl.torch_dtype, "cuda", wl.sink_boost)
    o = torch.empty_like(q)
    lib = swa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    dt = 0 if wl.dtype == "bf16" else 1
    if hybrid:
        wf = swa_inputs.hedgehog_weights(d, wl.seed).to("cuda")
        nws = lib.swa_hybrid_prefill_workspace_size(B, H, L, d)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), wf.data_ptr(), o.data_ptr(), None, None, B, H, L, d, w, s,
                wl.scale, ws.data_ptr(), nws, dt, stream)
        call = lib.swa_hybrid_prefill
    elif blocksparse is not None:
        globals_, block, rand = blocksparse
        g = np.ascontiguousarray(globals_, dtype=np.int32)
        rb = np.ascontiguousarray(rand, dtype=np.int32)
        nws = lib.swa_sink_prefill_blocksparse_workspace_size(L, g.size, block, rb.shape[1])
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, B, H, L, d, w, s, wl.scale,
                g.ctypes.data, g.size, block, rb.ctypes.data, rb.shape[1], ws.data_ptr(), nws, dt, stream)
        call = lib.swa_sink_prefill_blocksparse
    elif dilation:  # bf16, d = 128: in place, no workspace
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, B, H, L, d, w, s, dilation, wl.scale,
                None, 0, dt, stream)
        call = lib.swa_sink_prefill_dilated
    elif rope:
        nws = lib.swa_sink_prefill_rope_workspace_size(B, H, L, d, s)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, B, H, L, d, w, s, wl.scale, 10000.0,
                ws.data_ptr(), nws, dt, stream)
        call = lib.swa_sink_prefill_rope
    else:
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, None, None, 0, B, H, L, d, w, s,
                wl.scale, dt, stream)
        call = lib.swa_sink_prefill

    def step():
        rc = call(*args)
        if rc:
            raise RuntimeError(swa.last_error())

    t = time_loop(step, steps, warmup, world, clocks, window)
    _check_status(swa)
    if hybrid:
        flops = hybrid_flops(B, H, L, d, w, s)
        launches = 5  # the SWA prefill, the feature-map weights, the chunk states, their scan, the linear pass
    elif blocksparse is not None:
        flops = 4.0 * B * H * d * blocksparse_pairs(L, w, s, globals_, block, rand)
        launches = 2 if any(int(x) >= w for x in globals_) else 1  # global rows past the window: second pass
    else:
        flops = dilated_flops(B, H, L, d, w, s, dilation) if dilation else banded_flops(B, H, L, d, w)
        # dilated: the tensor-core pass, then the sink rows and the rows past the last whole group of r
        launches = (2 if s > 0 or L % dilation else 1) if dilation else 2 if rope else 1
    res = {"flops_per_step": flops, "seconds": t, "steps": steps, "tflops": flops * steps / t / 1e12,
           "ms_per_step": t / steps * 1e3, "launches": launches * steps}
    if e2e:
        # the same prefill through the public host-buffer call: every step copies q/k/v from pinned host
        # memory and o back (the library pipelines the copies against the compute over row groups)
        qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
        oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hargs = (qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), None, q.data_ptr(), k.data_ptr(),
                 v.data_ptr(), o.data_ptr(), None, B, H, L, d, w, s, wl.scale, 0 if wl.dtype == "bf16" else 1, stream)

        def step_e2e():
            rc = lib.swa_sink_prefill_host(*hargs)
            if rc:
                raise RuntimeError(swa.last_error())

        te = time_loop(step_e2e, steps, min(warmup, 3), world, None)
        _check_status(swa)
        res["e2e"] = {"seconds": te, "tflops": flops * steps / te / 1e12,
                      "h2d_bytes_per_step": 3 * q.numel() * q.element_size(),
                      "d2h_bytes_per_step": o.numel() * o.element_size()}
    del q, k, v, o
    torch.cuda.empty_cache()
    return res


def chunked_leg(swa, wl, steps, warmup, world, rank, clocks, rope=False):
    """Chunked prefill steps; with ``rope`` the chunked prefill with RoPE at the positions inside the cache
    (one rotation pass over the sequence, then per chunk the prefill and two rolling writes)."""
    import torch
    import swa_inputs
    B, H, L, d, w, s, C = wl.B, wl.H, wl.L, wl.d, wl.w, wl.s, wl.chunk
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, wl.seed + 7919 * rank, wl.torch_dtype, "cuda", wl.sink_boost)
    o = torch.empty_like(q)
    kc = torch.empty((B, H, w, d), dtype=q.dtype, device="cuda")
    vc = torch.empty_like(kc)
    lib = swa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    if rope:
        nws = lib.swa_sink_prefill_chunked_rope_workspace_size(B, H, L, d, w, s)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, kc.data_ptr(), vc.data_ptr(), B, H, L,
                d, w, s, wl.scale, C, 10000.0, ws.data_ptr(), nws, 0, stream)
        call = lib.swa_sink_prefill_chunked_rope
    else:
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, kc.data_ptr(), vc.data_ptr(), B, H, L,
                d, w, s, wl.scale, C, 0, stream)
        call = lib.swa_sink_prefill_chunked

    def step():
        rc = call(*args)
        if rc:
            raise RuntimeError(swa.last_error())

    t = time_loop(step, steps, warmup, world, clocks)
    _check_status(swa)
    flops = banded_flops(B, H, L, d, w)
    nch = (L + C - 1) // C
    groups = 2 if B * H >= 16 else 1  # the library walks >= 16 (b, h) rows as two row groups
    del q, k, v, o, kc, vc
    torch.cuda.empty_cache()
    per_chunk = 3 if rope else 2
    return {"flops_per_step": flops, "seconds": t, "steps": steps, "tflops": flops * steps / t / 1e12,
            "ms_per_step": t / steps * 1e3, "launches": steps * (per_chunk * nch * groups + (1 if rope else 0))}


def decode_leg(swa, wl, world, rank, clocks, steps=None, rope=False, dilation=0):
    """The whole streaming run: per step one rolling write of the new key/value and one decode (with
    ``rope``: the decode with RoPE at the positions inside the cache, base 10000, unrotated keys; with
    ``dilation``: the dilated window, one rolling cache per residue class)."""
    import torch
    import swa_inputs
    B, H, d, w, s = wl.B, wl.H, wl.d, wl.w, wl.s
    T = wl.L if steps is None else steps
    seed = wl.seed + 7919 * rank
    qs = swa_inputs.normal((T, B, H, d), seed, swa_inputs.TID_Q, wl.torch_dtype, "cuda")
    ks = swa_inputs.normal((T, B, H, d), seed, swa_inputs.TID_K, wl.torch_dtype, "cuda")
    vs = swa_inputs.normal((T, B, H, d), seed, swa_inputs.TID_V, wl.torch_dtype, "cuda")
    if wl.sink_boost:
        ks[:4] *= 4.0
    kc = torch.zeros(((dilation,) if dilation else ()) + (B, H, w, d), dtype=qs.dtype, device="cuda")
    vc = torch.zeros_like(kc)
    o = torch.empty((B, H, d), dtype=qs.dtype, device="cuda")
    lib = swa.lib()
    nws = (lib.swa_sink_decode_rope_workspace_size(B, H, d, w) if rope
           else swa.swa_sink_decode_workspace_size(B, H, d, w))
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    row = B * H * d * qs.element_size()
    qp, kp, vp = qs.data_ptr(), ks.data_ptr(), vs.data_ptr()
    dt = 0 if wl.dtype == "bf16" else 1

    def run(t0, t1):
        for t in range(t0, t1):
            if dilation:
                rc = lib.swa_sink_dilated_cache_write(kc.data_ptr(), vc.data_ptr(), kp + t * row, vp + t * row, B, H,
                                                      d, w, s, dilation, t, dt, stream)
                rc |= lib.swa_sink_decode_step_dilated(qp + t * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                                       None, B, H, d, w, s, dilation, t, wl.scale, ws.data_ptr(), nws,
                                                       dt, stream)
                if rc:
                    raise RuntimeError(swa.last_error())
                continue
            rc = lib.kv_rolling_write(kc.data_ptr(), vc.data_ptr(), kp + t * row, vp + t * row, B, H, d, w, s, t, 1,
                                      dt, stream)
            if rope:
                rc |= lib.swa_sink_decode_step_rope(qp + t * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, B,
                                                    H, d, w, s, t, wl.scale, 10000.0, ws.data_ptr(), nws, dt, stream)
            else:
                rc |= lib.swa_sink_decode_step(qp + t * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, B, H,
                                               d, w, s, t, wl.scale, ws.data_ptr(), nws, dt, stream)
            if rc:
                raise RuntimeError(swa.last_error())

    run(0, min(T, 64))  # warm-up on the first positions, then start the stream again from an empty cache
    kc.zero_()
    vc.zero_()
    t = time_loop(lambda: run(0, T), 1, 0, world, clocks)
    _check_status(swa)
    kv_bytes = 2 * d * qs.element_size() * B * H * sum(min(x + 1, w) for x in range(T))
    res = {"steps": T, "seconds": t, "tok_per_s": B * T / t, "kv_bytes_read": kv_bytes,
           "launches": 2 * T}
    # the decode kernel alone at a full cache, for its roofline
    R = 200
    tl = T - 1

    def dstep():
        if dilation:
            rc = lib.swa_sink_decode_step_dilated(qp + tl * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, B,
                                                  H, d, w, s, dilation, tl, wl.scale, ws.data_ptr(), nws, dt, stream)
        elif rope:
            rc = lib.swa_sink_decode_step_rope(qp + tl * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, B, H,
                                               d, w, s, tl, wl.scale, 10000.0, ws.data_ptr(), nws, dt, stream)
        else:
            rc = lib.swa_sink_decode_step(qp + tl * row, kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, B, H, d,
                                          w, s, tl, wl.scale, ws.data_ptr(), nws, dt, stream)
        if rc:
            raise RuntimeError(swa.last_error())

    tk = time_loop(dstep, R, 5, world, clocks)
    _check_status(swa)
    nvalid = min(tl + 1, w)
    step_bytes = B * H * (2 * nvalid * d + 2 * d) * qs.element_size()
    res["kernel"] = {"name": "decode_kernel", "avg_us": tk / R * 1e6, "bytes_per_launch": step_bytes,
                     "gbs": step_bytes / (tk / R) / 1e9}
    del qs, ks, vs, kc, vc
    torch.cuda.empty_cache()
    return res


def hybrid_decode_leg(swa, wl, world, rank, clocks, steps=200):
    """Decode steps of the SWA + linear-attention hybrid at a full cache (positions T, T+1, ...): per step the
    state pass (fold of the evicted key, rolling write, phi(q) S), the SWA decode and the combination."""
    import torch
    import swa_inputs
    B, H, d, w, s = wl.B, wl.H, wl.d, wl.w, wl.s
    T = wl.L
    seed = wl.seed + 7919 * rank
    kc = swa_inputs.normal((B, H, w, d), seed, swa_inputs.TID_K, wl.torch_dtype, "cuda")
    vc = swa_inputs.normal((B, H, w, d), seed, swa_inputs.TID_V, wl.torch_dtype, "cuda")
    qs = swa_inputs.normal((steps, B, H, d), seed + 1, swa_inputs.TID_Q, wl.torch_dtype, "cuda")
    ks = swa_inputs.normal((steps, B, H, d), seed + 1, swa_inputs.TID_K, wl.torch_dtype, "cuda")
    vs = swa_inputs.normal((steps, B, H, d), seed + 1, swa_inputs.TID_V, wl.torch_dtype, "cuda")
    S = torch.zeros((B, H, d, d), dtype=torch.float32, device="cuda")
    z = torch.zeros((B, H, d), dtype=torch.float32, device="cuda")
    wf = swa_inputs.hedgehog_weights(d, wl.seed).to("cuda")
    o = torch.empty((B, H, d), dtype=qs.dtype, device="cuda")
    lib = swa.lib()
    nws = lib.swa_hybrid_decode_workspace_size(B, H, d, w)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    row = B * H * d * qs.element_size()
    qp, kp, vp = qs.data_ptr(), ks.data_ptr(), vs.data_ptr()
    cnt = [0]

    def step():
        i = cnt[0] % steps
        rc = lib.swa_hybrid_decode_step(qp + i * row, kp + i * row, vp + i * row, kc.data_ptr(), vc.data_ptr(),
                                        S.data_ptr(), z.data_ptr(), wf.data_ptr(), o.data_ptr(), B, H, d, w, s,
                                        T + cnt[0], wl.scale, ws.data_ptr(), nws, 0, stream)
        cnt[0] += 1
        if rc:
            raise RuntimeError(swa.last_error())

    t = time_loop(step, steps, 5, world, clocks)
    _check_status(swa)
    # bytes per step: the cache (w keys and values), q / k_new / v_new / o, the state read and written
    step_bytes = B * H * (2 * w * d * 2 + 4 * d * 2 + 2 * (d * d + d) * 4)
    res = {"steps": steps, "seconds": t, "tok_per_s": B * steps / t, "us_per_step": t / steps * 1e6,
           "bytes_per_step": step_bytes, "gbs": step_bytes / (t / steps) / 1e9, "launches": 4 * steps}
    del kc, vc, qs, ks, vs, S, z
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------------------ oracle legs
def oracle_sample_inputs(wl, heads: int):
    """Host copies of the first `heads` heads of the workload's inputs (drawn on the CPU)."""
    import swa_inputs
    q, k, v = swa_inputs.prefill_inputs(1, heads, wl.L, wl.d, wl.seed, wl.torch_dtype, "cpu", wl.sink_boost)
    return q, k, v


def oracle_run(wl, q, k, v, rows: int):
    """The oracle over rows [0, rows) of the given heads; returns (seconds, banded flops computed)."""
    import numpy as np
    import oracle
    H, d = q.shape[1], q.shape[3]
    pos = np.arange(rows, dtype=np.int64)
    qq, kk, vv = (oracle._f64(x[0, :, :rows]) for x in (q, k, v))
    t0 = time.perf_counter()
    oracle.attend(qq, pos, kk, vv, pos, wl.w, wl.s, wl.scale)
    t = time.perf_counter() - t0
    return t, 4 * H * d * banded_pairs(rows, wl.w)


def cpu_baseline_leg(wl, budget_s: float = 10.0):
    """The oracle on the host cores over the whole workload, repeated until about `budget_s` seconds."""
    import oracle
    q, k, v = oracle_sample_inputs(wl, wl.H)
    tot_t, tot_f, reps = 0.0, 0, 0
    while tot_t < budget_s and reps < 20:
        t, f = oracle_run(wl, q, k, v, wl.L)
        tot_t += t
        tot_f += f
        reps += 1
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"all {wl.H} heads x {wl.L} rows of {wl.name}, {reps} pass(es), fp64 C, {tot_t:.1f} s",
            "seconds": tot_t}


def reference_main(args, world, rank):
    """The reference arm: the oracle, as it stands, on the host cores, a bounded sample per step."""
    import oracle
    import swa_inputs
    if rank != 0:
        return 0
    wl = swa_inputs.WORKLOADS[PRIMARY]
    q, k, v = oracle_sample_inputs(wl, 1)
    rows = 2048  # one head, the first 2048 rows: a bounded sample of the workload per step
    for _ in range(args.warmup):
        oracle_run(wl, q, k, v, rows)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        t, f = oracle_run(wl, q, k, v, rows)
        tot_t += t
        tot_f += f
    value = tot_f / tot_t / 1e12
    sample = f"per step: head 0, rows 0..{rows - 1} of {wl.name} (fp64 C oracle)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_config(wl):
    c = {"workload": wl.name, "B": wl.B, "H": wl.H, "L": wl.L, "d": wl.d, "w": wl.w, "s": wl.s, "dtype": wl.dtype,
         "parallelism": "replicas (weak)", "l2": "inputs larger than L2 (129 MB) every step"}
    if wl.chunk:
        c["chunk"] = wl.chunk
    return c


# ------------------------------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--primary-only", action="store_true", help="only the primary prefill leg")
    ap.add_argument("--legs", default="primary,mistral,chunked,decode,decode_rope,prefill_rope,chunked_rope,dilated,"
                                      "decode_dilated,blocksparse,hybrid,decode_hybrid",
                    help="comma list of legs to run (profiling runs pick one)")
    ap.add_argument("--decode-steps", type=int, default=None, help="shorter decode stream (profiling only)")
    args = ap.parse_args()
    legs = set(args.legs.split(","))
    if args.primary_only:
        legs = {"primary"}
    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_main(args, world, rank)
    args.warmup = max(args.warmup, 3)

    import torch
    import sliding_window_softmax_swa_gb300 as swa
    import swa_inputs

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    swa.lib(build_if_missing=True)
    peaks, peak_src = load_peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)

    wl = swa_inputs.WORKLOADS[PRIMARY]
    prim_window = NvmlWindowSampler(uuid)
    prim = prefill_leg(swa, wl, args.steps, args.warmup, world, rank, clocks, e2e=True,
                       window=prim_window) if "primary" in legs else None
    secondary = {}
    if "mistral" in legs:
        for name in ("prefill_mistral_B2_L32768_w4096_s0", "prefill_mistral_B2_L32768_w4096_s4"):
            r = prefill_leg(swa, swa_inputs.WORKLOADS[name], max(3, args.steps // 20), 3, world, rank, clocks)
            secondary[name] = {"metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
                               "ms_per_step": r["ms_per_step"],
                               "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"]}
    if "prefill_rope" in legs:
        r = prefill_leg(swa, wl, max(3, args.steps // 2), 3, world, rank, clocks, rope=True)
        secondary["prefill_rope_llama7b_L8192_w1024_s4"] = {
            "metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
            "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
            "what": "RoPE at the positions inside the cache (base 10000): rotation pass + tensor-core prefill",
            "launches_per_step": 2}
    if "chunked" in legs:
        cw = swa_inputs.WORKLOADS["chunked_mistral_L131072_w4096_s4_C4096"]
        r = chunked_leg(swa, cw, 3, 1, world, rank, clocks)
        secondary[cw.name] = {"metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
                              "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
                              "launches_per_step": r["launches"] // 3}
    if "dilated" in legs:
        r = prefill_leg(swa, wl, max(3, args.steps // 2), 3, world, rank, clocks, dilation=2)
        secondary["prefill_dilated_llama7b_L8192_w1024_s4_r2"] = {
            "metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
            "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
            "what": "dilated window with sinks, r = 2 (FLOPs over the dilated key sets): tensor-core prefill "
                    "reading each residue class through 4-D tensor maps, in place, + the sink rows on CUDA cores",
            "launches_per_step": 2}
    if "blocksparse" in legs:
        globals_, rand = swa_inputs.bigbird_pattern(wl.L, 64, 2, 3, seed=2024)
        r = prefill_leg(swa, wl, max(3, args.steps // 2), 3, world, rank, clocks, blocksparse=(globals_, 64, rand))
        secondary["prefill_blocksparse_llama7b_L8192_w1024_s4_g128_b64_r3"] = {
            "metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
            "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
            "what": "block-sparse: window + sinks + 128 global tokens + 3 random key blocks of 64 per query block "
                    "(FLOPs over those key sets): host tile lists + their upload, tensor-core prefill (+ the global "
                    "rows at or past w, none here: every global row below w is complete after the tiled pass)",
            "launches_per_step": r["launches"] // max(3, args.steps // 2)}
    if "hybrid" in legs:
        r = prefill_leg(swa, wl, max(3, args.steps // 2), 3, world, rank, clocks, hybrid=True)
        secondary["prefill_hybrid_linear_llama7b_L8192_w1024_s4"] = {
            "metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
            "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
            "what": "SWA + Hedgehog linear-attention branch for the evicted keys (FLOPs: banded SWA + the "
                    "recurrent linear branch, 8 d^2 per evicted key): SWA prefill, feature-map weights, chunk "
                    "states, scan, linear pass with the combination", "launches_per_step": 5}
    if "decode_hybrid" in legs:
        dw = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
        r = hybrid_decode_leg(swa, dw, world, rank, clocks)
        secondary["decode_hybrid_linear_llama13b_B64_w1024_s4_20480"] = {
            "metric": "decode tok/s", "value": aggregate_rate(r["tok_per_s"], world, 1.0), "unit": "tok/s",
            "us_per_step": r["us_per_step"], "what": "SWA + linear-attention hybrid at a full cache: state pass "
            "(evicted-key fold, rolling write, phi(q) S) + SWA decode + combination",
            "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": r["gbs"] / peaks["hbm_gbs"], "bytes_per_step": r["bytes_per_step"],
                         "note": "whole step (3 launches), cache + state bytes"}}
    if "chunked_rope" in legs:
        cw = swa_inputs.WORKLOADS["chunked_mistral_L131072_w4096_s4_C4096"]
        r = chunked_leg(swa, cw, 3, 1, world, rank, clocks, rope=True)
        secondary["chunked_rope_mistral_L131072_w4096_s4_C4096"] = {
            "metric": METRIC, "value": aggregate_rate(r["tflops"], world, 1.0), "unit": "TFLOP/s",
            "ms_per_step": r["ms_per_step"], "frac_of_bf16_peak": r["tflops"] / peaks["bf16_tflops"],
            "what": "RoPE at the positions inside the cache (base 10000): one rotation pass, then per chunk the "
                    "prefill and the rolling writes of rotated and unrotated keys",
            "launches_per_step": r["launches"] // 3}
    if "decode" in legs:
        dw = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
        r = decode_leg(swa, dw, world, rank, clocks, steps=args.decode_steps)
        secondary[dw.name] = {"metric": "decode tok/s", "value": aggregate_rate(r["tok_per_s"], world, 1.0),
                              "unit": "tok/s", "seconds": r["seconds"],
                              "kv_read_gbs": r["kv_bytes_read"] / r["seconds"] / 1e9,
                              "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": r["kernel"]["gbs"],
                                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                           "frac": r["kernel"]["gbs"] / peaks["hbm_gbs"],
                                           "frac_of_8tbs_nominal": r["kernel"]["gbs"] / 8000.0,
                                           "avg_us": r["kernel"]["avg_us"]}}
    if "decode_dilated" in legs:
        dw = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
        r = decode_leg(swa, dw, world, rank, clocks, steps=args.decode_steps, dilation=2)
        secondary["decode_dilated_llama13b_B64_w1024_s4_r2_20480"] = {
            "metric": "decode tok/s", "value": aggregate_rate(r["tok_per_s"], world, 1.0), "unit": "tok/s",
            "seconds": r["seconds"], "what": "dilated window with sinks, r = 2: one rolling cache per residue class",
            "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": r["kernel"]["gbs"],
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": r["kernel"]["gbs"] / peaks["hbm_gbs"],
                         "avg_us": r["kernel"]["avg_us"]}}
    if "decode_rope" in legs:
        dw = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
        r = decode_leg(swa, dw, world, rank, clocks, steps=args.decode_steps, rope=True)
        secondary["decode_rope_llama13b_B64_w1024_s4_20480"] = {
            "metric": "decode tok/s", "value": aggregate_rate(r["tok_per_s"], world, 1.0), "unit": "tok/s",
            "seconds": r["seconds"], "what": "RoPE at the positions inside the cache (base 10000), unrotated keys",
            "roofline": {"bound": "hbm", "kernel": "decode_kernel (rope)", "achieved": r["kernel"]["gbs"],
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": r["kernel"]["gbs"] / peaks["hbm_gbs"],
                         "avg_us": r["kernel"]["avg_us"],
                         "note": "bytes = the cache K/V rows + q/o (the per-pair angle rates are kernel parameters; sin/cos are computed in registers)"}}
    ck = clocks.stop()

    if rank != 0:
        return 0
    if prim is None:  # a profiling run of secondary legs only
        print(json.dumps({"metric": METRIC, "value": None, "secondary": secondary}))
        return 0
    t = prim["seconds"]
    value = aggregate_rate(prim["flops_per_step"] * prim["steps"] / 1e12, world, t)
    achieved = prim["flops_per_step"] / (t / prim["steps"]) / 1e12
    kfiles = ["sliding_window_softmax_swa_gb300/csrc/prefill_tc.cu", "sliding_window_softmax_swa_gb300/csrc/swa_device.cuh"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded iid N(0,1))",
        "config": workload_config(wl),
        "roofline": {"bound": "tensor", "kernel": "swa_prefill_tc_kernel", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "peak_source": f"{peak_src} bf16 burst", "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "traffic": traffic_for("swa_prefill_tc_kernel", kfiles, wl.name)},
        "e2e": {"value": aggregate_rate(prim["flops_per_step"] * prim["steps"] / 1e12, world, prim["e2e"]["seconds"]),
                "unit": "TFLOP/s", "h2d_bytes_per_step": prim["e2e"]["h2d_bytes_per_step"],
                "d2h_bytes_per_step": prim["e2e"]["d2h_bytes_per_step"]},
        "gpu_launches": prim["launches"],
        "clocks": {"sm_mhz": ck["sm_mhz"], "sm_max_mhz": ck["sm_max_mhz"], "reasons": ck["reasons"],
                   "samples": ck["samples"],
                   # NVML read every ~0.5 ms inside the primary timed region itself (nvidia-smi's 200 ms
                   # samples above cover all timed regions of the run)
                   "primary_window": prim_window.summary()},
        "secondary": secondary,
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline_leg(wl)
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
