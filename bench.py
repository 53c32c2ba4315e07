#!/usr/bin/env python
"""Benchmark of the fused masked multi-head attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-extra] [--no-cpu-baseline]

A step is one call of the hot path (one kernel launch) on one batch of
synthetic inputs already resident in HBM.  Input sets rotate so the data read
per step is not served from L2 (their total exceeds twice the L2 size).  The
metric is mask-aware attention TFLOP/s (4*B*H*Lq*Lk*D, halved for causal; for
the padding mask the valid keys 4*H*D*Lq*sum_b len_b), with us per call and
the fraction of the roofline of the dominant kernel.

Rank 0 prints one JSON line.  Under torchrun each rank runs its own replica
of the workload (weak scaling, no collective on the data path); the time is
the max over ranks.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from masked_head_attention_gb300 import synthetic  # noqa: E402

METRIC = "mask-aware attention TFLOP/s and µs/call at 1 GB300; % of roofline"
DEFAULT_WORKLOAD = "c5_long_causal_bf16"
DEFAULT_L2 = 129 * 1024 * 1024
KERNEL_OF = {  # dominant kernel of each workload
    "mha:f32": "mha_fwd_f32_kernel",      # D = 128; D = 64 runs attn_fwd_tf32x3_kernel
    "mha:bf16": "attn_fwd_bf16_kernel",
    "prenorm:bf16": "attn_fwd_bf16_kernel<prenorm>",   # one launch: statistics formed inside
    "prenorm_residual:bf16": "attn_fwd_bf16_kernel<prenorm>",
    "mha_bwd:f32": "mha_bwd_f32_kernel",
    "mha_bwd:bf16": "attn_bwd_bf16_kernel",   # tensor cores: key- and query-stationary kernels
}
SMALL_F32_MAX_KD = 16384   # the fp32 path stages all keys at once when Lk * D is at most this
DECODE_MAX_ROWS = 8        # bf16 self-attention with at most this many query rows: decode kernel
TF32X3_D = 64              # fp32 inputs with this head dimension run on the tensor cores (3xTF32)
# Dense tf32 tensor rate relative to bf16 (nominal 1.1 vs 2.25 PFLOP/s per GPU); the
# tf32 peak is the measured bf16 peak times this ratio.
TF32_OVER_BF16 = 1.1 / 2.25


# fp32 forward kernel choice (--f32-kernel): 0 automatic (3xTF32 for D = 64),
# 1 the tiled CUDA-core kernel, 2 the short-key-range CUDA-core kernel where it
# applies (else the tiled one).
F32_KERNEL = 0


def uses_tf32x3(w):
    return w.kind == "mha" and w.dtype == "f32" and w.D == TF32X3_D and F32_KERNEL == 0


def kernel_of(w):
    if uses_tf32x3(w):
        return "attn_fwd_tf32x3_kernel"
    if (w.kind == "mha" and w.dtype == "f32" and w.Lk * w.D <= SMALL_F32_MAX_KD
            and F32_KERNEL != 1):
        return "mha_fwd_f32_small_kernel"
    if w.kind == "mha" and w.dtype == "bf16" and w.Lq <= DECODE_MAX_ROWS:
        return "attn_decode_bf16_kernel"
    return KERNEL_OF["%s:%s" % (w.kind, w.dtype)]


# ------------------------------------------------------------------ helpers --
def visible_lengths(w, lens):
    if lens is None:
        return [w.Lk] * w.B
    return [max(0, min(int(x), w.Lk)) for x in lens]


def flops_per_pair(w):
    """FLOP per (query row, key, feature): 4 for the forward (QK^T and PV);
    10 for the backward (S = QK^T and dP = dout V^T formed again, then dV,
    dK and dQ: five products of 2 FLOP each)."""
    return 10.0 if w.kind == "mha_bwd" else 4.0


def mask_aware_flops(w, lens):
    """4*B*H*Lq*Lk*D halved for causal; for kv lengths 4*H*D*Lq*sum(len)
    (10 instead of 4 for the backward)."""
    c = flops_per_pair(w)
    if w.mask & synthetic.MASK_KV_LEN:
        f = c * w.H * w.D * w.Lq * sum(visible_lengths(w, lens))
        return f / 2 if w.mask & synthetic.MASK_CAUSAL else f
    f = c * w.B * w.H * w.Lq * w.Lk * w.D
    return f / 2 if w.mask & synthetic.MASK_CAUSAL else f


def nominal_flops(w):
    return flops_per_pair(w) * w.B * w.H * w.Lq * w.Lk * w.D


def algorithmic_bytes(w, lens):
    """Bytes a perfect kernel moves: Q (or x) and O once, K/V of visible keys
    once.  Backward: q, o, dout, lse read and dq written once; K/V of visible
    keys read once; dk, dv written once for every key."""
    e = 4 if w.dtype == "f32" else 2
    kv_rows = sum(visible_lengths(w, lens)) * w.H
    if w.kind == "mha_bwd":
        rows_q = w.B * w.H * w.Lq
        return (4 * rows_q * w.D * e + 4 * rows_q + 2 * kv_rows * w.D * e
                + 2 * w.B * w.H * w.Lk * w.D * e)
    qo = 2 * w.B * w.H * w.Lq * w.D * e
    extra = 2 * 4 * w.H * w.D if w.kind != "mha" else 0   # gamma, beta
    return qo + 2 * kv_rows * w.D * e + extra


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "_source": "fallback"}


def fp32_alu_peak_tflops(n_sm, mhz):
    """FFMA ceiling: SMs x 128 fp32 lanes x 2 FLOP x clock."""
    return n_sm * 128 * 2 * mhz * 1e6 / 1e12


def source_hash(paths):
    """First 16 hex digits of the SHA-256 of the files' contents, in order."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (the kernel's translation unit and the
    device primitives it includes); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(kernel_key)
        if not rec:
            return None
        srcs = rec.get("sources") or [rec["source"]]
        return rec if source_hash(srcs) == rec["source_sha256_16"] else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is busy."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["sm"] > 0.5 * r["smax"]] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(busy)}


# ------------------------------------------------------------- GPU workload --
class GpuWorkload:
    """Device-resident rotating input sets and the launch of one step."""

    def __init__(self, w, seed, device, l2_bytes, max_bytes=6 << 30):
        import masked_head_attention_gb300 as mha
        self.mha = mha
        self.w = w
        self.host = synthetic.make(w, seed)
        self.lens = None if self.host["kv_lengths"] is None else self.host["kv_lengths"].tolist()
        self.device = device
        keys = {"mha": ["q", "k", "v"], "mha_bwd": ["q", "k", "v", "dout"]}.get(
            w.kind, ["x", "gamma", "beta", "k", "v"])
        self.in_keys = keys
        set_bytes = sum(self.host[k].numel() * self.host[k].element_size() for k in keys)
        out_like = self.host["q"] if w.kind in ("mha", "mha_bwd") else self.host["x"]
        set_bytes += out_like.numel() * out_like.element_size()
        if w.kind == "mha_bwd":   # o and lse (inputs), dq, dk, dv (outputs)
            e = out_like.element_size()
            set_bytes += 2 * out_like.numel() * e + out_like.numel() // w.D * 4 + self.host["k"].numel() * 2 * e
        self.set_bytes = set_bytes
        n = max(1, math.ceil(2 * l2_bytes / set_bytes))
        n = max(1, min(n, max_bytes // set_bytes))
        self.sets = []
        for _ in range(n):
            s = {k: self.host[k].to(device) for k in keys}
            s["out"] = torch.empty_like(out_like, device=device)
            self.sets.append(s)
        self.kv = None if self.host["kv_lengths"] is None else self.host["kv_lengths"].to(device)
        self.i = 0
        if w.kind == "mha_bwd":
            # The forward's output and row statistic are inputs of the backward
            # step; they are formed once, outside any timed region.
            for s in self.sets:
                s["o"], s["lse"] = mha.mha_fwd_lse(s["q"], s["k"], s["v"], w.mask, self.kv,
                                                   scale=w.scale)
                s["dk"] = torch.empty_like(s["k"])
                s["dv"] = torch.empty_like(s["v"])
                need = mha.mha_bwd_workspace_size(w.B, w.H, w.Lq, w.D,
                                                  mha.F32 if w.dtype == "f32" else mha.BF16)
                s["ws"] = torch.empty((max(need, 1),), dtype=torch.uint8, device=device)
            torch.cuda.synchronize()

    def step(self, s=None):
        w = self.w
        if s is None:
            s = self.sets[self.i % len(self.sets)]
            self.i += 1
        if w.kind == "mha":
            self.mha.mha_fwd(s["q"], s["k"], s["v"], w.mask, self.kv, out=s["out"], scale=w.scale)
        elif w.kind == "mha_bwd":   # s["out"] receives dq
            self.mha.mha_bwd(s["q"], s["k"], s["v"], s["o"], s["dout"], s["lse"], w.mask, self.kv,
                             dq=s["out"], dk=s["dk"], dv=s["dv"], scale=w.scale,
                             workspace=s["ws"])
        elif w.kind == "prenorm":
            self.mha.prenorm_cross_attn_fwd(s["x"], s["gamma"], s["beta"], w.eps, s["k"], s["v"],
                                            self.kv, out=s["out"], scale=w.scale)
        else:
            self.mha.prenorm_cross_attn_residual_fwd(s["x"], s["gamma"], s["beta"], w.eps, s["k"],
                                                     s["v"], self.kv, out=s["out"], scale=w.scale)

    def input_bytes(self):
        b = sum(self.host[k].numel() * self.host[k].element_size() for k in self.in_keys)
        if self.host["kv_lengths"] is not None:
            b += self.host["kv_lengths"].numel() * 4
        return b

    def output_bytes(self):
        o = self.sets[0]["out"]
        n = o.numel() * o.element_size()
        if self.w.kind == "mha_bwd":
            n += 2 * self.sets[0]["dk"].numel() * self.sets[0]["dk"].element_size()
        return n


class nvtx_range:
    """An NVTX range around a phase of the run (visible to a profiler's
    timeline); a no-op where NVTX is unavailable."""

    def __init__(self, name):
        self.name = name
        self.pushed = False

    def __enter__(self):
        try:
            torch.cuda.nvtx.range_push(self.name)
            self.pushed = True
        except Exception:
            pass
        return self

    def __exit__(self, *a):
        if self.pushed:
            try:
                torch.cuda.nvtx.range_pop()
            except Exception:
                pass


def time_steps(wl, steps, warmup, sync_ranks=None):
    """Warm up, then time exactly `steps` back-to-back steps between two CUDA
    events on the launching stream; returns the total in ms.

    No events are recorded between the steps: a pair around every step adds
    about 4.4 us of device time to each (measured on GB300 for every workload),
    which is no part of the work.  Every step is one launch of the workload's
    kernel (the backward: the row pass and the main kernel), so total / steps
    is the average launch duration the roofline uses."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    if sync_ranks:
        sync_ranks()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with nvtx_range("timed %d steps: %s" % (steps, wl.w.name)):
        t0.record(stream)
        for _ in range(steps):
            wl.step()
        t1.record(stream)
        torch.cuda.synchronize()
    if sync_ranks:
        sync_ranks()
    return t0.elapsed_time(t1)


def time_e2e(wl, steps, warmup):
    """Same metric through the public API with pinned host buffers: each step
    copies its inputs host->device, runs the call and reads the output back.
    Self-attention workloads use the host-tensor entry point (mha_fwd_host),
    which overlaps the copies of successive pieces with the kernels; the
    others copy with torch around the device call.  Returns (ms per step,
    description of the path)."""
    w = wl.w
    host = {k: wl.host[k].pin_memory() for k in wl.in_keys}
    kv_host = None if wl.host["kv_lengths"] is None else wl.host["kv_lengths"].pin_memory()
    s = wl.sets[0]
    out_host = torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory()
    if w.kind == "mha":
        mha = wl.mha
        B, H, Lq, D = host["q"].shape
        Lk = host["k"].shape[2]
        dt = mha.BF16 if host["q"].dtype == torch.bfloat16 else mha.F32
        ws = torch.empty((max(mha.mha_fwd_host_workspace_size(B, H, Lq, Lk, D, dt), 1),),
                         dtype=torch.uint8, device=s["out"].device)
        path = "mha_fwd_host: pieces of heads through two device slots, copies overlapped"

        def one():
            mha.mha_fwd_host(host["q"], host["k"], host["v"], w.mask, kv_host, out=out_host,
                             scale=w.scale, workspace=ws)
    else:
        path = "torch copies around the device call"

        def one():
            for k in wl.in_keys:
                s[k].copy_(host[k], non_blocking=True)
            if kv_host is not None:
                wl.kv.copy_(kv_host, non_blocking=True)
            wl.step(s)
            out_host.copy_(s["out"], non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with nvtx_range("e2e %d steps: %s" % (steps, w.name)):
        a.record()
        for _ in range(steps):
            one()
        b.record()
        torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, path


def roofline_for(w, lens, kernel_ms, peaks, n_sm):
    """The binding roofline of the workload's dominant kernel: compute (FFMA
    for fp32 inputs on CUDA cores; the tensor cores for bf16 and for fp32 on
    the 3xTF32 path) or HBM, whichever takes longer for the algorithmic
    work; achieved and peak in that roofline's unit (TFLOP/s or GB/s).

    Only the method's own work counts: 4*D FLOP per (row, visible key) of
    the forward (10*D for the backward) and the algorithmic bytes.  The
    3xTF32 kernel executes three tf32 MMAs per product to emulate fp32; that
    emulation is overhead, not work, so its compute roof is the method's
    FLOPs against the tf32 peak, and `tensor_issue_frac` reports separately
    how busy the three MMAs keep the tf32 pipe."""
    flops = mask_aware_flops(w, lens)
    nbytes = algorithmic_bytes(w, lens)
    kkey = kernel_of(w)
    extra = {}
    if uses_tf32x3(w):
        cpeak = peaks["bf16_tflops"] * TF32_OVER_BF16
        cbound, csrc = "tensor", " bf16 burst x 1.1/2.25 (tf32)"
        extra["tensor_issue_frac"] = round(3 * flops / (kernel_ms * 1e-3) / 1e12 / cpeak, 4)
    elif w.dtype == "f32":
        cpeak = fp32_alu_peak_tflops(n_sm, peaks.get("sm_max_mhz", 2070.0))
        cbound, csrc = "alu", " (SMs x 128 lanes x 2 x max SM clock)"
    else:
        cpeak = peaks["bf16_tflops"]
        cbound, csrc = "tensor", " bf16 burst"
    rec = traffic_record("%s/%s" % (kkey, w.name))
    t_compute = flops / (cpeak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_hbm > t_compute:
        achieved = nbytes / (kernel_ms * 1e-3) / 1e9
        bound, unit, peak, psrc = "hbm", "GB/s", peaks["hbm_gbs"], " HBM copy"
    else:
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        bound, unit, peak, psrc = cbound, "TFLOP/s", cpeak, csrc
    out = {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 1),
           "unit": unit, "frac": round(achieved / peak, 4),
           "traffic": None if rec is None else rec["dram_bytes_per_launch"],
           "algorithmic_bytes": int(nbytes),
           "kernel": kkey, "peak_source": peaks["_source"] + psrc}
    out.update(extra)
    return out


# --------------------------------------------------------------- CPU oracle --
def row_visible_keys(w, lens):
    """Visible keys of every query row, [B, Lq] (the same for every head)."""
    vl = np.array(visible_lengths(w, lens), np.int64)[:, None]
    if w.mask & synthetic.MASK_CAUSAL:
        return np.minimum(vl, np.arange(1, w.Lq + 1, dtype=np.int64)[None, :])
    return np.repeat(vl, w.Lq, axis=1)


def sample_rows_even(w, lens, target_flops, offset=0):
    """(b, h, i) rows spread evenly over the whole workload (every `stride`-th
    row of the flattened [B, H, Lq] index, starting at `offset`), about
    `target_flops` of mask-aware work.  Returns (rows [n, 3], exact FLOPs)."""
    vis = row_visible_keys(w, lens)
    total = mask_aware_flops(w, lens)
    n_all = w.B * w.H * w.Lq
    stride = max(1, int(round(total / max(target_flops, 1.0))))
    idx = np.arange(offset % stride, n_all, stride, dtype=np.int64)
    b, rem = np.divmod(idx, w.H * w.Lq)
    h, i = np.divmod(rem, w.Lq)
    rows = np.stack([b, h, i], axis=1)
    # The sample's share of the exact work, in the metric's own count (which
    # halves the causal work rather than counting L(L+1)/2 pairs).
    share = float(vis[b, i].sum()) / (w.H * float(vis.sum())) if vis.sum() > 0 else 0.0
    return rows, mask_aware_flops(w, lens) * share


class OracleRunner:
    """The fp64 oracle, as it stands, on the workload's host tensors (upcast
    once, outside any timing).  A step is an evenly spread sample of rows
    (self-attention and Pre-LN) or of whole (b, h) problems (backward), so
    its OpenMP loop keeps every host thread busy."""

    def __init__(self, w, host):
        import oracle
        self.oracle = oracle
        self.w = w
        self.host = host
        self.threads = oracle.num_threads()
        self.lens = None if host["kv_lengths"] is None else host["kv_lengths"].numpy()
        self.lens_list = None if self.lens is None else self.lens.tolist()
        f64 = lambda t: t.double().numpy()   # noqa: E731
        if w.kind == "mha":
            self.q, self.k, self.v = f64(host["q"]), f64(host["k"]), f64(host["v"])
        elif w.kind == "mha_bwd":
            BH = w.B * w.H
            self.q = f64(host["q"]).reshape(BH, 1, w.Lq, w.D)
            self.k = f64(host["k"]).reshape(BH, 1, w.Lk, w.D)
            self.v = f64(host["v"]).reshape(BH, 1, w.Lk, w.D)
            self.g = f64(host["dout"]).reshape(BH, 1, w.Lq, w.D)
            self.plens = None if self.lens is None else np.repeat(self.lens, w.H).astype(np.int32)
        else:
            self.x, self.k, self.v = f64(host["x"]), f64(host["k"]), f64(host["v"])
            self.gamma, self.beta = host["gamma"].double().numpy(), host["beta"].double().numpy()
        self.offset = 0

    def step(self, target_flops):
        """One timed sample; returns (FLOPs, seconds, description)."""
        w, o = self.w, self.oracle
        if w.kind == "mha_bwd":
            BH = w.B * w.H
            per = flops_per_pair(w) * w.D * w.Lq * (w.Lk / 2 if w.mask & synthetic.MASK_CAUSAL
                                                     else w.Lk)
            n = int(min(BH, max(self.threads, round(target_flops / per))))
            p0 = self.offset % BH
            sel = [(p0 + j) % BH for j in range(n)]
            self.offset += n
            lb = None if self.plens is None else self.plens[sel]
            t0 = time.perf_counter()
            o.mha_bwd(self.q[sel], self.k[sel], self.v[sel], self.g[sel], w.mask, lb, w.scale)
            secs = time.perf_counter() - t0
            sub = synthetic.Workload(w.name, w.kind, w.dtype, n, 1, w.Lq, w.Lk, w.D, w.mask)
            return (mask_aware_flops(sub, None if lb is None else lb.tolist()), secs,
                    "%d of %d (b,h) problems" % (n, BH))
        rows, flops = sample_rows_even(w, self.lens_list, target_flops, self.offset)
        self.offset += 1
        t0 = time.perf_counter()
        if w.kind == "mha":
            o.mha_rows(self.q, self.k, self.v, rows, w.mask, self.lens, w.scale)
        else:
            fn = o.prenorm_rows if w.kind == "prenorm" else o.prenorm_residual_rows
            fn(self.x, self.gamma, self.beta, w.eps, self.k, self.v, rows, self.lens, w.scale)
        secs = time.perf_counter() - t0
        return flops, secs, "%d of %d rows spread evenly over all (b,h)" % (
            len(rows), w.B * w.H * w.Lq)


def oracle_sample(w, host, budget_s, step_flops=3e10):
    """Time the fp64 oracle on evenly spread samples of the workload until the
    budget is spent.  Returns (mask-aware TFLOP/s, seconds, description,
    threads)."""
    r = OracleRunner(w, host)
    flops, t_total, desc = 0.0, 0.0, ""
    steps = 0
    while t_total < budget_s:
        f, s, desc = r.step(step_flops)
        flops += f
        t_total += s
        steps += 1
    return flops / t_total / 1e12, t_total, "%d samples of %s" % (steps, desc), r.threads


# -------------------------------------------------------------------- main --
def combine_ranks(total_ms, flops_per_step, steps, world, reduce_max=None):
    """Whole-job throughput of `world` replicas: every rank ran `steps` steps of
    `flops_per_step`; the job time is the slowest rank's.  `reduce_max` turns a
    local float into the max over ranks (identity for one rank).
    Returns (ms_per_step, TFLOP/s)."""
    t = reduce_max(total_ms) if reduce_max is not None else total_ms
    ms = t / steps
    return ms, world * flops_per_step / (ms * 1e-3) / 1e12


def torch_reduce_max(device):
    import torch.distributed as dist

    def f(x):
        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return f


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def run_reference(args, world, rank):
    """The oracle arm: each step is an evenly spread sample of the workload
    (about 3e10 mask-aware FLOP, under a second on 16 host cores)."""
    if rank != 0:
        return
    w = synthetic.WORKLOADS[args.workload]
    host = synthetic.make(w, seed=0)
    r = OracleRunner(w, host)
    vals = []
    for i in range(args.warmup + args.steps):
        f, secs, desc = r.step(3e10)
        if i >= args.warmup:
            vals.append((f / secs / 1e12, secs, desc))
    tf = statistics.median(v[0] for v in vals)
    secs = statistics.median(v[1] for v in vals)
    line = {"metric": METRIC, "impl": "reference", "value": round(tf, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "D": w.D,
                       "note": w.note},
            "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": r.threads,
                             "kind": "oracle", "sample": vals[0][2] + " per step"},
            "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def time_graph(wl, calls, reps=5):
    """Per-call time of `calls` back-to-back steps captured in one CUDA graph
    and replayed (host launch cost removed); median over `reps` replays."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            wl.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            wl.step()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / calls)
    del g
    return statistics.median(times)


def measure_config(w, args, device, peaks, n_sm, l2):
    wl = GpuWorkload(w, 0, device, l2)
    if args.extra_steps > 0:
        steps = args.extra_steps
    else:
        probe_ms = time_steps(wl, 3, 2)
        steps = max(5, min(2000, int(300.0 / max(probe_ms / 3, 1e-3))))
    total_ms = time_steps(wl, steps, max(3, args.warmup))
    call_ms = total_ms / steps
    flops = mask_aware_flops(w, wl.lens)
    r = roofline_for(w, wl.lens, call_ms, peaks, n_sm)
    out = {"us_per_call": round(call_ms * 1e3, 3), "tflops": round(flops / call_ms / 1e9, 3),
           "nominal_tflops": round(nominal_flops(w) / call_ms / 1e9, 3), "steps": steps,
           "roofline": {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                          "tensor_issue_frac") if k in r},
           "hbm_gbs": round(algorithmic_bytes(w, wl.lens) / call_ms / 1e6, 1),
           "input_sets": len(wl.sets)}
    if w.kind in ("prenorm", "prenorm_residual"):
        # Heads per chunk of shared row statistics, cluster pairs, prologue
        # chunks per CTA: the plan the launch used.
        out["launch_plan"] = wl.mha.plan_prenorm(w.B, w.H, w.Lq, w.Lk, w.D, n_sm)
    if call_ms < 0.05:
        # Short calls are bound by the host's launch rate when issued one by
        # one from Python; a CUDA graph of back-to-back calls shows the GPU side.
        g_ms = time_graph(wl, calls=max(64, len(wl.sets) * 2))
        out["graph"] = {"us_per_call": round(g_ms * 1e3, 3),
                        "tflops": round(flops / g_ms / 1e9, 3),
                        "hbm_gbs": round(algorithmic_bytes(w, wl.lens) / g_ms / 1e6, 1),
                        "hbm_frac": round(algorithmic_bytes(w, wl.lens) / g_ms / 1e6
                                          / peaks["hbm_gbs"], 4),
                        "timing": "CUDA graph of back-to-back calls over rotating inputs"}
    del wl
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--no-extra", action="store_true", help="skip the other four workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--extra-steps", type=int, default=0,
                    help="fixed timed steps for the other workloads (0 = about 0.3 s each)")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this batch size instead (profiling captures "
                         "of a smaller case of the same kernel); 0 = the workload's own")
    ap.add_argument("--f32-kernel", type=int, default=0, choices=[0, 1, 2],
                    help="fp32 forward kernel: 0 automatic, 1 tiled CUDA-core kernel, 2 "
                         "short-key-range CUDA-core kernel where it applies (profiling)")
    ap.add_argument("--settle-s", type=float, default=1.0,
                    help="untimed back-to-back steps before the timed region (clock settling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    global F32_KERNEL
    F32_KERNEL = args.f32_kernel
    if args.batch > 0:
        import dataclasses
        w0 = synthetic.WORKLOADS[args.workload]
        synthetic.WORKLOADS[args.workload] = dataclasses.replace(w0, B=args.batch)

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import masked_head_attention_gb300 as mha
    mha.lib()   # fails loudly when the extension is missing
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if F32_KERNEL:
        mha.set_f32_kernel(F32_KERNEL)
    props = torch.cuda.get_device_properties(device)
    n_sm = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 0) or DEFAULT_L2
    peaks = load_peaks()
    w = synthetic.WORKLOADS[args.workload]

    sync = None
    if world > 1:
        import torch.distributed as dist
        sync = dist.barrier

    wl = GpuWorkload(w, seed=rank, device=device, l2_bytes=l2)
    # Settle clocks under this load, then the timed region, with clock samples.
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        t_end = time.time() + args.settle_s
        while time.time() < t_end:
            for _ in range(20):
                wl.step()
            torch.cuda.synchronize()
        total_ms = time_steps(wl, args.steps, args.warmup, sync)
    flops = mask_aware_flops(w, wl.lens)
    ms_per_step, value = combine_ranks(total_ms, flops, args.steps, world,
                                       torch_reduce_max(device) if world > 1 else None)
    # This rank's average launch duration (one launch of the kernel per step).
    kernel_ms = total_ms / args.steps
    roof = roofline_for(w, wl.lens, kernel_ms, peaks, n_sm)

    e2e_ms, e2e_path = time_e2e(wl, max(3, min(args.steps, 50)), 3)
    e2e = {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(wl.input_bytes()),
           "d2h_bytes_per_step": int(wl.output_bytes()), "ms_per_step": round(e2e_ms, 4),
           "path": e2e_path}
    status = mha.device_status()

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
                "us_per_call": round(ms_per_step * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": ("f32 (3xTF32 on tensor cores, fp32 accumulate)" if uses_tf32x3(w)
                          else "f32" if w.dtype == "f32" else "bf16 (fp32 accumulate)"),
                "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk,
                           "D": w.D, "mask": w.mask, "note": w.note,
                           "nominal_tflops": round(world * nominal_flops(w) / ms_per_step / 1e9, 3),
                           "l2_policy": "%d rotating input sets of %.1f MB (> 2x L2 %.0f MB)" % (
                               len(wl.sets), wl.set_bytes / 1e6, l2 / 1e6),
                           "parallelism": "replicas x%d (weak scaling, no collective)" % world,
                           **({"f32_kernel": kernel_of(w)} if F32_KERNEL else {})},
                "roofline": roof, "e2e": e2e, "gpu_launches": args.steps,
                "clocks": clk.summary(), "device_status": status}
        del wl
        torch.cuda.empty_cache()
        if not args.no_cpu_baseline and world == 1:
            host = synthetic.make(w, seed=0)
            tf, secs, desc, thr = oracle_sample(w, host, args.cpu_budget)
            line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": thr,
                                    "kind": "oracle", "sample": "%s, %.1f s" % (desc, secs)}
        if not args.no_extra and world == 1:
            extra = {}
            for name, ow in synthetic.WORKLOADS.items():
                if name == w.name:
                    continue
                extra[name] = measure_config(ow, args, device, peaks, n_sm, l2)
            line["other_workloads"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
