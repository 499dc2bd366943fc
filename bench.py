#!/usr/bin/env python3
"""Benchmark of the AttnRes read operator, forward + backward, on GB300.

Default workload (`--workload long`): one step = attnres_fwd + attnres_bwd
(every step of the hot path: key statistics, softmax routing, weighted read,
output RMSNorm, dot pass, dvalues write, dq/dw_o partial sums and their
finalize) over one batch of the long-sequence workload S=10 sources,
N=32768 tokens, D=4096, bf16, output RMSNorm on (the shape of the first row
of the benchmark table in "[Perf] Parallelize AttnRes long-sequence
reduction", Test plan).

The other rows of that table and the pages' other workloads have their own
lines, each the same contract with its own byte model:
  `--workload short`   S=8, N=8192, D=2048 (the table's last row; narrow
                       rows: two backward CTAs per SM)
  `--workload sliced`  the Block schedule's sliced read: 8 block sums + the
                       partial sum (S=9), N=16384, D=4096, R=1024, 2% zero
                       rows; one step reads with the key in the first R
                       channels and again with it in the final R channels
                       ("Fast Attention Residuals", sections "Full and Block
                       schedules" and "Sliced LR-AttnRes")
  `--workload deep`    S=64, N=8192, D=8192, output RMSNorm on (the table's
                       third row; 8.6 GB of sources)
  `--workload multi`   attnres_multi_fwd + attnres_multi_bwd with M=2
                       queries of rank R=1024 over the long workload's
                       sources ("Fast Attention Residuals", section
                       "Multi-query AttnRes": two queries route two roles
                       from one read)
  `--workload selected`  per-token queries from an 8-row bank, K=2 slots
  `--workload block`   the fused block-partial read

The metric is effective HBM bandwidth: the algorithmic bytes one step must
move (sources read in the forward and again in the backward, dvalues
written, outputs written, upstream gradients read, saved statistics and the
FP32 partial sums) divided by the measured step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long|short|sliced|deep|multi|selected|block]

Prints ONE JSON line on rank 0.  With --gpus N > 1 run it under
torch.distributed.run: every rank processes its own full batch (weak
scaling, data parallel) and each step ends with the one exchange the method
has, the sum of the FP32 dq (and dw_o) over ranks (an all-reduce of R + D
floats).  --impl reference times the FP64 CPU oracle on the host cores
instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AttnRes fwd+bwd ms and effective HBM GB/s (% of roofline), bf16, 1×GB300"
WORKLOAD_CFG = 3
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e data-sheet bandwidth (context for the measured-peak fraction)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attnres_bwd_traffic.json")
PROFILE_TRAFFIC_MULTI = os.path.join(ROOT, "profiles", "attnres_multi_bwd_traffic.json")
PROFILE_TRAFFIC_MULTI16 = os.path.join(ROOT, "profiles", "attnres_multi16_bwd_traffic.json")
PROFILE_TRAFFIC_SELECTED = os.path.join(ROOT, "profiles", "attnres_selected_bwd_traffic.json")
PROFILE_TRAFFIC_BLOCK = os.path.join(ROOT, "profiles", "attnres_block_bwd_traffic.json")


# --------------------------------------------------------------------------
# Byte model
# --------------------------------------------------------------------------
def algorithmic_bytes(S, N, D, R, out_norm, P, o_pre=False):
    """Bytes each kernel must move (bf16 = 2 B, fp32 = 4 B): the forward reads
    the sources and writes y plus the per-token statistics; the backward reads
    the sources again, reads dy and the statistics, writes dvalues and moves
    the FP32 partial sums of dq/dw_o (P rows written, then read).  With
    o_pre, the forward also writes the FP32 pre-norm mixture and the
    backward reads it (what the plan does when a token's rows cannot stay
    on chip through the backward)."""
    v = S * N * D * 2
    row = N * D * 2
    stats = 3 * N * S * 4 + (N * 4 if out_norm else 0)
    opre = N * D * 4 if (out_norm and o_pre) else 0
    fwd = v + row + stats + opre
    W = R + (D if out_norm else 0)
    bwd = 2 * v + row + stats + 2 * P * W * 4 + opre
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}


def multi_algorithmic_bytes(S, N, D, R, M, P):
    """Multi-query read: the forward reads the sources once for all M
    queries and writes M outputs plus alpha/logit [N, M, S] and rstd [N, S];
    the backward reads the sources, the M upstream gradients and the
    statistics, writes dvalues and moves the [P, M*R] FP32 partial sums."""
    v = S * N * D * 2
    out = M * N * D * 2
    stats = (2 * M * S + S) * N * 4
    fwd = v + out + stats
    bwd = 2 * v + out + stats + 2 * P * M * R * 4
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}


SINGLE_SOURCES = ["attnres_api.cu", "attnres_bwd.cu", "attnres_bwd_cluster.cu", "attnres_bwd_kernel.cuh",
                  "attnres_bwd_norm.cu", "attnres_bwd_opre.cu", "attnres_fwd.cu", "attnres_fwd_kernel.cuh",
                  "attnres_jit.cu", "device_utils.cuh", "kernels.cuh"]
MULTI_SOURCES = ["attnres_api.cu", "attnres_bwd.cu", "attnres_bwd_kernel.cuh", "attnres_jit.cu",
                 "attnres_multi_bwd.cu", "attnres_multi_fwd.cu", "attnres_multi_fwd_kernel.cuh", "device_utils.cuh",
                 "kernels.cuh"]
# the sixteen-query read: the tensor-core forward and the general backward
GENERAL_SOURCES = MULTI_SOURCES + ["attnres_multi_fwd_mma.cu", "attnres_multi_general.cu", "attnres_multi_grad_mma.cu"]


def kernel_sources_hash(names=None):
    """Hash of the kernel sources a profile was captured from (the
    single-query kernels and what they compile from, by default)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_residuals_gb300", "csrc")
    for name in (names or SINGLE_SOURCES):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs", "hbm"):
            if key in peaks and isinstance(peaks[key], (int, float)):
                return float(peaks[key]), "measured"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(config_key, path=PROFILE_TRAFFIC, names=None):
    """DRAM bytes per backward launch from the committed ncu summary, only if
    the kernel sources are unchanged since that capture."""
    try:
        with open(path) as f:
            doc = json.load(f)
        if doc.get("sources_hash") == kernel_sources_hash(names) and doc.get("config") == config_key:
            return doc.get("traffic_bytes_per_launch")
    except Exception:
        pass
    return None


# --------------------------------------------------------------------------
# Clock sampling during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or 1e30)]
        used = inside if inside else rows[-3:]
        sm = [float(p[1]) for _, p in used if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in used if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in used:
            for k, name in enumerate(names):
                if p[4 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples_in_window": len(inside)}


# --------------------------------------------------------------------------
# Distributed helpers
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------
# Workloads: what one step runs, its bytes, its end-to-end variant and its
# oracle (the CPU baseline and the reference arm)
# --------------------------------------------------------------------------
class SingleRead:
    """Single-query read of one of the pages' workloads (seeded synthetic
    inputs, attention_residuals_gb300.workloads).  One step = the forward and
    backward for every key offset in `key_offsets` (two reads of the same
    sources for the sliced workload)."""
    key = "long"
    cfg = 3
    key_offsets = (0,)
    label = "long-sequence"
    roofline_kernel = "attnres_bwd_kernel (+ finalize)"
    traffic_path = PROFILE_TRAFFIC
    traffic_key = "cfg3"
    e2e_chunk = 8192      # tokens per chunk of the host-buffer step
    cpu_tokens = 8192     # oracle sample for the CPU baseline
    ref_tokens = 1024     # oracle sample per reference-arm step

    def __init__(self, tokens=None, seed=0, device="cpu"):
        from attention_residuals_gb300.workloads import make_workload
        wl = make_workload(self.cfg, N=tokens, seed=self.cfg + 1000 * seed, device=device)
        self.wls = [dataclasses.replace(wl, key_offset=ko) for ko in self.key_offsets]
        self.wl = self.wls[0]
        self.o_pre = False

    def bytes_for(self, P):
        tot = {"fwd": 0, "bwd": 0, "total": 0}
        for wl in self.wls:
            b = algorithmic_bytes(wl.S, wl.N, wl.D, wl.R, wl.out_norm, P, self.o_pre)
            for k in tot:
                tot[k] += b[k]
        return tot

    def describe(self):
        wl = self.wl
        ko = "/".join(str(w.key_offset) for w in self.wls)
        return (f"S={wl.S} N={wl.N} D={wl.D} R={wl.R} key_offset={ko}{' out-norm' if wl.out_norm else ''} "
                f"bf16 ({self.label})")

    # ---------------------------------------------------------------- GPU
    def prepare(self, dev):
        import torch
        from attention_residuals_gb300 import attnres_plan_info
        wl = self.wl
        S, N, D, R = wl.S, wl.N, wl.D, wl.R
        self.infos = [attnres_plan_info(w.values, R, key_offset=w.key_offset, out_norm=w.out_norm)
                      for w in self.wls]
        self.info = self.infos[0]
        self.o_pre = bool(wl.out_norm and not self.info["bwd_resident"])
        self.bytes = self.bytes_for(self.info["grid"])
        f32 = dict(dtype=torch.float32, device=dev)
        self.outs = []
        for _ in self.wls:
            o = {"y": torch.empty((N, D), dtype=torch.bfloat16, device=dev),
                 "alpha": torch.empty((N, S), **f32), "rstd": torch.empty((N, S), **f32),
                 "logit": torch.empty((N, S), **f32)}
            if wl.out_norm:
                o["o_rstd"] = torch.empty((N,), **f32)
                if self.o_pre:
                    o["o_pre"] = torch.empty((N, D), **f32)
            self.outs.append(o)
        self.dv = torch.empty_like(wl.values)
        self.ws = torch.empty((64 << 20,), dtype=torch.uint8, device=dev)
        self.launches = sum(2 + (1 if i["bwd_split"] else 0) for i in self.infos)
        self.f = [None] * len(self.wls)

    def fwd(self, stream, values=None, q=None, w=None):
        from attention_residuals_gb300 import attnres_fwd
        for i, wl in enumerate(self.wls):
            self.f[i] = attnres_fwd(wl.values if values is None else values, wl.q if q is None else q,
                                    w_o=wl.w_o if w is None else w, key_offset=wl.key_offset, out=self.outs[i],
                                    save_o_pre=self.o_pre, stream=stream)
        return self.f

    def bwd(self, stream, values=None, q=None, w=None, dy=None):
        from attention_residuals_gb300 import attnres_bwd
        res = None
        for i, wl in enumerate(self.wls):
            res = attnres_bwd(wl.values if values is None else values, wl.q if q is None else q,
                              wl.dy if dy is None else dy, self.f[i], w_o=wl.w_o if w is None else w,
                              key_offset=wl.key_offset, workspace=self.ws, dvalues=self.dv, stream=stream)
        return res

    def grads(self, res):
        """The step's FP32 reduced gradients (what data parallelism sums over ranks)."""
        return [res["dq_f32"], res.get("dw_o_f32")]

    def e2e(self, stream, chunk_tokens=None):
        """A step through the C ABI's host-buffer call (attnres_step_host):
        sources, query, weight and dy in page-locked host memory, y,
        dvalues, dq and dw_o copied back to it, transfers overlapped with
        the kernels chunk by chunk (once per key offset)."""
        import torch
        from attention_residuals_gb300 import attnres_step_host
        chunk_tokens = chunk_tokens or self.e2e_chunk
        wl = self.wl
        v, q, w, dy = wl.values, wl.q, wl.w_o, wl.dy
        S, N, D, R = wl.S, wl.N, wl.D, wl.R
        pin = dict(pin_memory=True)
        h = {"v": torch.empty(v.shape, dtype=v.dtype, **pin), "q": q.cpu().pin_memory(),
             "w": None if w is None else w.cpu().pin_memory(),
             "dy": torch.empty(dy.shape, dtype=dy.dtype, **pin)}
        h["v"].copy_(v)
        h["dy"].copy_(dy)
        out = {"y": torch.empty((N, D), dtype=torch.bfloat16, **pin),
               "dvalues": [torch.empty((N, D), dtype=torch.bfloat16, **pin) for _ in range(S)],
               "dq": torch.empty((R,), dtype=torch.bfloat16, **pin),
               "dq_f32": torch.empty((R,), dtype=torch.float32, **pin)}
        if w is not None:
            out["dw_o"] = torch.empty((D,), dtype=torch.bfloat16, **pin)
            out["dw_o_f32"] = torch.empty((D,), dtype=torch.float32, **pin)
        ws = {}

        def step():
            for x in self.wls:
                r = attnres_step_host(h["v"], h["q"], h["dy"], w_o=h["w"], key_offset=x.key_offset,
                                      chunk_tokens=chunk_tokens, out=out, workspace=ws.get("t"))
                ws["t"] = r["workspace"]

        reads = len(self.wls)
        wd = 0 if w is None else D
        h2d = reads * (v.numel() + dy.numel() + R + wd) * 2
        d2h = reads * ((N * D + S * N * D + R + wd) * 2 + (R + wd) * 4)
        self.e2e_detail = {"api": "attnres_step_host (C ABI, host buffers)", "chunk_tokens": chunk_tokens}
        return step, h2d, d2h, (h, out, ws)

    def traffic(self):
        return profiled_traffic(self.traffic_key, self.traffic_path)

    # ---------------------------------------------------------------- CPU
    def oracle_seconds(self, cores):
        from oracle import attnres_oracle
        t = time.perf_counter()
        for wl in self.wls:
            attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=wl.key_offset,
                           nthreads=cores, want_dvalues=True)
        return time.perf_counter() - t


class LongRead(SingleRead):
    """S=10, N=32768, D=4096, output RMSNorm on: the split-N reduction path."""


class ShortRead(SingleRead):
    """S=8, N=8192, D=2048: narrow rows, two backward CTAs per SM."""
    key = "short"
    cfg = 2
    label = "short"
    roofline_kernel = "attnres_bwd_kernel (+ finalize)"
    traffic_path = os.path.join(ROOT, "profiles", "attnres_short_bwd_traffic.json")
    traffic_key = "cfg2"


class SlicedRead(SingleRead):
    """The Block schedule's sliced low-rank read: R = D/4 = 1024 key channels,
    read once with the key in the first R channels and once in the final R."""
    key = "sliced"
    cfg = 4
    key_offsets = (0, 3072)
    label = "sliced block schedule, 8 block sums + partial, 2% zero rows, both key placements"
    roofline_kernel = "attnres_bwd_kernel x2 (+ finalize)"
    traffic_path = os.path.join(ROOT, "profiles", "attnres_sliced_bwd_traffic.json")
    traffic_key = "cfg4"


class DeepRead(SingleRead):
    """S=64, N=8192, D=8192, output RMSNorm on: a token's rows are 1 MB."""
    key = "deep"
    cfg = 5
    label = "deep"
    roofline_kernel = "attnres_bwd_kernel (+ finalize)"
    traffic_path = os.path.join(ROOT, "profiles", "attnres_deep_bwd_traffic.json")
    traffic_key = "cfg5"
    e2e_chunk = 1024
    cpu_tokens = 512
    ref_tokens = 64


class MultiRead:
    """Multi-query read: two rank-1024 queries over the long-sequence sources."""
    key = "multi"
    roofline_kernel = "attnres_multi_bwd_kernel (+ finalize)"

    def __init__(self, tokens=None, seed=0, device="cpu"):
        from attention_residuals_gb300.workloads import make_multi_workload
        self.wl = make_multi_workload("long", N=tokens, seed=200 + 1000 * seed, device=device)

    def bytes_for(self, P):
        wl = self.wl
        return multi_algorithmic_bytes(wl.S, wl.N, wl.D, wl.R, wl.M, P)

    def describe(self):
        wl = self.wl
        return (f"multi-query M={wl.M} S={wl.S} N={wl.N} D={wl.D} R={wl.R} key_offset={wl.key_offset} "
                f"bf16 (two queries over the long-sequence sources)")

    # ---------------------------------------------------------------- GPU
    def prepare(self, dev):
        import torch
        from attention_residuals_gb300 import attnres_multi_plan_info
        wl = self.wl
        self.info = attnres_multi_plan_info(wl.values, wl.M, wl.R, key_offset=wl.key_offset)
        self.bytes = self.bytes_for(self.info["grid"] % 1000)
        self.ws = torch.empty((64 << 20,), dtype=torch.uint8, device=dev)
        self.launches = 3
        self.f = None

    def fwd(self, stream, values=None, queries=None):
        from attention_residuals_gb300 import attnres_multi_fwd
        wl = self.wl
        self.f = attnres_multi_fwd(wl.values if values is None else values,
                                   wl.queries if queries is None else queries,
                                   key_offset=wl.key_offset, stream=stream)
        return self.f

    def bwd(self, stream, values=None, queries=None, dy=None):
        from attention_residuals_gb300 import attnres_multi_bwd
        wl = self.wl
        return attnres_multi_bwd(wl.values if values is None else values,
                                 wl.queries if queries is None else queries,
                                 wl.dy if dy is None else dy, self.f, key_offset=wl.key_offset,
                                 stream=stream, workspace=self.ws)

    def e2e(self, stream):
        import torch
        wl = self.wl
        v, Q, dy = wl.values, wl.queries, wl.dy
        h = {"v": torch.empty(v.shape, dtype=v.dtype, pin_memory=True), "q": Q.cpu().pin_memory(),
             "dy": torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True),
             "y": torch.empty(dy.shape, dtype=torch.bfloat16, pin_memory=True),
             "dv": torch.empty(v.shape, dtype=v.dtype, pin_memory=True),
             "dq": torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=True)}
        h["v"].copy_(v)
        h["dy"].copy_(dy)
        d = {"v": torch.empty_like(v), "q": torch.empty_like(Q), "dy": torch.empty_like(dy)}

        def step():
            for k in ("v", "q", "dy"):
                d[k].copy_(h[k], non_blocking=True)
            f = self.fwd(stream, d["v"], d["q"])
            b = self.bwd(stream, d["v"], d["q"], d["dy"])
            h["y"].copy_(f["y"], non_blocking=True)
            h["dv"].copy_(b["dvalues"], non_blocking=True)
            h["dq"].copy_(b["dq"], non_blocking=True)

        h2d = sum(h[k].numel() for k in ("v", "q", "dy")) * 2
        d2h = sum(h[k].numel() for k in ("y", "dv", "dq")) * 2
        return step, h2d, d2h, h

    def grads(self, res):
        return [res["dq_f32"]]

    def traffic(self):
        return profiled_traffic("multi-long", PROFILE_TRAFFIC_MULTI, MULTI_SOURCES)

    # ---------------------------------------------------------------- CPU
    def oracle_seconds(self, cores):
        from oracle.multi import attnres_multi_oracle
        wl = self.wl
        t = time.perf_counter()
        attnres_multi_oracle(wl.values, wl.queries, dy=wl.dy, key_offset=wl.key_offset,
                             nthreads=cores, want_dvalues=True)
        return time.perf_counter() - t


class Multi16Read(MultiRead):
    """Multi-query read with the most queries the page allows: sixteen
    full-rank queries over 1024-channel rows (the tensor-core forward; the
    general backward -- coefficient kernel, then the tensor-core gradient
    kernel -- whose sources and dy are read twice, though the algorithmic
    bytes count them once)."""
    key = "multi16"
    roofline_kernel = "attnres_multi_coef_kernel + attnres_multi_grad_mma_kernel (+ finalize)"
    cpu_tokens = 4096
    ref_tokens = 512

    def __init__(self, tokens=None, seed=0, device="cpu"):
        from attention_residuals_gb300.workloads import make_multi_workload
        self.wl = make_multi_workload("sixteen", N=tokens, seed=300 + 1000 * seed, device=device)

    def describe(self):
        wl = self.wl
        return (f"multi-query M={wl.M} S={wl.S} N={wl.N} D={wl.D} R={wl.R} key_offset={wl.key_offset} "
                f"bf16 (sixteen full-rank queries)")

    def prepare(self, dev):
        import torch
        from attention_residuals_gb300 import attnres_multi_plan_info
        wl = self.wl
        self.info = attnres_multi_plan_info(wl.values, wl.M, wl.R, key_offset=wl.key_offset)
        # the general form's partial rows: one per token group
        self.bytes = self.bytes_for(self.info["bwd_token_groups"])
        self.ws = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
        self.launches = 4
        self.f = None

    def traffic(self):
        return profiled_traffic("multi16", PROFILE_TRAFFIC_MULTI16, GENERAL_SOURCES)


def selected_algorithmic_bytes(S, N, D, R, K, E, P):
    """Selected-query read: as the multi-query read with K slots per token,
    plus the ids [N, K] (int64) read by both kernels and the [P, E*R] FP32
    bank-gradient partial rows."""
    b = multi_algorithmic_bytes(S, N, D, R, K, 0)
    ids = N * K * 8
    return {"fwd": b["fwd"] + ids, "bwd": b["bwd"] + ids + 2 * P * E * R * 4,
            "total": b["fwd"] + b["bwd"] + 2 * ids + 2 * P * E * R * 4}


def block_algorithmic_bytes(S, N, D, R, P):
    """Fused block-partial read, S sources counting the partial sum: the
    forward reads S-1 completed sources, the previous partial and delta, and
    writes the new partial, y and the statistics; the backward reads the S
    sources (the new partial among them), dy and the new partial's extra
    gradient, and writes dvalues."""
    row = N * D * 2
    stats = 3 * N * S * 4
    fwd = (S + 1) * row + 2 * row + stats
    bwd = 2 * S * row + 2 * row + stats + 2 * P * R * 4
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}


class SelectedRead(MultiRead):
    """Selected-query read: an 8-row query bank, two slots per token, over
    the long-sequence sources."""
    key = "selected"
    roofline_kernel = "attnres_multi_bwd_kernel with a query bank (+ finalize)"

    def __init__(self, tokens=None, seed=0, device="cpu"):
        from attention_residuals_gb300.workloads import make_selected
        self.wl = make_selected(10, 32768 if tokens is None else tokens, 4096, 1024, 8, 2,
                                seed=300 + 1000 * seed, src_scale=(0.5, 2.0), device=device)

    def bytes_for(self, P):
        wl = self.wl
        return selected_algorithmic_bytes(wl.S, wl.N, wl.D, wl.R, wl.K, wl.E, P)

    def describe(self):
        wl = self.wl
        return (f"selected-query K={wl.K} E={wl.E} S={wl.S} N={wl.N} D={wl.D} R={wl.R} "
                f"key_offset={wl.key_offset} bf16 (bank of 8 queries over the long-sequence sources)")

    def prepare(self, dev):
        import torch
        from attention_residuals_gb300 import attnres_multi_plan_info
        wl = self.wl
        self.info = attnres_multi_plan_info(wl.values, wl.K, wl.R, key_offset=wl.key_offset)
        self.bytes = self.bytes_for(self.info["grid"] % 1000)
        self.ws = torch.empty((64 << 20,), dtype=torch.uint8, device=dev)
        self.launches = 3
        self.f = None

    def fwd(self, stream, values=None, bank=None, ids=None):
        from attention_residuals_gb300 import attnres_selected_fwd
        wl = self.wl
        self.f = attnres_selected_fwd(wl.values if values is None else values, wl.bank if bank is None else bank,
                                      wl.ids if ids is None else ids, key_offset=wl.key_offset, stream=stream)
        return self.f

    def bwd(self, stream, values=None, bank=None, ids=None, dy=None):
        from attention_residuals_gb300 import attnres_selected_bwd
        wl = self.wl
        return attnres_selected_bwd(wl.values if values is None else values, wl.bank if bank is None else bank,
                                    wl.ids if ids is None else ids, wl.dy if dy is None else dy, self.f,
                                    key_offset=wl.key_offset, stream=stream, workspace=self.ws)

    def e2e(self, stream):
        import torch
        wl = self.wl
        h = {"v": torch.empty(wl.values.shape, dtype=torch.bfloat16, pin_memory=True),
             "bank": wl.bank.cpu().pin_memory(), "ids": wl.ids.cpu().pin_memory(),
             "dy": torch.empty(wl.dy.shape, dtype=torch.bfloat16, pin_memory=True),
             "y": torch.empty(wl.dy.shape, dtype=torch.bfloat16, pin_memory=True),
             "dv": torch.empty(wl.values.shape, dtype=torch.bfloat16, pin_memory=True),
             "db": torch.empty(wl.bank.shape, dtype=torch.bfloat16, pin_memory=True)}
        h["v"].copy_(wl.values)
        h["dy"].copy_(wl.dy)
        d = {k: torch.empty_like(getattr(wl, n)) for k, n in (("v", "values"), ("bank", "bank"), ("ids", "ids"),
                                                                ("dy", "dy"))}

        def step():
            for k in ("v", "bank", "ids", "dy"):
                d[k].copy_(h[k], non_blocking=True)
            f = self.fwd(stream, d["v"], d["bank"], d["ids"])
            b = self.bwd(stream, d["v"], d["bank"], d["ids"], d["dy"])
            h["y"].copy_(f["y"], non_blocking=True)
            h["dv"].copy_(b["dvalues"], non_blocking=True)
            h["db"].copy_(b["dbank"], non_blocking=True)

        h2d = (h["v"].numel() + h["bank"].numel() + h["dy"].numel()) * 2 + h["ids"].numel() * 8
        d2h = (h["y"].numel() + h["dv"].numel() + h["db"].numel()) * 2
        return step, h2d, d2h, (h, d)

    def grads(self, res):
        return [res["dbank_f32"]]

    def traffic(self):
        return profiled_traffic("selected-long", PROFILE_TRAFFIC_SELECTED, MULTI_SOURCES)

    def oracle_seconds(self, cores):
        from oracle.multi import attnres_selected_oracle
        wl = self.wl
        t = time.perf_counter()
        attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=wl.key_offset,
                                nthreads=cores, want_dvalues=True)
        return time.perf_counter() - t


class BlockRead:
    """Block-schedule read with the partial-block sum fused in: eight
    completed block sums and the running partial sum (S=9 sources), the
    newest writer output added inside the read, sliced key R=1024."""
    key = "block"
    roofline_kernel = "attnres_bwd_kernel with the added gradient (+ finalize)"

    def __init__(self, tokens=None, seed=0, device="cpu"):
        import torch
        from attention_residuals_gb300.workloads import make_workload
        wl = make_workload(4, N=tokens, seed=400 + 1000 * seed, device=device)
        self.wl = wl
        self.completed = wl.values[:-1]
        self.partial = wl.values[-1]
        g = torch.Generator(device=device)
        g.manual_seed(401 + 1000 * seed)
        self.delta = torch.randn(self.partial.shape, generator=g, device=device).to(torch.bfloat16)
        self.gp = torch.randn(self.partial.shape, generator=g, device=device).to(torch.bfloat16)

    def bytes_for(self, P):
        wl = self.wl
        return block_algorithmic_bytes(wl.S, wl.N, wl.D, wl.R, P)

    def describe(self):
        wl = self.wl
        return (f"block schedule S={wl.S} (8 completed block sums + the partial sum, delta added in the "
                f"read) N={wl.N} D={wl.D} R={wl.R} key_offset={wl.key_offset} bf16")

    def prepare(self, dev):
        import torch
        from attention_residuals_gb300 import attnres_plan_info
        wl = self.wl
        self.comp = list(self.completed.unbind(0))
        self.info = attnres_plan_info(wl.values, wl.R, key_offset=wl.key_offset, out_norm=False)
        self.bytes = self.bytes_for(self.info["grid"])
        self.pout = torch.empty_like(self.partial)
        self.launches = 2 + (1 if self.info["bwd_split"] else 0)
        self.f = None

    def fwd(self, stream):
        from attention_residuals_gb300 import attnres_partial_fwd
        self.f = attnres_partial_fwd(self.comp, self.partial, self.delta, self.wl.q, key_offset=self.wl.key_offset,
                                     partial_out=self.pout, stream=stream)
        return self.f

    def bwd(self, stream):
        from attention_residuals_gb300 import attnres_partial_bwd
        return attnres_partial_bwd(self.comp, self.pout, self.wl.q, self.wl.dy, self.f, g_partial=self.gp,
                                   key_offset=self.wl.key_offset, stream=stream)

    def e2e(self, stream):
        import torch
        wl = self.wl
        pin = dict(dtype=torch.bfloat16, pin_memory=True)
        h = {"c": torch.empty(self.completed.shape, **pin), "p": torch.empty(self.partial.shape, **pin),
             "d": torch.empty(self.partial.shape, **pin), "dy": torch.empty(wl.dy.shape, **pin),
             "g": torch.empty(self.partial.shape, **pin), "y": torch.empty(wl.dy.shape, **pin),
             "pn": torch.empty(self.partial.shape, **pin), "dc": torch.empty(self.completed.shape, **pin),
             "dp": torch.empty(self.partial.shape, **pin)}
        h["c"].copy_(self.completed)
        h["p"].copy_(self.partial)
        h["d"].copy_(self.delta)
        h["dy"].copy_(wl.dy)
        h["g"].copy_(self.gp)
        d = {k: torch.empty_like(h[k], device=stream.device) for k in ("c", "p", "d", "dy", "g")}
        from attention_residuals_gb300 import attnres_partial_bwd, attnres_partial_fwd

        def step():
            for k in ("c", "p", "d", "dy", "g"):
                d[k].copy_(h[k], non_blocking=True)
            comp = list(d["c"].unbind(0))
            f = attnres_partial_fwd(comp, d["p"], d["d"], wl.q, key_offset=wl.key_offset, stream=stream)
            b = attnres_partial_bwd(comp, f["partial_new"], wl.q, d["dy"], f, g_partial=d["g"],
                                    key_offset=wl.key_offset, stream=stream)
            h["y"].copy_(f["y"], non_blocking=True)
            h["pn"].copy_(f["partial_new"], non_blocking=True)
            h["dc"].copy_(torch.stack(b["d_completed"]), non_blocking=True)
            h["dp"].copy_(b["d_partial"], non_blocking=True)

        h2d = sum(h[k].numel() for k in ("c", "p", "d", "dy", "g")) * 2
        d2h = sum(h[k].numel() for k in ("y", "pn", "dc", "dp")) * 2
        return step, h2d, d2h, (h, d)

    def grads(self, res):
        return [res["dq_f32"], res.get("dw_o_f32")]

    def traffic(self):
        return profiled_traffic("block", PROFILE_TRAFFIC_BLOCK)

    def oracle_seconds(self, cores):
        from oracle.partial import attnres_partial_oracle
        wl = self.wl
        t = time.perf_counter()
        attnres_partial_oracle(self.completed, self.partial, self.delta, wl.q, dy=wl.dy, g_partial=self.gp,
                               key_offset=wl.key_offset, nthreads=cores)
        return time.perf_counter() - t


WORKLOADS = {"long": LongRead, "short": ShortRead, "sliced": SlicedRead, "deep": DeepRead, "multi": MultiRead,
             "multi16": Multi16Read,
             "selected": SelectedRead, "block": BlockRead}
FULL_TOKENS = {"long": 32768, "short": 8192, "sliced": 16384, "deep": 8192, "multi": 32768, "multi16": 32768,
               "selected": 32768, "block": 16384}


def make_exchange(pg, work):
    """The step's data-parallel exchange: the FP32 reduced gradients of one
    step (dq, dw_o or the bank gradient) summed over ranks in place -- the
    method's one exchange step, R + D floats.  `pg` is torch.distributed (or
    None for one process); `work` names the gradients of a backward result."""
    def exchange(res):
        if pg is not None:
            for g in work.grads(res):
                if g is not None:
                    pg.all_reduce(g)
        return res
    return exchange


def run_step(work, stream, exchange):
    """One step: forward, backward, exchange."""
    work.fwd(stream)
    return exchange(work.bwd(stream))


# --------------------------------------------------------------------------
# Reference arm: the FP64 oracle on the host cores
# --------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import build_oracle
    build_oracle()
    W = WORKLOADS[args.workload]
    sample = args.ref_tokens or getattr(W, "ref_tokens", 1024)
    wl = W(tokens=sample)
    n_full = FULL_TOKENS[args.workload]
    b = wl.bytes_for(1)["total"]
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):  # untimed warm-up steps on the timed sample itself
        wl.oracle_seconds(cores)
    times = [wl.oracle_seconds(cores) for _ in range(max(1, args.steps))]
    t = sum(times) / len(times)
    gbs = b / t / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": wl.describe().replace(f"N={sample}", f"N={n_full}"),
                   "sample_tokens": sample,
                   # what a whole step of n_full tokens would take at the measured rate (not run)
                   "ms_per_step_extrapolated": t * 1e3 * (n_full / sample)},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} of {n_full} tokens per step, fwd+bwd in FP64; ms_per_step is "
                                   f"the measured time of that sample"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------
def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from attention_residuals_gb300 import _lib
    from attention_residuals_gb300.build import build
    from attention_residuals_gb300.dist import max_over_ranks, weak_scaling_throughput
    build()
    _lib.load()
    W = WORKLOADS[args.workload]

    # CPU baseline sample is generated before any GPU work (rank 0, N=1 only).
    cpu_tokens = args.cpu_tokens or getattr(W, "cpu_tokens", 8192)
    cpu_wl = W(tokens=cpu_tokens) if (rank == 0 and world == 1 and not args.no_cpu) else None

    work = W(tokens=args.tokens, seed=rank, device=str(dev))
    work.prepare(dev)
    nbytes = work.bytes
    stream = torch.cuda.current_stream(dev)

    exchange = make_exchange(pg, work)
    for _ in range(max(3, args.warmup)):
        work.fwd(stream)
        exchange(work.bwd(stream))
    torch.cuda.synchronize()

    # One process, one GPU: the step's launches are captured once in two CUDA
    # graphs (forward, backward) and replayed, so the timed region is the
    # kernels back to back with no host launch gaps (the calls are
    # asynchronous and capturable; the run-time compiled forward already
    # exists after the warm-up).  With N > 1 ranks the step stays eager, its
    # exchange being an NCCL all-reduce outside any graph.
    graphs = None
    if world == 1 and not args.no_graph:
        gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf):
            work.fwd(torch.cuda.current_stream())
        with torch.cuda.graph(gb):
            work.bwd(torch.cuda.current_stream())
        for _ in range(max(3, args.warmup)):
            gf.replay()
            gb.replay()
        torch.cuda.synchronize()
        graphs = (gf, gb)

    def step_fwd():
        if graphs is not None:
            graphs[0].replay()
        else:
            work.fwd(stream)

    def step_bwd():
        if graphs is not None:
            graphs[1].replay()
        else:
            exchange(work.bwd(stream))

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.mark("begin")
    nvtx = torch.cuda.nvtx  # named ranges for a profiler's timeline (no cost without one)
    nvtx.range_push(f"attnres {args.workload}: {K} timed steps")
    e_start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        nvtx.range_push("forward")
        step_fwd()
        nvtx.range_pop()
        ev[k][1].record(stream)
        nvtx.range_push("backward + exchange")
        step_bwd()
        nvtx.range_pop()
        ev[k][2].record(stream)
    e_end.record(stream)
    torch.cuda.synchronize()
    nvtx.range_pop()
    sampler.mark("end")
    if pg is not None:
        pg.barrier()
    clocks = sampler.stop()
    total_ms = e_start.elapsed_time(e_end)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_step = total_ms / K
    if pg is not None:  # the slowest rank sets the step time
        ms_step, fwd_ms, bwd_ms = max_over_ranks([ms_step, fwd_ms, bwd_ms], device=dev)

    # --------------------- device copy bandwidth on this GPU (context only)
    copy_gbs = None
    if not args.no_copy_probe:
        src = torch.empty((2 << 30,), dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        for _ in range(3):
            dst.copy_(src)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(10):
            dst.copy_(src)
        c1.record(stream)
        torch.cuda.synchronize()
        copy_gbs = 10 * 2 * src.numel() / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del src, dst

    # ---------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        e2e_step, h2d, d2h, host = (work.e2e(stream, args.e2e_chunk) if isinstance(work, SingleRead)
                                    else work.e2e(stream))
        e2e_step()
        torch.cuda.synchronize()
        KE = max(1, min(args.e2e_steps, K))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()
        nvtx.range_push(f"attnres {args.workload}: {KE} end-to-end steps from host memory")
        s0.record(stream)
        for _ in range(KE):
            e2e_step()
        s1.record(stream)
        nvtx.range_pop()
        torch.cuda.synchronize()
        e2e_ms = s0.elapsed_time(s1) / KE
        if pg is not None:
            e2e_ms = max_over_ranks([e2e_ms], device=dev)[0]
        e2e = {"value": weak_scaling_throughput(nbytes["total"], world, e2e_ms), "unit": "GB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "host_link_gbs": (h2d + d2h) / (e2e_ms * 1e-3) / 1e9}
        e2e.update(getattr(work, "e2e_detail", {}))
        del host

    # ---------------------------------------------------------- CPU baseline
    cpu = None
    if cpu_wl is not None:
        cores = os.cpu_count() or 1
        # the sample is read again until about args.cpu_seconds of CPU time
        # have been measured (a bounded sample, not the whole workload)
        secs, reps = 0.0, 0
        while reps == 0 or (secs < args.cpu_seconds and secs * (reps + 1) / reps < 3 * args.cpu_seconds):
            secs += cpu_wl.oracle_seconds(cores)
            reps += 1
        cb = cpu_wl.bytes_for(1)["total"] * reps
        cpu = {"value": cb / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{cpu_tokens} of {work.wl.N} tokens of the same workload, fwd+bwd in "
                         f"FP64, {reps} times ({secs:.1f} s)"}

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0

    peak, peak_kind = read_peak()
    achieved = nbytes["bwd"] / (bwd_ms * 1e-3) / 1e9
    value = weak_scaling_throughput(nbytes["total"], world, ms_step)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": work.describe(),
                   "bytes_per_step": nbytes["total"],
                   "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                   "frac_of_peak_step": value / world / peak,
                   "device_copy_gbs": copy_gbs,
                   "l2": f"inputs larger than L2 ({work.wl.values.numel() * 2 / 1e9:.2f} GB of sources per step); "
                         f"no flush",
                   "parallelism": (f"data parallel x{world} (own batch per rank, dq/dw_o all-reduced)"
                                   if world > 1 else "single GPU"),
                   "launch": "CUDA graph replay (forward graph, backward graph)" if graphs is not None
                             else "eager (one host call per operator)",
                   "plan": work.info},
        "roofline": {"bound": "hbm", "kernel": work.roofline_kernel,
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     # the committed counters describe the full-size launch only
                     "traffic": work.traffic() if args.tokens in (None, FULL_TOKENS[args.workload]) else None},
        "clocks": clocks,
        "gpu_launches": work.launches * K,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk", type=int, default=None,
                    help="tokens per chunk of the host-buffer step (single-query workloads)")
    ap.add_argument("--cpu-tokens", type=int, default=None, help="oracle sample (default: per workload)")
    ap.add_argument("--ref-tokens", type=int, default=None, help="reference-arm sample (default: per workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-copy-probe", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every timed step eagerly (no CUDA graphs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time the oracle baseline measures (its sample repeated)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="fewer tokens of the same workload (profiling captures only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
