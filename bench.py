#!/usr/bin/env python
"""Benchmark of the attention hot path on B300, printing ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-parts] [--no-cpu-baseline] [--case NAME [--batch B]]

Main line: bf16 dense causal GQA prefill, B2 H32 Hkv8 d128 Tq=Tk=8192, TFLOP/s counted from
the algorithmic causal FLOPs (4 d per allowed (query, key) pair: QK^T and PV, 2 FLOP per
multiply-add), with q/k/v resident in HBM.  A step is one ga_attend over that batch; L2 is
flushed (a 256 MiB write, then a 256 MiB read of another buffer so that none of the written lines
is still dirty in L2) before every timed step, outside the timed events.  "e2e" is the same call
from pinned host buffers with every step's copies in and out timed, pipelined over steps on three
streams (see e2e_times).

"parts" (N = 1, rank 0 only) measures the other workloads of the path with the same timing
rules: KV-cache decode (GB/s of K/V read), the Tq=512 chunk at absolute positions, window
1024 + sink at d=256 and the same inputs full causal, and the 128K block-sparse prefill (block
statistics, block selection, sparse attention at several densities).

Multi-GPU (torchrun): every rank runs its own replica of the main workload (no data-path
collective: the units are independent), timing is the max over ranks, value is the total
over ranks ("scaling": "weak").

--impl reference times the float64 CPU oracle on a bounded sample of the same workload and
metric (the pages give no GPU implementation to run).
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV-read GB/s, as % of B300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------------------------ utilities
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def causal_pairs(Tq, Tk, window=0):
    """Allowed (query, key) pairs of one head: rows at absolute positions Tk-Tq .. Tk-1."""
    i = np.arange(Tk - Tq, Tk, dtype=np.int64)
    n = i + 1
    if window:
        n = np.minimum(n, window)
    return int(n.sum())


# CUDA sources each profiled kernel is built from: a traffic figure taken on other
# versions of these files is not reported.
KERNEL_SOURCES = {"prefill_wide_kernel<128,false,0>": ("prefill_wide.cuh", "ptx.cuh", "common.cuh")}


def kernel_source_hash(kernel="prefill_wide_kernel<128,false,0>"):
    """Hash of the kernel's sources with // comments and blank lines removed (a comment edit
    does not change the kernel)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sparse_prefill_gqa_b300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(d, f)) as fh:
            code = [re.sub(r"\s*//.*$", "", line).rstrip() for line in fh]
        h.update(f.encode() + "\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def traffic_record(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    src = kernel_source_hash(kernel)
    with open(p) as f:
        for line in f:
            m = re.match(r"(\S+)\s+(\S+)\s+bytes=(\d+)\s+src=(\w+)", line.strip())
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == src:
                return int(m.group(3))
    return None


def e2e_times(torch, ga, q, k, v, out, steps):
    """Per-step time (ms) of the main-line call end to end from pinned host buffers: (1) serial,
    each step's copy in, call and copy out on one stream; (2) pipelined, the copies of the next and
    previous steps overlapping the call on their own streams (two device buffer sets).  Both time
    every step's full host-to-device and device-to-host traffic."""
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    bufs = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(out))
            for _ in range(2)]

    def serial_step():
        qd, kd, vd, od = bufs[0]
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        ga.ga_attend(qd, kd, vd, od)
        oh.copy_(od, non_blocking=True)

    serial = statistics.mean(timed_steps(torch, serial_step, steps, 2))
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        ev_cmp, ev_out = [], []
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_in)
        s_cmp.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            qd, kd, vd, od = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])      # the call two steps back has read this set
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(e_in)
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])     # this set's previous output is copied out
                ga.ga_attend(qd, kd, vd, od)
                ev_cmp.append(torch.cuda.Event())
                ev_cmp[-1].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[-1])
                oh.copy_(od, non_blocking=True)
                ev_out.append(torch.cuda.Event())
                ev_out[-1].record(s_out)
        end.record(s_out)                                # after the last copy out, itself after all
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n

    pipelined(2)                                         # warm-up
    return serial, pipelined(steps)


class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi every 20 ms; a reader
    thread stamps each line on arrival, and mark() / summary() keep only the samples taken
    between the two marks (the timed region)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.lines = []          # (host time, csv line)
        self.t0 = self.t1 = None
        self._reader = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def __enter__(self):
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._reader is not None:
                self._reader.join(timeout=5)

    def summary(self):
        mhz, mx, reasons, power = [], None, set(), []
        for t, ln in self.lines:
            if self.t0 is not None and not (self.t0 <= t <= (self.t1 or t) + 0.1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                mhz.append(float(f[0]))
                mx = float(f[1])
                power.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz),
                "power_w_max": max(power) if power else None,
                "source": "nvidia-smi -lms 20, samples inside the timed region"}


# ------------------------------------------------------------------------------ inputs
def device_bf16(torch, seed, tag, shape, lengths=None):
    from workloads import randn_bhtd
    bits = randn_bhtd(seed, tag, shape, "bf16", lengths=lengths)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def timed_steps(torch, fn, steps, warmup, flush=None, stream=None):
    """Per-step CUDA-event times (ms) on the launching stream, L2 flushed before each step."""
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    times = []
    s = stream or torch.cuda.current_stream()
    for _ in range(steps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        times.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


# ------------------------------------------------------------------------------ parts
def part_decode_and_chunk(torch, ga, steps, warmup, flush, peaks, batch=None, which=("decode", "chunk")):
    from workloads import get_config, uniform_lengths
    c = get_config(3)
    B, H, n_kv, d, Tk = batch or c.batch, c.n_heads, c.n_kv, c.d, c.Tk
    lens = uniform_lengths(c.seed, B, *c.k_len_range)
    k = device_bf16(torch, c.seed, "k", (B, n_kv, Tk, d), lengths=lens)
    v = device_bf16(torch, c.seed, "v", (B, n_kv, Tk, d), lengths=lens)
    k_lens = torch.from_numpy(lens).cuda()
    res = {}
    if "decode" not in which:
        return dict(res, **_chunk(torch, ga, c, B, H, n_kv, d, k, v, k_lens, lens, steps, warmup, flush))
    # decode Tq = 1
    q = device_bf16(torch, c.seed, "q", (B, H, 1, d))
    out = torch.empty_like(q)
    ws = torch.empty(max(1, ga.ga_workspace_size(B, H, n_kv, d, 1, Tk, torch.bfloat16)),
                     dtype=torch.uint8, device="cuda")
    t = timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, k_lens=k_lens, workspace=ws),
                    steps, warmup, flush)
    kv_bytes = 2 * 2 * d * n_kv * int(lens.sum())
    ms = statistics.mean(t)
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    res["decode"] = {"workload": c.name + " [Tq=1]", "ms": ms, "GB/s": gbs,
                     "frac_hbm": gbs / peaks["hbm_gbs"], "kv_bytes": kv_bytes,
                     "launches_per_step": 2}
    del q, out
    if "chunk" in which:
        res.update(_chunk(torch, ga, c, B, H, n_kv, d, k, v, k_lens, lens, steps, warmup, flush))
    return res


def _chunk(torch, ga, c, B, H, n_kv, d, k, v, k_lens, lens, steps, warmup, flush):
    """Tq = 512 chunk at absolute positions Tk_b - 512 + t over the decode workload's cache."""
    Tq = c.extra["chunk_Tq"]
    q = device_bf16(torch, c.seed, "q512", (B, H, Tq, d))
    out = torch.empty_like(q)
    t = timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, k_lens=k_lens), steps, warmup, flush)
    flops = 4 * d * H * sum(causal_pairs(Tq, int(n)) for n in lens)
    ms = statistics.mean(t)
    return {"chunk": {"workload": c.name + " [Tq=512]", "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
                      "flops": flops, "launches_per_step": 1}}


def part_window_sink(torch, ga, steps, warmup, flush, peaks):
    from workloads import get_config
    c = get_config(4)
    B, H, n_kv, d, T, W = c.batch, c.n_heads, c.n_kv, c.d, c.Tq, c.window
    q = device_bf16(torch, c.seed, "q", (B, H, T, d))
    k = device_bf16(torch, c.seed, "k", (B, n_kv, T, d))
    v = device_bf16(torch, c.seed, "v", (B, n_kv, T, d))
    rng = np.random.Generator(np.random.PCG64(c.seed))
    sink = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).cuda()
    out = torch.empty_like(q)
    tw = statistics.mean(timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, window=W, sink=sink),
                                     steps, warmup, flush))
    tf = statistics.mean(timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, sink=sink),
                                     steps, warmup, flush))
    fw = 4 * d * H * B * causal_pairs(T, T, W)
    ff = 4 * d * H * B * causal_pairs(T, T)
    return {"window": {"workload": c.name + " [window]", "ms": tw, "TFLOP/s": fw / (tw * 1e-3) / 1e12,
                       "flops": fw},
            "full_causal": {"workload": c.name + " [full causal]", "ms": tf,
                            "TFLOP/s": ff / (tf * 1e-3) / 1e12, "flops": ff},
            "composite_5to1": {"TFLOP/s": (5 * fw + ff) / ((5 * tw + tf) * 1e-3) / 1e12}}


def part_ring(torch, ga, steps, warmup, flush, peaks):
    """Decode over W-slot ring caches (the decode side of the window + sink workload): its
    heads (H16 Hkv8 d256), window W = 1024 and sink, a decode batch of 64 sequences (the
    batch of the KV-cache decode workload) whose token counters n are drawn from U[W/2, 4W],
    so most rings have wrapped.  A ring is any set of W keys in any order, so its contents
    are seeded N(0, 1) draws.  Timed: ga_attend_ring (K/V bytes = min(n, W) keys per
    sequence and kv head); the append of one token per sequence is timed on its own."""
    from workloads import get_config
    c = get_config(4)
    B, H, n_kv, d, W = 64, c.n_heads, c.n_kv, c.d, c.window
    q = device_bf16(torch, c.seed, "ring_q", (B, H, 1, d))
    k_ring = device_bf16(torch, c.seed, "ring_k", (B, n_kv, W, d))
    v_ring = device_bf16(torch, c.seed, "ring_v", (B, n_kv, W, d))
    rng = np.random.Generator(np.random.PCG64(c.seed + 17))
    n = rng.integers(W // 2, 4 * W + 1, size=B).astype(np.int32)
    n_seen = torch.from_numpy(n).cuda()
    sink = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).cuda()
    out = torch.empty_like(q)
    ws = torch.empty(max(1, ga.ga_workspace_size(B, H, n_kv, d, 1, W, torch.bfloat16)),
                     dtype=torch.uint8, device="cuda")
    t = timed_steps(torch, lambda: ga.ga_attend_ring(q, k_ring, v_ring, n_seen, out, sink=sink,
                                                     workspace=ws), steps, warmup, flush)
    kv_bytes = 2 * 2 * d * n_kv * int(np.minimum(n, W).sum())
    ms = statistics.mean(t)
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    k_new = device_bf16(torch, c.seed, "ring_k_new", (B, n_kv, 1, d)).view(B, n_kv, d)
    v_new = device_bf16(torch, c.seed, "ring_v_new", (B, n_kv, 1, d)).view(B, n_kv, d)
    n_app = n_seen.clone()
    ta = statistics.mean(timed_steps(torch, lambda: ga.ga_ring_append(k_ring, v_ring, k_new, v_new, n_app),
                                     steps, warmup, flush))
    return {"ring_decode": {"workload": "bf16 ring-buffer decode B64 H16 Hkv8 d256 W1024 + sink, "
                                        "counters U[512, 4096]", "ms": ms, "GB/s": gbs,
                            "frac_hbm": gbs / peaks["hbm_gbs"], "kv_bytes": kv_bytes,
                            "append_us": ta * 1e3}}


def part_diff(torch, ga, steps, warmup, flush, peaks):
    """Differential attention (A1 - lam A2) V on the dense workload's shape (B2 H32 Hkv8 d128
    T8192, causal), lam = 0.8: two attention passes over the same values, the second fusing the
    fp32 difference into its epilogue.  Algorithmic FLOPs: twice the causal attention's."""
    from workloads import get_config
    c = get_config(2)
    B, H, n_kv, d, T = c.batch, c.n_heads, c.n_kv, c.d, c.Tq
    q1 = device_bf16(torch, c.seed, "diff_q1", (B, H, T, d))
    q2 = device_bf16(torch, c.seed, "diff_q2", (B, H, T, d))
    k1 = device_bf16(torch, c.seed, "diff_k1", (B, n_kv, T, d))
    k2 = device_bf16(torch, c.seed, "diff_k2", (B, n_kv, T, d))
    v = device_bf16(torch, c.seed, "diff_v", (B, n_kv, T, d))
    out = torch.empty_like(q1)
    ws = torch.empty(B * H * T * d * 4, dtype=torch.uint8, device="cuda")
    t = statistics.mean(timed_steps(torch, lambda: ga.ga_attend_diff(q1, k1, q2, k2, v, 0.8, out, workspace=ws),
                                    steps, warmup, flush))
    flops = 2 * 4 * d * H * B * causal_pairs(T, T)
    return {"diff_attention": {"workload": "bf16 differential attention B2 H32 Hkv8 d128 T8192 causal, lambda 0.8",
                               "ms": t, "TFLOP/s": flops / (t * 1e-3) / 1e12, "flops": flops,
                               "launches_per_step": 2}}


def part_dsa(torch, ga, steps, warmup, flush, peaks, batch=None):
    """Token top-k sparse decode on the KV-cache decode workload (B64 H32 Hkv8 d128, lengths
    U[16384, 32768]): an indexer of 8 heads x 128 dims scores every cached token, the top
    k = 2048 are kept, and attention reads only those.  Stages timed one by one and together;
    the dense decode of the same cache is timed beside it."""
    from workloads import get_config, uniform_lengths
    c = get_config(3)
    B, H, n_kv, d, Tk = batch or c.batch, c.n_heads, c.n_kv, c.d, c.Tk
    Hi, di, topk = 8, 128, 2048
    lens = uniform_lengths(c.seed, B, *c.k_len_range)
    k = device_bf16(torch, c.seed, "k", (B, n_kv, Tk, d), lengths=lens)
    v = device_bf16(torch, c.seed, "v", (B, n_kv, Tk, d), lengths=lens)
    q = device_bf16(torch, c.seed, "q", (B, H, 1, d))
    qi = device_bf16(torch, c.seed, "dsa_qi", (B, 1, Hi, di)).view(B, Hi, di)
    ki = device_bf16(torch, c.seed, "dsa_ki", (B, 1, Tk, di), lengths=lens).view(B, Tk, di)
    rng = np.random.Generator(np.random.PCG64(c.seed + 31))
    wi = torch.from_numpy(np.abs(rng.standard_normal((B, Hi))).astype(np.float32)).cuda()
    k_lens = torch.from_numpy(lens).cuda()
    scores = torch.empty(B, Tk, dtype=torch.float32, device="cuda")
    idx = torch.empty(B, topk, dtype=torch.int32, device="cuda")
    n_sel = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(int(ga.lib().ga_attend_gather_workspace_size(B, H, n_kv, d, topk)), dtype=torch.uint8,
                     device="cuda")
    t_idx = statistics.mean(timed_steps(torch, lambda: ga.ga_dsa_indexer(qi, wi, ki, k_lens, scores),
                                        steps, warmup, flush))
    t_top = statistics.mean(timed_steps(torch, lambda: ga.ga_topk_indices(scores, topk, k_lens, idx, n_sel),
                                        steps, warmup, flush))
    t_att = statistics.mean(timed_steps(torch, lambda: ga.ga_attend_gather(q, k, v, idx, n_sel, out, workspace=ws),
                                        steps, warmup, flush))

    def step():
        ga.ga_dsa_indexer(qi, wi, ki, k_lens, scores)
        ga.ga_topk_indices(scores, topk, k_lens, idx, n_sel)
        ga.ga_attend_gather(q, k, v, idx, n_sel, out, workspace=ws)
    t_all = statistics.mean(timed_steps(torch, step, steps, warmup, flush))
    dws = torch.empty(max(1, ga.ga_workspace_size(B, H, n_kv, d, 1, Tk, torch.bfloat16)), dtype=torch.uint8,
                      device="cuda")
    dense_out = torch.empty_like(q)
    t_dense = statistics.mean(timed_steps(torch, lambda: ga.ga_attend(q, k, v, dense_out, k_lens=k_lens,
                                                                      workspace=dws), steps, warmup, flush))
    idx_bytes = int(lens.sum()) * di * 2
    sel_kv = B * n_kv * topk * d * 2 * 2                # selected K and V rows, read once
    return {"dsa_decode": {"workload": f"bf16 top-k sparse decode B{B} H32 Hkv8 d128, lengths U[16384, 32768], "
                                       "indexer 8 x 128, k 2048",
                           "ms": t_all, "indexer_ms": t_idx, "indexer_GB/s": idx_bytes / (t_idx * 1e-3) / 1e9,
                           "indexer_frac_hbm": idx_bytes / (t_idx * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "topk_ms": t_top, "gather_decode_ms": t_att, "selected_kv_bytes": sel_kv,
                           "gather_decode_GB/s": sel_kv / (t_att * 1e-3) / 1e9,
                           "gather_decode_frac_hbm": sel_kv / (t_att * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "dense_decode_ms": t_dense,
                           "launches_per_step": 4}}       # indexer, top-k, gathered decode, combine


def part_mla(torch, ga, steps, warmup, flush, peaks):
    """MLA decode, absorbed form, at DeepSeek-V2-Lite's sizes (16 heads, latent 512, rope 64, head
    dims 128): a decode batch of 64 sequences (the batch of the KV-cache decode workload) with
    cache lengths U[4096, 8192].  Bytes: the latent cache read once (576 bf16 per token)."""
    from workloads import uniform_lengths
    B, H, L_max, seed = 64, 16, 8192, 1006
    lens = uniform_lengths(seed, B, 4096, 8192)
    q_nope = device_bf16(torch, seed, "mla_qn", (B, 1, H, 128)).view(B, H, 128)
    q_rope = device_bf16(torch, seed, "mla_qp", (B, 1, H, 64)).view(B, H, 64)
    latent = device_bf16(torch, seed, "mla_lat", (B, 1, L_max, 576), lengths=lens).view(B, L_max, 576)
    rng = np.random.Generator(np.random.PCG64(seed))
    w = torch.from_numpy((rng.standard_normal((2, H, 512, 128)) / np.sqrt(128)).astype(np.float32)).to(torch.bfloat16)
    w_uk, w_uv = w[0].cuda().contiguous(), w[1].cuda().contiguous()
    lens_t = torch.from_numpy(lens).cuda()
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(int(ga.lib().ga_mla_decode_workspace_size(B, H, L_max)), dtype=torch.uint8, device="cuda")
    t = statistics.mean(timed_steps(torch, lambda: ga.ga_mla_decode(q_nope, q_rope, latent, w_uk, w_uv, lens_t,
                                                                   out, workspace=ws), steps, warmup, flush))
    lat_bytes = int(lens.sum()) * 576 * 2
    gbs = lat_bytes / (t * 1e-3) / 1e9
    return {"mla_decode": {"workload": "bf16 MLA decode (absorbed) B64 H16, latent 512 + rope 64, lengths U[4096, 8192]",
                           "ms": t, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "latent_bytes": lat_bytes,
                           "launches_per_step": 4}}


OUTLIER_SCALES = {"8sqrtd": "8*sqrt(d)*u", "8": "8*u (literal)"}


def planted_scale(name, d):
    """Norm of the 128K workload's planted key under each reading of "8x a random unit direction"."""
    return 8.0 * math.sqrt(d) if name == "8sqrtd" else 8.0


def part_sparse_once(torch, ga, steps, warmup, flush, peaks, tau=0.01, heads=None):
    """The 128K block-sparse workload once per step at a fixed mean threshold: block statistics,
    selection and the sparse attention, each timed on its own (a short case for profiling;
    ``heads`` keeps the first query heads and their kv heads only)."""
    from workloads import f32_to_bf16_bits, get_config, planted_outliers, randn_bhtd
    c = get_config(5)
    B, H, n_kv, d, T, qb, kb = c.batch, c.n_heads, c.n_kv, c.d, c.Tq, c.q_block, c.k_block
    if heads:
        H, n_kv = heads, max(1, heads // c.g)
    q = device_bf16(torch, c.seed, "q", (B, H, T, d))
    kbits = randn_bhtd(c.seed, "k", (B, n_kv, T, d), "bf16")
    for kvh, blk, tok, vec in planted_outliers(c.seed, n_kv, T, d, kb, c.planted_fraction):
        kbits[0, kvh, tok] = f32_to_bf16_bits(vec)
    k = torch.from_numpy(kbits.view(np.int16)).view(torch.bfloat16).cuda()
    del kbits
    v = device_bf16(torch, c.seed, "v", (B, n_kv, T, d))
    nQb, nKb = T // qb, T // kb
    cen = torch.empty(B, n_kv, nKb, d, dtype=torch.float32, device="cuda")
    rad = torch.empty(B, n_kv, nKb, dtype=torch.float32, device="cuda")
    mask = torch.empty(B, H, nQb, nKb, dtype=torch.uint8, device="cuda")
    nsel = torch.empty(B, H, nQb, dtype=torch.int32, device="cuda")
    ws = torch.empty(int(ga.lib().ga_select_workspace_size(B, H, n_kv, d, T, T, qb, kb, 0)), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(q)
    ts = timed_steps(torch, lambda: ga.ga_block_stats(k, kb, centroid=cen, radius=rad), steps, warmup, flush)
    tsel = timed_steps(torch, lambda: ga.ga_select_blocks(q, cen, rad, Tk=T, q_block=qb, k_block=kb, tau_mean=tau,
                                                          lambda_radius=c.extra["lambda_radius"], block_mask=mask,
                                                          n_selected=nsel, workspace=ws), steps, warmup, flush)
    ta = timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, block_mask=mask, q_block=qb, k_block=kb),
                     steps, warmup, flush)
    return {"sparse_once": {"heads": H, "tau_mean": tau, "density_blocks": float(mask.sum()) / float(mask.numel()),
                            "stats_ms": statistics.mean(ts), "select_ms": statistics.mean(tsel),
                            "attend_ms": statistics.mean(ta)}}


def part_sparse(torch, ga, steps, warmup, flush, peaks, select_only=False, outlier_scale="8sqrtd"):
    from workloads import f32_to_bf16_bits, get_config, planted_outliers, randn_bhtd
    c = get_config(5)
    B, H, n_kv, d, T, qb, kb = c.batch, c.n_heads, c.n_kv, c.d, c.Tq, c.q_block, c.k_block
    scale_used = planted_scale(outlier_scale, d)
    q = device_bf16(torch, c.seed, "q", (B, H, T, d))
    kbits = randn_bhtd(c.seed, "k", (B, n_kv, T, d), "bf16")
    for kvh, blk, tok, vec in planted_outliers(c.seed, n_kv, T, d, kb, c.planted_fraction, scale=scale_used):
        kbits[0, kvh, tok] = f32_to_bf16_bits(vec)
    k = torch.from_numpy(kbits.view(np.int16)).view(torch.bfloat16).cuda()
    del kbits
    v = device_bf16(torch, c.seed, "v", (B, n_kv, T, d))
    lam = c.extra["lambda_radius"]
    nQb, nKb = T // qb, T // kb
    # allowed (query, key) pairs inside each (query block, key block) of the causal mask
    a = torch.arange(nQb, device="cuda", dtype=torch.int64)[:, None]
    bidx = torch.arange(nKb, device="cuda", dtype=torch.int64)[None, :]
    rows_i = a * qb + torch.arange(qb, device="cuda")[None, :]          # [nQb, qb] positions
    pairs = torch.zeros(nQb, nKb, dtype=torch.int64, device="cuda")
    for r in range(qb):
        i = rows_i[:, r:r + 1]
        pairs += torch.clamp(i + 1 - bidx * kb, 0, kb)
    allowed_blocks = int((pairs > 0).sum()) * H

    res = {}
    cen = torch.empty(B, n_kv, nKb, d, dtype=torch.float32, device="cuda")
    rad = torch.empty(B, n_kv, nKb, dtype=torch.float32, device="cuda")
    ts = timed_steps(torch, lambda: ga.ga_block_stats(k, kb, centroid=cen, radius=rad), steps, warmup, flush)
    stats_bytes = k.numel() * 2 + cen.numel() * 4 + rad.numel() * 4
    res["block_stats"] = {"ms": statistics.mean(ts),
                          "GB/s": stats_bytes / (statistics.mean(ts) * 1e-3) / 1e9,
                          "frac_hbm": stats_bytes / (statistics.mean(ts) * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    mask = torch.empty(B, H, nQb, nKb, dtype=torch.uint8, device="cuda")
    nsel = torch.empty(B, H, nQb, dtype=torch.int32, device="cuda")
    sel_ws = torch.empty(int(ga.lib().ga_select_workspace_size(B, H, n_kv, d, T, T, qb, kb, 0)),
                         dtype=torch.uint8, device="cuda")

    def select(tau):
        ga.ga_select_blocks(q, cen, rad, Tk=T, q_block=qb, k_block=kb, tau_mean=tau, lambda_radius=lam,
                            block_mask=mask, n_selected=nsel, workspace=sel_ws)

    def density():
        return float(mask.sum()) / allowed_blocks

    tsel = timed_steps(torch, lambda: select(0.05), steps, warmup, flush)
    sel_bytes = q.numel() * 2 + cen.numel() * 4 + mask.numel()
    res["block_select"] = {"ms": statistics.mean(tsel),
                           "GB/s": sel_bytes / (statistics.mean(tsel) * 1e-3) / 1e9,
                           "frac_hbm": sel_bytes / (statistics.mean(tsel) * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "algorithmic_bytes": sel_bytes}
    # Selection variants at tau_mean = 0.02 (about density 0.1): the mean branch alone, with the
    # radius rescue (z-score or median/MAD, lambda from the workload), and with the bound branch
    # as the rescue instead (bound >= best mean score + 3, no radius branch); time, density and
    # the recall of the planted outlier blocks (visible (query block, planted block) pairs kept).
    planted = torch.zeros(n_kv, nKb, dtype=torch.bool, device="cuda")
    for kvh, blk, tok, vec in planted_outliers(c.seed, n_kv, T, d, kb, c.planted_fraction):
        planted[kvh, blk] = True
    target = planted.repeat_interleave(H // n_kv, dim=0)[:, None, :] & (pairs > 0)[None]
    variants = {}
    for name, rule, lm, tb, grp in (("mean only", "z", math.inf, None, False), ("z rescue", "z", lam, None, False),
                                    ("mad rescue", "mad", lam, None, False),
                                    ("bound rescue", "z", math.inf, -3.0, False),
                                    ("z rescue, group-shared", "z", lam, None, True)):
        def run_sel(tau_m):
            ga.ga_select_blocks(q, cen, rad, Tk=T, q_block=qb, k_block=kb, tau_mean=tau_m,
                                lambda_radius=lm, block_mask=mask, n_selected=nsel,
                                radius_rule=rule, tau_bound=tb, group_shared=grp, workspace=sel_ws)
        tau_v = 0.02
        if grp:        # the pooled query's scores spread less: match the per-head density instead
            ref_dens = variants["z rescue"]["density"]
            lo, hi = 0.0, 0.02
            for _ in range(14):
                tau_v = 0.5 * (lo + hi)
                run_sel(tau_v)
                lo, hi = (tau_v, hi) if density() < ref_dens else (lo, tau_v)
            tau_v = hi
        tv = statistics.mean(timed_steps(torch, lambda: run_sel(tau_v), max(3, steps // 2), min(warmup, 2), flush))
        run_sel(tau_v)
        recall = float((mask[0].bool() & target).sum()) / max(1, int(target.sum()))
        variants[name] = {"ms": tv, "tau_mean": tau_v, "density": density(), "planted_recall": recall}
    res["block_select_variants"] = variants
    # Both readings of the planted key's scale: the same blocks, slots and directions at norm
    # 8 sqrt(d) and at norm 8; the radius z-scores of the planted blocks (population statistics
    # over each kv head's blocks, as the radius branch takes them) and the share it rescues.
    try:
        readings = {}
        for name, label in OUTLIER_SCALES.items():
            sc = planted_scale(name, d)
            if sc == scale_used:
                r = rad[0].double()
            else:
                plants = planted_outliers(c.seed, n_kv, T, d, kb, c.planted_fraction, scale=sc)
                k_alt = k.clone()
                kv_i = torch.tensor([p[0] for p in plants], device="cuda")
                tok_i = torch.tensor([p[2] for p in plants], device="cuda")
                bits = np.stack([f32_to_bf16_bits(p[3]) for p in plants]).view(np.int16)
                k_alt[0, kv_i, tok_i] = torch.from_numpy(bits).view(torch.bfloat16).cuda()
                cen_alt, rad_alt = torch.empty_like(cen), torch.empty_like(rad)
                ga.ga_block_stats(k_alt, kb, centroid=cen_alt, radius=rad_alt)
                r = rad_alt[0].double()
                del k_alt, cen_alt, rad_alt
            z = (r - r.mean(dim=1, keepdim=True)) / r.std(dim=1, correction=0, keepdim=True)
            zp = z[planted]
            readings[label] = {"planted_z_mean": float(zp.mean()), "planted_z_min": float(zp.min()),
                               "rescued_at_lambda": float((zp >= lam).double().mean())}
        res["planted_key_scale"] = {"in_use": OUTLIER_SCALES[outlier_scale], "lambda_radius": lam,
                                    "readings": readings}
    except Exception as e:  # report, never hide
        res["planted_key_scale"] = {"error": repr(e)}
    if select_only:
        return res
    # tau for target densities (bisection on the measured density)
    targets = [0.05, 0.1, 0.2, 0.4]
    sweep = []
    out = torch.empty_like(q)
    for tgt in targets + [1.0]:
        if tgt >= 1.0:
            tau = math.inf
        else:
            lo, hi = 0.0, 0.2
            for _ in range(14):
                mid = 0.5 * (lo + hi)
                select(mid)
                if density() < tgt:
                    lo = mid
                else:
                    hi = mid
            tau = hi
        select(tau)
        dens = density()
        sel_pairs = int((mask[0].to(torch.int64) * pairs[None]).sum())
        flops = 4 * d * sel_pairs
        t = statistics.mean(timed_steps(torch, lambda: ga.ga_attend(q, k, v, out, block_mask=mask,
                                                                    q_block=qb, k_block=kb),
                                        max(2, steps // 2), min(warmup, 2), flush))
        sweep.append({"tau_mean": tau if math.isfinite(tau) else "inf", "density": dens, "ms": t, "TFLOP/s": flops / (t * 1e-3) / 1e12})
    dens = np.array([s["density"] for s in sweep])
    tms = np.array([s["ms"] for s in sweep])
    A = np.vstack([dens, np.ones_like(dens)]).T
    coef, resid, *_ = np.linalg.lstsq(A, tms, rcond=None)
    pred = A @ coef
    r2 = 1 - ((tms - pred) ** 2).sum() / ((tms - tms.mean()) ** 2).sum()
    res["sparse_attention"] = {"workload": c.name, "sweep": sweep, "linear_fit_ms": list(coef),
                               "r2": float(r2), "sparse_over_dense_at_0.1": float(tms[1] / tms[-1])}
    return res


# ------------------------------------------------------------------------------ CPU oracle
def cpu_oracle_timed(budget_s=None, n_pairs=None):
    """The float64 oracle on 256 sampled query rows of (batch, head) pairs of the dense causal
    workload, one pair after another, until ``budget_s`` seconds of oracle time or ``n_pairs``
    pairs.  Returns (TFLOP/s on the sampled rows, cores, sample text, oracle seconds, pairs)."""
    import oracle
    from workloads import get_config, normal_slices, bf16_bits_to_f32, sample_rows
    cores = len(os.sched_getaffinity(0))
    c = get_config(2)
    rows = sample_rows(c.Tq, 256, seed=c.seed)
    limit = c.batch * c.n_heads if n_pairs is None else min(n_pairs, c.batch * c.n_heads)
    tot_flops, tot_time, heads = 0, 0.0, 0
    while heads < limit and (budget_s is None or tot_time < budget_s):
        b, h = divmod(heads, c.n_heads)
        kvh = h // c.g
        q = bf16_bits_to_f32(normal_slices(c.seed, "q", b, h, c.Tq, c.d))[None, None].astype(np.float64)
        k = bf16_bits_to_f32(normal_slices(c.seed, "k", b, kvh, c.Tk, c.d))[None, None].astype(np.float64)
        v = bf16_bits_to_f32(normal_slices(c.seed, "v", b, kvh, c.Tk, c.d))[None, None].astype(np.float64)
        ts = time.perf_counter()
        oracle.attend(q, k, v, rows=rows)
        tot_time += time.perf_counter() - ts
        tot_flops += 4 * c.d * int((rows + 1).sum())
        heads += 1
    sample = (f"{heads} (batch, head) pairs x {len(rows)} sampled query rows of the B2 H32 Hkv8 d128 "
              f"T8192 causal workload through the float64 NumPy oracle (input generation excluded)")
    return tot_flops / tot_time / 1e12, cores, sample, tot_time, heads


def reference_arm(args, warmup, flops_step, workload):
    """--impl reference: the oracle, as it stands, on the host cores.  A step is a fixed sample
    (256 rows of each of P (batch, head) pairs), P chosen from one timed pair so that the
    warm-up and timed steps together take about two minutes; ms_per_step is that step's
    measured wall time, and the full workload's time is reported apart, as an extrapolation."""
    per_pair = cpu_oracle_timed(n_pairs=1)[3]
    n_steps = warmup + args.steps
    pairs = int(max(1, min(64, 120.0 / max(1, n_steps) / max(per_pair, 1e-3))))
    vals, walls = [], []
    cores, sample = 0, ""
    for i in range(n_steps):
        t0 = time.perf_counter()
        v, cores, sample, _, _ = cpu_oracle_timed(n_pairs=pairs)
        wall = (time.perf_counter() - t0) * 1e3
        if i >= warmup:
            vals.append(v)
            walls.append(wall)
    val = statistics.mean(vals)
    ms_step = statistics.mean(walls)
    sample += f"; one step = these {pairs} pairs, {ms_step / 1e3:.2f} s wall per step (input generation included)"
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64 N(0,1), cast to bf16 on the host, upcast to f64)",
            "config": workload,
            "extrapolated_full_step_ms": {"value": flops_step / (val * 1e12) * 1e3,
                                          "what": "an extrapolation, not a measurement: the whole B2 H32 "
                                                  "T8192 step's FLOPs at the sampled rows' rate"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _r(x, n=4):
    """x rounded to n significant digits (None stays None)."""
    if x is None or not isinstance(x, (int, float)) or not math.isfinite(x):
        return x
    return float(f"{x:.{n}g}")


def targets_summary(line, peaks):
    """The per-workload figures the targets are judged on, in one short object (printed last,
    so that a reader of the line's tail sees them): TFLOP/s and GB/s with their fractions of
    the measured burst peaks."""
    p = line.get("parts", {})
    bf, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    def g(part, key):
        d = p.get(part)
        return d.get(key) if isinstance(d, dict) else None
    t = {"prefill_TFLOPs": _r(line["roofline"]["achieved"]), "prefill_frac": _r(line["roofline"]["frac"], 3)}
    for key, part in (("decode", "decode"), ("ring", "ring_decode")):
        gbs = g(part, "GB/s")
        t[key + "_GBs"] = _r(gbs)
        t[key + "_frac"] = _r(gbs / hbm, 3) if gbs else None
    for key, part in (("chunk", "chunk"), ("window", "window"), ("full", "full_causal"), ("diff", "diff_attention")):
        tf = g(part, "TFLOP/s")
        t[key + "_TFLOPs"] = _r(tf)
        t[key + "_frac"] = _r(tf / bf, 3) if tf else None
    t["composite_TFLOPs"] = _r(g("composite_5to1", "TFLOP/s"))
    t["stats_frac"] = _r(g("block_stats", "frac_hbm"), 3)
    t["select_ms"] = _r(g("block_select", "ms"), 3)
    t["select_frac"] = _r(g("block_select", "frac_hbm"), 3)
    sp = p.get("sparse_attention", {})
    if isinstance(sp, dict) and sp.get("sweep"):
        t["sparse_r2"] = _r(sp.get("r2"), 3)
        t["sparse_ratio_0.1"] = _r(sp.get("sparse_over_dense_at_0.1"), 3)
        t["sparse_TFLOPs_by_density"] = {f"{s['density']:.2f}": _r(s["TFLOP/s"]) for s in sp["sweep"]}
    t["dsa_ms"] = _r(g("dsa_decode", "ms"), 3)
    t["gather_frac"] = _r(g("dsa_decode", "gather_decode_frac_hbm"), 3)
    t["mla_frac"] = _r(g("mla_decode", "frac_hbm"), 3)
    t["peaks"] = f"measured burst: {hbm:g} GB/s, {bf:g} TFLOP/s bf16"
    return t


# ------------------------------------------------------------------------------ one case
def run_case(torch, ga, args, warmup, flush, peaks, c):
    """One workload alone (steps and warm-up as given); prints its JSON line."""
    if args.case == "prefill":
        B = args.batch or c.batch
        q = device_bf16(torch, c.seed, "q", (B, c.n_heads, c.Tq, c.d))
        k = device_bf16(torch, c.seed, "k", (B, c.n_kv, c.Tk, c.d))
        v = device_bf16(torch, c.seed, "v", (B, c.n_kv, c.Tk, c.d))
        out = torch.empty_like(q)
        t = timed_steps(torch, lambda: ga.ga_attend(q, k, v, out), args.steps, warmup, flush)
        flops = 4 * c.d * c.n_heads * B * causal_pairs(c.Tq, c.Tk)
        ms = statistics.mean(t)
        res = {"prefill": {"workload": f"dense causal B{B} H{c.n_heads} Hkv{c.n_kv} d{c.d} T{c.Tq}",
                           "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "flops": flops}}
    elif args.case in ("decode", "chunk"):
        res = part_decode_and_chunk(torch, ga, args.steps, warmup, flush, peaks, batch=args.batch,
                                    which=(args.case,))
    elif args.case == "window":
        res = part_window_sink(torch, ga, args.steps, warmup, flush, peaks)
    elif args.case == "ring":
        res = part_ring(torch, ga, args.steps, warmup, flush, peaks)
    elif args.case == "diff":
        res = part_diff(torch, ga, args.steps, warmup, flush, peaks)
    elif args.case == "dsa":
        res = part_dsa(torch, ga, args.steps, warmup, flush, peaks, batch=args.batch)
    elif args.case == "mla":
        res = part_mla(torch, ga, args.steps, warmup, flush, peaks)
    elif args.case == "sparse_once":
        res = part_sparse_once(torch, ga, args.steps, warmup, flush, peaks, tau=args.tau, heads=args.heads)
    else:
        res = part_sparse(torch, ga, args.steps, warmup, flush, peaks, select_only=args.case == "select",
                          outlier_scale=args.outlier_scale)
    print(json.dumps({"case": args.case, "steps": args.steps, "warmup": warmup, **res}))
    return 0


# ------------------------------------------------------------------------------ main
def max_over_ranks(torch, dist, total_ms, device):
    """The job's timed total: the slowest rank's (every rank waits at the closing barrier)."""
    if dist is None:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_step, steps, total_ms):
    """Whole-job throughput: each of the `world` ranks runs its own replica of the step."""
    return world * flops_step * steps / (total_ms * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-parts", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default="all",
                    choices=["all", "prefill", "decode", "chunk", "window", "ring", "diff", "dsa", "mla", "sparse", "select",
                             "sparse_once"],
                    help="run one workload alone and print its own JSON line (for profiling)")
    ap.add_argument("--outlier-scale", default="8sqrtd", choices=sorted(OUTLIER_SCALES),
                    help="norm of the 128K workload's planted keys: 8*sqrt(d) (default) or the literal 8")
    ap.add_argument("--heads", type=int, default=None,
                    help="with --case sparse_once: the first query heads only (profiling captures)")
    ap.add_argument("--tau", type=float, default=0.01,
                    help="with --case sparse_once: the mean-branch threshold")
    ap.add_argument("--batch", type=int, default=None,
                    help="with --case prefill/decode/chunk: a smaller batch (profiling captures)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from workloads import get_config
    c = get_config(2)
    flops_step = 4 * c.d * c.n_heads * c.batch * causal_pairs(c.Tq, c.Tk)
    workload = {"workload": "bf16 dense causal GQA prefill B2 H32 Hkv8 d128 Tq=Tk=8192",
                "global_batch": c.batch * world, "seq_len": c.Tq, "n_heads": c.n_heads,
                "n_kv": c.n_kv, "head_dim": c.d, "parallelism": f"replicas x{world}",
                "l2": "flushed before every timed step (256 MiB write, then 256 MiB read of another buffer; outside the timed events)"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args, warmup, flops_step, workload)))
        return 0

    import torch
    import sparse_prefill_gqa_b300 as ga
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    peaks, peaks_src = load_peaks()
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    flush_read = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device="cuda")

    def flush():
        # The write evicts the inputs; the read of a second buffer then evicts the written lines,
        # so their write-back is not charged to the timed step.
        flush_buf.fill_(1)
        flush_read.sum()

    if args.case != "all":
        return run_case(torch, ga, args, warmup, flush, peaks, c)

    B, H, n_kv, d, T = c.batch, c.n_heads, c.n_kv, c.d, c.Tq
    q = device_bf16(torch, c.seed, "q", (B, H, T, d))
    k = device_bf16(torch, c.seed, "k", (B, n_kv, T, d))
    v = device_bf16(torch, c.seed, "v", (B, n_kv, T, d))
    out = torch.empty_like(q)

    def step():
        ga.ga_attend(q, k, v, out)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev = []
        s = torch.cuda.current_stream()
        clk.mark_start()
        for _ in range(args.steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b_ = torch.cuda.Event(enable_timing=True)
            a.record(s)
            step()
            b_.record(s)
            ev.append((a, b_))
        torch.cuda.synchronize()
        clk.mark_end()
    if dist:
        dist.barrier()
    times = [a.elapsed_time(b_) for a, b_ in ev]
    total_ms = max_over_ranks(torch, dist, sum(times), "cuda")
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops_step, args.steps, total_ms)
    kern_tflops = flops_step / (statistics.mean(times) * 1e-3) / 1e12

    # end to end: pinned host buffers, every step's copies inside the timed region
    # (whole job: every rank's replica, the slowest rank's time, as for the main value)
    e2e_steps = max(3, min(args.steps, 10))
    if dist:
        dist.barrier()
    e2e_serial_ms, e2e_ms = e2e_times(torch, ga, q, k, v, out, e2e_steps)
    e2e_serial_ms = max_over_ranks(torch, dist, e2e_serial_ms, "cuda")
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, "cuda")
    e2e_val = job_tflops(world, flops_step, 1, e2e_ms)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak_key = "bf16_tflops"
    roof = {"kernel": "prefill_wide_kernel<128,false,0>", "bound": "tensor", "achieved": kern_tflops,
            "peak": peaks[peak_key], "unit": "TFLOP/s", "frac": kern_tflops / peaks[peak_key],
            "peak_source": f"{peaks_src} ({peak_key}, burst: the kernel is timed alone)",
            "algorithmic_flops_per_launch": flops_step,
            "traffic": traffic_record("prefill_wide_kernel<128,false,0>", "dense-causal-B2-H32-Hkv8-d128-T8192")}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded PCG64 N(0,1) drawn in fp32, cast to bf16 on the host)",
            "config": workload, "roofline": roof, "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "e2e": {"value": e2e_val, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
                    "d2h_bytes_per_step": out.numel() * 2,
                    "ms_per_step": e2e_ms,
                    "how": "pipelined over steps: step i+1's inputs copied in, step i computed and step "
                           "i-1's output copied out on three streams, two device buffer sets; every "
                           "step's copies inside the timed region",
                    "serial_value": job_tflops(world, flops_step, 1, e2e_serial_ms)}}

    if not args.no_parts and world == 1:
        parts = {}
        ps, pw = max(3, min(20, args.steps // 4)), 3
        for name, fn in (("decode_chunk", part_decode_and_chunk), ("window_sink", part_window_sink),
                         ("ring", part_ring), ("diff", part_diff), ("dsa", part_dsa), ("mla", part_mla),
                         ("sparse_128k", functools.partial(part_sparse, outlier_scale=args.outlier_scale))):
            try:
                parts.update(fn(torch, ga, ps, pw, flush, peaks))
            except Exception as e:  # report, never hide
                parts[name] = {"error": repr(e)}
            torch.cuda.empty_cache()
        line["parts"] = parts
    if not args.no_cpu_baseline:
        val, cores, sample, _, _ = cpu_oracle_timed(12.0, 64)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if "parts" in line:                       # the parts last but one, the short summary last
        line["parts"] = line.pop("parts")
        line["targets"] = targets_summary(line, peaks)
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
