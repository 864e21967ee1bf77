#!/usr/bin/env python3
"""Benchmark of the weight-streaming projection path on GB300.

Prints ONE JSON line.  The headline workload is the q8 decode layer (B = 1, hidden
4096, kv 1024, inter 14336: q, k, v, o, up, down in the q8 block format, 179,306,496
weight bytes): value = weight GB/s over the whole step (add+RMSNorm fused into the
first launch, relu² fused into up, two launches).  The other workloads (the tiny f16
MLP block, the 32-layer B = 64 prefill pass, the MoE prefill layer and the vocab head)
are reported under "workloads" with their own metric, roofline and launch counts.

Rules kept: W >= 3 warm-up steps; weights rotate over copies whose total exceeds the
L2 (or exceed it on their own); CUDA events on the launching stream; clocks sampled
with nvidia-smi during the timed region; the oracle (``--impl reference`` or the
``cpu_baseline`` leg) runs on the host cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "weight GB/s & % of HBM roofline (B=1 decode); positions/s (B=64 prefill)"
FALLBACK_HBM = 6800.0


# ------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=FALLBACK_HBM, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "prefill_gemv_q8_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, files):
    """DRAM bytes per launch from a committed ncu capture, or None when the kernel's
    source changed since the capture (or there is none)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_sha") != source_sha(files):
        return None
    return d.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].isdigit():
                    rows.append(f)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [int(r[1]) for r in rows]
        mx = max(int(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workloads
Q8_FILES = ["gemv_tma.cu", "gemv.cu", "tc.cuh", "common.cuh", "kernels.cuh"]


class Q8DecodeLayer:
    """q8 decode layer, B = 1.  Step = {norm+q,k,v,o,up} launch + {down} launch."""
    name = "q8 decode layer B=1 (hidden 4096, kv 1024, inter 14336)"

    def __init__(self, torch, pgq, synth, copies=3):
        c = synth.Q8_LAYER
        self.t, self.pgq = torch, pgq
        self.H, self.KV, self.I = c["hidden"], c["kv"], c["inter"]
        wl = c["workload"]
        base = synth.q8_layer(wl, 0, self.H, self.KV, self.I, "torch", "cuda")
        # copies of the weights at distinct addresses: 3 x 179 MB > 129 MB L2
        self.layers = [base] + [{s: (cc.clone(), pp.clone()) for s, (cc, pp) in base.items()}
                                for _ in range(copies - 1)]
        self.x = synth.normal((1, self.H), 1.0, wl, synth.T_X, "torch", "cuda")
        self.xo = synth.normal((1, self.H), 1.0, wl, synth.T_XO, "torch", "cuda")
        self.g = synth.gamma(self.H, wl, backend="torch", device="cuda")
        f = lambda n: torch.empty(1, n, dtype=torch.float32, device="cuda")  # noqa: E731
        self.out = dict(q=f(self.H), k=f(self.KV), v=f(self.KV), o=f(self.H), u=f(self.I), down=f(self.H))
        self.out1 = {k: v[0] for k, v in self.out.items()}
        sizes = {"q": (self.H, self.H), "k": (self.KV, self.H), "v": (self.KV, self.H), "o": (self.H, self.H),
                 "up": (self.I, self.H), "down": (self.H, self.I)}
        self.bytes = {s: r * c_ + r * (c_ // 32) * 4 for s, (r, c_) in sizes.items()}
        self.step_bytes = sum(self.bytes.values())
        self.k1_bytes = self.step_bytes - self.bytes["down"]
        self.launches_per_step = 2
        self.i = 0

    def launch1(self, L):
        o = self.out
        self.pgq.gemv_q8_multi(
            [dict(codes=L["q"][0], params=L["q"][1], y=o["q"], input=0),
             dict(codes=L["k"][0], params=L["k"][1], y=o["k"], input=0),
             dict(codes=L["v"][0], params=L["v"][1], y=o["v"], input=0),
             dict(codes=L["o"][0], params=L["o"][1], y=o["o"], input=1),
             dict(codes=L["up"][0], params=L["up"][1], y=o["u"], input=0, epilogue="relu2")],
            [(self.x, self.g), (self.xo, None)], eps=1e-6)

    def launch2(self, L):
        self.pgq.gemv_q8(L["down"][0], L["down"][1], self.out["u"], y=self.out["down"])

    def step(self, L):
        """The layer through its entry point; the weights are loaded once, so each
        launch may stream its weights while the kernel before it finishes."""
        self.pgq.q8_decode_layer(L, self.x[0], self.xo[0], self.g, 1e-6, out=self.out1, weights_stable=True)

    def next_layer(self):
        L = self.layers[self.i % len(self.layers)]
        self.i += 1
        return L

    def e2e_setup(self):
        """Host buffers of the end-to-end step: x and x_o in one pinned buffer (one
        copy in), the six outputs in one device buffer and one pinned buffer (one copy
        out); the layer descriptors built once."""
        t = self.t
        H, KV, I = self.H, self.KV, self.I
        self.xin = t.empty((2, H), dtype=t.float32, device="cuda")
        self.hin = t.empty((2, H), dtype=t.float32).pin_memory()
        self.hin[0].copy_(self.x[0].cpu())
        self.hin[1].copy_(self.xo[0].cpu())
        sizes = (("q", H), ("k", KV), ("v", KV), ("o", H), ("u", I), ("down", H))
        n = sum(m for _, m in sizes)
        self.obuf = t.empty(n, dtype=t.float32, device="cuda")
        self.hobuf = t.empty(n, dtype=t.float32).pin_memory()
        self.eout, o = {}, 0
        for k, m in sizes:
            self.eout[k] = self.obuf[o:o + m]
            o += m
        self.structs = [self.pgq.q8_layer_struct(L) for L in self.layers]
        self.h2d = self.hin.numel() * 4
        self.d2h = n * 4

    def e2e_step(self):
        """Public API end to end: the inputs in from pinned host memory, the layer
        call, the outputs back to pinned host memory."""
        self.xin.copy_(self.hin, non_blocking=True)
        L = self.structs[self.i % len(self.structs)]
        self.i += 1
        self.pgq.q8_decode_layer(L, self.xin[0], self.xin[1], self.g, 1e-6, out=self.eout, weights_stable=True)
        self.hobuf.copy_(self.obuf, non_blocking=True)


def _capture(torch, fn):
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_q8_layer(torch, W, steps, warmup):
    """`steps` consecutive layer steps (2 launches each, through the layer entry point,
    the weight copies in rotation) as one CUDA graph, replayed once for the timed
    region after a graph of `warmup` such steps: returns (total ms over `steps`, mean
    ms of the dominant launch, mean ms of the down launch), the launch means from
    their own graphs' replays."""
    st = torch.cuda.current_stream()
    n = len(W.layers)
    g_warm = _capture(torch, lambda: [W.step(W.layers[i % n]) for i in range(warmup)])
    g_all = _capture(torch, lambda: [W.step(W.layers[i % n]) for i in range(steps)])
    g_all.replay()    # the first replay of a graph also uploads it (about 1.4 us per step here)
    g_warm.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    g_all.replay()
    b.record(st)
    torch.cuda.synchronize()
    total = a.elapsed_time(b)

    def per_launch(fn):
        """mean ms of one launch in a graph of `steps` of them back to back"""
        g = _capture(torch, lambda: [fn(W.layers[i % n]) for i in range(steps)])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    return total, per_launch(W.launch1), per_launch(W.launch2)


PREFILL_FILES = ["prefill.cu", "tc.cuh", "common.cuh", "kernels.cuh"]


class PrefillPass:
    """32-layer batched prefill pass, B = 64 positions, hidden 4096 (the q8 decode
    layer's projections per layer, 5,737,807,872 weight bytes per pass)."""
    name = "prefill pass B=64, 32 layers (hidden 4096, kv 1024, inter 14336)"

    def __init__(self, torch, pgq, synth, layers=None):
        c = synth.PREFILL
        self.t, self.pgq = torch, pgq
        self.B, self.H, self.KV, self.I = c["B"], c["hidden"], c["kv"], c["inter"]
        self.L = layers or c["layers"]
        wl = c["workload"]
        self.layers = [synth.q8_layer(wl, l, self.H, self.KV, self.I, "torch", "cuda") for l in range(self.L)]
        self.PL = pgq.PassLayers(self.layers)
        self.h0 = synth.normal((self.B, self.H), 1.0, wl, synth.T_X, "torch", "cuda")
        self.h = self.h0.clone()
        self.g1 = synth.uniform((self.L, self.H), 0.5, 1.5, wl, synth.T_GAMMA, "torch", "cuda")
        self.g2 = synth.uniform((self.L, self.H), 0.5, 1.5, wl, synth.T_GAMMA2, "torch", "cuda")
        self.ws = pgq.prefill_pass_workspace(self.H, self.KV, self.I, self.B)
        per_layer = sum(r * c_ + r * (c_ // 32) * 4 for r, c_ in synth.q8_layer_shapes(self.H, self.KV, self.I).values())
        self.step_bytes = per_layer * self.L
        self.flops = 2 * self.B * sum(r * c_ for r, c_ in synth.q8_layer_shapes(self.H, self.KV, self.I).values()) * self.L
        # launches per pass: per PASS_LMAX layers one input kernel and one persistent launch
        self.persistent_launches = (self.L + pgq.PASS_LMAX - 1) // pgq.PASS_LMAX
        self.launches_per_step = 2 * self.persistent_launches

    def step(self):
        self.h.copy_(self.h0)
        self.pgq.prefill_pass(self.PL, self.h, self.g1, self.g2, 1e-6, workspace=self.ws)


class PrefillPassQ82F(PrefillPass):
    """The same pass with the layers in the q8_2f format (int8 body, binary16 row
    scale, binary16 column field)."""
    name = "q8_2f prefill pass B=64, 32 layers (hidden 4096, kv 1024, inter 14336)"

    def __init__(self, torch, pgq, synth, layers=None):
        c = synth.PREFILL
        self.t, self.pgq = torch, pgq
        self.B, self.H, self.KV, self.I = c["B"], c["hidden"], c["kv"], c["inter"]
        self.L = layers or c["layers"]
        wl = c["workload"]
        self.layers = [synth.q82f_layer(wl, l, self.H, self.KV, self.I, "torch", "cuda") for l in range(self.L)]
        self.PL = pgq.Q82PassLayers(self.layers)
        self.h0 = synth.normal((self.B, self.H), 1.0, wl, synth.T_X, "torch", "cuda")
        self.h = self.h0.clone()
        self.g1 = synth.uniform((self.L, self.H), 0.5, 1.5, wl, synth.T_GAMMA, "torch", "cuda")
        self.g2 = synth.uniform((self.L, self.H), 0.5, 1.5, wl, synth.T_GAMMA2, "torch", "cuda")
        self.ws = pgq.prefill_pass_workspace(self.H, self.KV, self.I, self.B)
        shapes = synth.q8_layer_shapes(self.H, self.KV, self.I).values()
        self.step_bytes = sum(r * c_ + 2 * r + 2 * c_ for r, c_ in shapes) * self.L
        self.persistent_launches = (self.L + pgq.PASS_LMAX - 1) // pgq.PASS_LMAX

    def step(self):
        self.h.copy_(self.h0)
        self.pgq.q82f_prefill_pass(self.PL, self.h, self.g1, self.g2, 1e-6, workspace=self.ws)


def time_prefill_q82f(torch, P, steps, warmup, pk):
    ms = time_graph(torch, P.step, steps, warmup)
    gbs = P.step_bytes / (ms * 1e-3) / 1e9
    return {"workload": P.name, "metric": "positions/s", "value": round(P.B / (ms * 1e-3), 1),
            "ms_per_pass": round(ms, 4), "weight_GBps": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
            "weight_bytes_per_pass": P.step_bytes, "launches_per_pass": 2 * P.persistent_launches,
            "timed": "CUDA-graph replay of the pass call"}


def time_prefill(torch, P, steps, warmup, pk):
    st = torch.cuda.current_stream()
    ms_api = time_loop(torch, P.step, steps, warmup)
    ms = time_graph(torch, P.step, steps, warmup)
    # dominant kernel alone: the up projection (14336 x 4096, relu²) of each of the
    # layers in turn, one CUDA graph of back-to-back calls (host launch cost removed)
    up_bytes = P.I * P.H + P.I * (P.H // 32) * 4
    X = P.h0
    U = torch.empty(P.B, P.I, device="cuda")
    gws = P.pgq.prefill_workspace([P.I], P.H, P.B)
    jobs = [[dict(codes=L["up"][0], params=L["up"][1], y=U, epilogue="relu2")] for L in P.layers]

    def ups():
        for j in jobs:
            P.pgq.prefill_q8(j, X, workspace=gws)
    k_ms = time_graph(torch, ups, max(2, steps // 4), max(1, warmup // 2)) / len(jobs)
    gbs = P.step_bytes / (ms * 1e-3) / 1e9
    ach = up_bytes / (k_ms * 1e-3) / 1e9
    tf = P.flops / (ms * 1e-3) / 1e12
    return {
        "workload": P.name, "metric": "positions/s", "value": round(P.B / (ms * 1e-3), 1),
        "ms_per_pass": round(ms, 4), "ms_per_pass_api": round(ms_api, 4),
        "timed": "CUDA-graph replay of the pass call (ms_per_pass_api: direct calls, host launch cost included)",
        "weight_GBps": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
        "tflops": round(tf, 1), "frac_of_bf16_tensor": round(tf / pk["bf16_sustained"], 4),
        "bound": "hbm", "weight_bytes_per_pass": P.step_bytes, "launches_per_pass": P.launches_per_step,
        # the pass is one persistent launch per PASS_LMAX layers (plus its input kernel):
        # the dominant kernel's roofline is the pass's weight bytes per launch (average)
        "roofline": {"bound": "hbm",
                     "kernel": f"pgq_prefill_pass_kernel ({P.pgq.PASS_LMAX} layers = {4 * P.pgq.PASS_LMAX} phases per "
                               f"launch, B=64; {P.persistent_launches} launches per pass)",
                     "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                     # (the capture's figure is for a launch of PASS_LMAX layers)
                     "traffic": ncu_traffic("prefill_pass_launch", PREFILL_FILES)
                     if P.L % P.pgq.PASS_LMAX == 0 else None,
                     "algorithmic_bytes_per_launch": P.step_bytes // P.persistent_launches,
                     "avg_launch_ms": round(ms / P.persistent_launches, 5),
                     "timed": "CUDA-graph replay of the pass; per launch = pass / persistent launches (input kernels "
                              "included)"},
        "up_alone": {"kernel": "pgq_prefill_pass_kernel, one phase (up 14336x4096, relu²) + input kernel",
                     "GBps": round(ach, 1), "frac": round(ach / pk["hbm"], 4), "bytes": up_bytes,
                     "avg_launch_ms": round(k_ms, 5),
                     "timed": "CUDA graph of one call per layer's up matrix, back to back; per call"},
    }


def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_loop(torch, fn, steps, warmup):
    """Average ms per call of fn() over `steps` calls, CUDA events on the current stream."""
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = _events(torch, 2)
    a.record(st)
    for _ in range(steps):
        fn()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def time_graph(torch, fn, steps, warmup):
    """The same through one CUDA graph capturing fn() (launch overhead removed)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return time_loop(torch, g.replay, steps, warmup)


def bench_tiny_mlp(torch, pgq, synth, steps, warmup, pk):
    """The tiny f16 MLP block (4 MiB of weights): launch-latency bound.  Timed three
    ways: direct calls of the two-launch form (host launch cost included), and CUDA
    graphs of K steps of the two-launch and of the one-launch (fused) form; value =
    the faster of the two graphs (named in `timed`)."""
    c = synth.TINY_MLP
    H, I, wl = c["hidden"], c["inter"], c["workload"]
    h = synth.normal((H,), 1.0, wl, synth.T_X, "torch", "cuda")
    g = synth.gamma(H, wl, backend="torch", device="cuda")
    Wu = synth.f16_matrix(I, H, wl, synth.T_WUP, "torch", "cuda")
    Wd = synth.f16_matrix(H, I, wl, synth.T_WDOWN, "torch", "cuda")
    copies = [(Wu, Wd)] + [(Wu.clone(), Wd.clone()) for _ in range(63)]   # 64 x 4 MiB > 2 x L2
    u = torch.empty(I, device="cuda")
    y = torch.empty(H, device="cuda")
    sync = pgq.layer_sync()
    it = [0]

    def step(fused=False):
        a, b = copies[it[0] % len(copies)]
        it[0] += 1
        if fused:
            pgq.mlp_f16_decode_fused(h, a, b, g, 1e-6, sync=sync, u=u, y=y)
        else:
            pgq.mlp_f16_decode(h, a, b, g, 1e-6, u=u, y=y)

    ms_direct = time_loop(torch, step, steps * 4, warmup)

    def graph_ms(fused):
        g_all = _capture(torch, lambda: [step(fused) for _ in range(steps)])
        g_all.replay()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        a, b = _events(torch, 2)
        a.record(st)
        g_all.replay()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms_two = graph_ms(False)
    ms_one = graph_ms(True)
    nbytes = 2 * H * I * 2
    one_faster = ms_one < ms_two
    ms = ms_one if one_faster else ms_two
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "tiny decode MLP block B=1 (hidden 512, inter 2048, f16)", "metric": "weight GB/s",
            "value": round(gbs, 1), "us_per_step": round(ms * 1e3, 2), "weight_bytes": nbytes,
            "launches_per_step": 1 if one_faster else 2, "frac_of_hbm": round(gbs / pk["hbm"], 4),
            "timed": "CUDA graph of K steps of the " + ("one-launch form (pgq_mlp_f16_decode_fused)" if one_faster
                                                        else "two-launch form (pgq_mlp_f16_decode)"),
            "one_launch_graph_us_per_step": round(ms_one * 1e3, 2),
            "two_launch_graph_us_per_step": round(ms_two * 1e3, 2),
            "two_launch_direct_us_per_step": round(ms_direct * 1e3, 2),
            "note": "launch-latency bound (4 MiB is 0.6 us at HBM peak); weights rotate over 64 copies"}


def bench_q82f_layer(torch, pgq, synth, steps, warmup, pk):
    """The decode layer's shapes in the pages' q8_2f format (int8 body, row scale,
    column field): one CUDA graph of `steps` layer calls (two launches each, weights
    loaded once, three weight copies in rotation), like the headline."""
    c = synth.Q8_LAYER
    H, KV, I, wl = c["hidden"], c["kv"], c["inter"], c["workload"]
    base = synth.q82f_layer(wl, 0, H, KV, I, "torch", "cuda")
    copies = [base] + [{s: tuple(t.clone() for t in m) for s, m in base.items()} for _ in range(2)]
    structs = [pgq.q82f_layer_struct(m) for m in copies]
    x = synth.normal((H,), 1.0, wl, synth.T_X, "torch", "cuda")
    xo = synth.normal((H,), 1.0, wl, synth.T_XO, "torch", "cuda")
    g = synth.gamma(H, wl, backend="torch", device="cuda")
    f = lambda n: torch.empty(n, dtype=torch.float32, device="cuda")  # noqa: E731
    out = dict(q=f(H), k=f(KV), v=f(KV), o=f(H), u=f(I), down=f(H))
    it = [0]

    def step():
        L = structs[it[0] % len(structs)]
        it[0] += 1
        pgq.q82f_decode_layer(L, x, xo, g, 1e-6, out=out, weights_stable=True)

    g_warm = _capture(torch, lambda: [step() for _ in range(warmup)])
    g_all = _capture(torch, lambda: [step() for _ in range(steps)])
    g_all.replay()
    g_warm.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = _events(torch, 2)
    a.record(st)
    g_all.replay()
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = sum(r * cc + 2 * r + 2 * cc for r, cc in synth.q8_layer_shapes(H, KV, I).values())
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "q8_2f decode layer B=1 (hidden 4096, kv 1024, inter 14336; int8 body, f16 row scale, "
                        "f16 column field)", "metric": "weight GB/s", "value": round(gbs, 1),
            "us_per_step": round(ms * 1e3, 3), "frac_of_hbm": round(gbs / pk["hbm"], 4), "weight_bytes": nbytes,
            "launches_per_step": 2, "timed": "one CUDA graph of the K steps, three weight copies in rotation"}


def bench_vocab(torch, pgq, synth, steps, warmup, pk):
    c = synth.VOCAB
    V, H, wl = c["vocab"], c["hidden"], c["workload"]
    W = synth.f16_matrix(V, H, wl, synth.T_W, "torch", "cuda")
    g = synth.gamma(H, wl, backend="torch", device="cuda")
    out = {}
    for B in (1, 8):
        x = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
        ids = torch.empty(B, dtype=torch.int32, device="cuda")
        ws = torch.empty(pgq.argmax_workspace_bytes(B), dtype=torch.uint8, device="cuda")
        fn = lambda: pgq.gemv_f16_argmax(W, x, gamma=g, logits=False, workspace=ws, ids=ids)  # noqa: E731
        ms = time_loop(torch, fn, max(5, steps // 2), warmup)
        gbs = W.numel() * 2 / (ms * 1e-3) / 1e9
        out[f"B{B}"] = {"workload": f"vocab head 262144 x 4096 f16, B={B}, fused RMSNorm + argmax",
                        "metric": "weight GB/s", "value": round(gbs, 1), "us_per_step": round(ms * 1e3, 2),
                        "frac_of_hbm": round(gbs / pk["hbm"], 4), "weight_bytes": W.numel() * 2,
                        "launches_per_step": 1}
    return out


def bench_moe(torch, pgq, synth, steps, warmup, pk, graph=True, q82f=False):
    """The MoE prefill layer (q82f: with q8_2f experts, the q8_2f bank payload)."""
    c = synth.MOE
    E, H, I, B, k, wl = c["experts"], c["hidden"], c["inter"], c["B"], c["topk"], c["workload"]
    router, up, down = (synth.moe_q82f_layer if q82f else synth.moe_layer)(wl, E, H, I, "torch", "cuda")
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
    g1 = synth.gamma(H, wl, backend="torch", device="cuda")
    g2 = synth.gamma(H, wl, synth.T_GAMMA2, "torch", "cuda")
    Wm = pgq.MoeQ82Weights(router, up, down, k) if q82f else pgq.MoeWeights(router, up[0], up[1], down[0], down[1], k)
    h = h0.clone()
    y = torch.empty_like(h0)
    ws = pgq.moe_layer_workspace(Wm, B)

    def step():
        h.copy_(h0)
        pgq.moe_prefill_layer(Wm, h, g1, g2, 1e-6, y=y, workspace=ws)

    ms = time_loop(torch, step, steps, warmup)
    ms_graph = time_graph(torch, step, steps, warmup) if graph else ms
    taps = pgq.moe_layer_taps(Wm, ws, B)
    touched = int((taps["counts"] > 0).sum().item())
    per_expert = 2 * (I * H + 2 * (I + H)) if q82f else 2 * (I * H + I * (H // 32) * 4)
    nbytes = touched * per_expert + E * H * 4
    gbs = nbytes / (ms_graph * 1e-3) / 1e9
    fmt = "q8_2f" if q82f else "q8"
    return {"workload": f"MoE prefill layer B=64 (hidden 2688, 128 experts of 1856x2688 {fmt}, top-6)",
            "metric": "positions/s", "value": round(B / (ms_graph * 1e-3), 1), "ms_per_layer": round(ms_graph, 4),
            "ms_per_layer_api": round(ms, 4), "touched_experts": touched, "weight_bytes": nbytes,
            "weight_GBps": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4), "launches_per_step": 7,
            "timed": ("CUDA-graph replay of the layer call (ms_per_layer_api: direct calls)" if graph
                      else "direct calls (no graph)")}


def time_q8_layer_fused(torch, pgq, W, steps, warmup):
    """ms per step of the one-launch form of the layer: one CUDA graph of `steps`
    calls over the rotating weight copies (after a warm-up replay)."""
    sync = pgq.layer_sync()
    structs = [pgq.q8_layer_struct(L) for L in W.layers]
    n = len(structs)

    def steps_of(k):
        for i in range(k):
            pgq.q8_decode_layer_fused(structs[i % n], W.x[0], W.xo[0], W.g, 1e-6, sync=sync, out=W.out1,
                                      weights_stable=True)

    g_all = _capture(torch, lambda: steps_of(steps))
    for _ in range(max(1, warmup // steps + 1)):
        g_all.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = _events(torch, 2)
    a.record(st)
    g_all.replay()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def time_e2e(torch, W, steps, warmup):
    W.e2e_setup()
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        W.e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(steps):
        W.e2e_step()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _host_layer_sample(frac):
    """A row sample of the decode layer's six q8 matrices drawn on the host (same
    recipe as the device copies), with its inputs; ``frac`` of each matrix's rows."""
    import synth
    c = synth.Q8_LAYER
    H, KV, I, wl = c["hidden"], c["kv"], c["inter"], c["workload"]
    mats, nb = {}, 0
    for s, (r, cc) in synth.q8_layer_shapes(H, KV, I).items():
        rr = max(4, int(r * frac))
        codes, params = synth.q8_matrix(rr, cc, wl, synth.q8_tensor_id(0, s))
        mats[s] = (codes, params)
        nb += codes.size + params.size * 2
    x = synth.normal((H,), 1.0, wl, synth.T_X)
    xo = synth.normal((H,), 1.0, wl, synth.T_XO)
    g = synth.gamma(H, wl)
    u = np.abs(synth.normal((I,), 1.0, wl, 99))
    return mats, x, xo, g, u, nb


def _time_oracle_sample(frac, reps=1):
    """Seconds of ``reps`` oracle passes over the row sample, and their weight bytes."""
    import oracle
    mats, x, xo, g, u, nb = _host_layer_sample(frac)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.q8_decode_layer(x, xo, g, 1e-6, mats, u_in=u)
    return time.perf_counter() - t0, nb * reps


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_q8(target_s=12.0):
    """The oracle as it stands, timed on the host cores on a row sample of the decode
    layer: with every core numpy uses (its matmuls are multi-threaded), and in a child
    process limited to one thread."""
    frac = 0.02
    dt, _ = _time_oracle_sample(frac)
    frac = min(1.0, frac * max(1.0, target_s / max(dt, 1e-3)))   # about target_s of work:
    dt, _ = _time_oracle_sample(frac)                            # a larger sample, then
    reps = max(1, min(30, int(round(target_s / max(dt, 1e-3)))))   # whole passes repeated
    dt, nb = _time_oracle_sample(frac, reps)
    one = None
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", repr(frac),
                            "--cpu-reps", str(reps)], env=env,
                           capture_output=True, text=True, timeout=600)
        rec = json.loads(r.stdout.strip().splitlines()[-1])
        one = dict(value=round(rec["bytes"] / rec["seconds"] / 1e9, 4), unit="GB/s", threads=1,
                   seconds=round(rec["seconds"], 2))
    except Exception as exc:   # reported, not fatal: the all-core figure stands
        one = dict(error=f"one-thread run failed: {type(exc).__name__}")
    return dict(value=round(nb / dt / 1e9, 4), unit="GB/s", cores=os.cpu_count(), threads=os.cpu_count(),
                kind="oracle", cpu_model=cpu_model(), one_thread=one,
                sample=f"{frac:.3f} of the rows of each of the decode layer's six q8 matrices, {reps} pass(es) "
                       f"({nb} weight bytes), {dt:.1f} s with all cores; numpy f64 oracle (matmuls multi-threaded, the rest "
                       f"single-threaded); one_thread: the same sample with every thread pool set to 1")


# ------------------------------------------------------------------ main
def max_over_ranks(torch, dist, vals, device):
    """Every rank's timings, after a barrier, replaced by their maximum over the ranks
    (the whole job is as fast as its slowest rank); one rank: the values as they are."""
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if dist is not None:
        dist.barrier()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(world, bytes_per_step, ms_per_step):
    """Whole-job weight GB/s: every rank streams bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pgq", choices=["pgq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true", help="only the headline decode layer")
    ap.add_argument("--only", choices=["decode", "prefill", "moe", "vocab", "q82f", "q82f_prefill", "q82f_moe"],
                    default=None,
                    help="profiling aid: run one workload and print its JSON object")
    ap.add_argument("--no-graph", action="store_true", help="profiling aid (--only moe): direct calls only")
    ap.add_argument("--prefill-layers", type=int, default=None, help="layers of the prefill pass (default 32)")
    ap.add_argument("--cpu-worker", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-reps", type=int, default=1, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker is not None:   # the one-thread oracle timing (a child of cpu_baseline_q8)
        dt, nb = _time_oracle_sample(args.cpu_worker, args.cpu_reps)
        print(json.dumps({"seconds": dt, "bytes": nb}), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import synth
    import prefill_gemv_q8_gb300 as pgq
    from prefill_gemv_q8_gb300 import build
    build.build()
    if pgq.lib().pgq_device_check() != pgq.OK:
        raise SystemExit("libpgq: " + pgq.lib().pgq_last_error().decode())

    pk = peaks()
    if args.only == "prefill":
        P = PrefillPass(torch, pgq, synth, layers=args.prefill_layers)
        print(json.dumps(time_prefill(torch, P, args.steps, args.warmup, pk)), flush=True)
        return
    if args.only == "q82f_prefill":
        P = PrefillPassQ82F(torch, pgq, synth, layers=args.prefill_layers)
        print(json.dumps(time_prefill_q82f(torch, P, args.steps, args.warmup, pk)), flush=True)
        return
    if args.only == "q82f_moe":
        print(json.dumps(bench_moe(torch, pgq, synth, args.steps, args.warmup, pk, graph=not args.no_graph, q82f=True)),
              flush=True)
        return
    if args.only == "moe":
        print(json.dumps(bench_moe(torch, pgq, synth, args.steps, args.warmup, pk, graph=not args.no_graph)),
              flush=True)
        return
    if args.only == "q82f":
        print(json.dumps(bench_q82f_layer(torch, pgq, synth, args.steps, args.warmup, pk)), flush=True)
        return
    if args.only == "vocab":
        print(json.dumps(bench_vocab(torch, pgq, synth, args.steps, args.warmup, pk)), flush=True)
        return
    W = Q8DecodeLayer(torch, pgq, synth)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with Clocks(local) as clk:
        total_ms, k1_ms, k2_ms = time_q8_layer(torch, W, args.steps, args.warmup)
    clocks = clk.summary()
    fused_ms = time_q8_layer_fused(torch, pgq, W, args.steps, args.warmup)
    e2e_ms = time_e2e(torch, W, args.steps, args.warmup)
    total_ms, e2e_ms = max_over_ranks(torch, dist, [total_ms, e2e_ms], "cuda")
    ms_step = total_ms / args.steps
    value = job_gbs(world, W.step_bytes, ms_step)
    achieved = W.k1_bytes / (k1_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "q8 weights (int8 + f16 scale/offset), f32 arithmetic", "data": "synthetic",
        "config": {"workload": W.name, "weight_bytes_per_step": W.step_bytes, "B": 1,
                   "l2": "weights rotate over 3 copies (538 MB > 129 MB L2)", "launches_per_step": 2,
                   "timing": "one CUDA graph of the K timed steps (2 launches each, weight copies in rotation), "
                             "uploaded by an untimed replay, after W warm-up steps",
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm": round(value / world / pk["hbm"], 4),
        "roofline": {"bound": "hbm", "kernel": "pgq_gemv_tma_kernel<q8,B=1> (norm + q,k,v,o,up)",
                     "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm"], 4), "peak_src": pk["src"],
                     "traffic": ncu_traffic("gemv_q8_layer_multi", Q8_FILES),
                     "algorithmic_bytes_per_launch": W.k1_bytes, "avg_launch_ms": round(k1_ms, 5),
                     "down_launch_ms": round(k2_ms, 5)},
        "e2e": {"value": round(job_gbs(world, W.step_bytes, e2e_ms), 1), "unit": "GB/s",
                "h2d_bytes_per_step": W.h2d, "d2h_bytes_per_step": W.d2h, "ms_per_step": round(e2e_ms, 5)},
        "one_launch_form": {"entry": "pgq_q8_decode_layer_fused", "us_per_step": round(fused_ms * 1e3, 3),
                            "value": round(W.step_bytes / (fused_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                            "note": "the same layer in one persistent launch (device-side dependency); "
                                    "slower than the two programmatic-dependent launches here"},
        "gpu_launches": W.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.skip_prefill and args.only != "decode":
        P = PrefillPass(torch, pgq, synth, layers=args.prefill_layers)
        with Clocks(local) as clk2:
            pre = time_prefill(torch, P, max(3, args.steps // 5), args.warmup, pk)
        pre["clocks"] = clk2.summary()
        line["workloads"] = {"prefill_pass": pre}
        del P
        torch.cuda.empty_cache()
        line["workloads"]["moe_layer"] = bench_moe(torch, pgq, synth, max(5, args.steps // 5), args.warmup, pk)
        torch.cuda.empty_cache()
        line["workloads"]["vocab_head"] = bench_vocab(torch, pgq, synth, args.steps, args.warmup, pk)
        torch.cuda.empty_cache()
        line["workloads"]["tiny_mlp"] = bench_tiny_mlp(torch, pgq, synth, args.steps, args.warmup, pk)
        torch.cuda.empty_cache()
        line["workloads"]["q8_2f_decode_layer"] = bench_q82f_layer(torch, pgq, synth, args.steps, args.warmup, pk)
        torch.cuda.empty_cache()
        P = PrefillPassQ82F(torch, pgq, synth, layers=args.prefill_layers)
        line["workloads"]["q8_2f_prefill_pass"] = time_prefill_q82f(torch, P, max(3, args.steps // 5), args.warmup,
                                                                    pk)
        del P
        torch.cuda.empty_cache()
        line["workloads"]["q8_2f_moe_layer"] = bench_moe(torch, pgq, synth, max(5, args.steps // 5), args.warmup, pk,
                                                         q82f=True)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_q8()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_reference(args, rank, world):
    """The oracle timed on the host cores, on the headline workload's metric."""
    if rank != 0:
        return
    import torch
    import synth

    class HostLayer:
        def __init__(self):
            self.mats, self.x, self.xo, self.g, self.u, self.nbytes = _host_layer_sample(1.0 / 8)

    import oracle
    Wh = HostLayer()
    for _ in range(args.warmup):
        oracle.q8_decode_layer(Wh.x, Wh.xo, Wh.g, 1e-6, Wh.mats, u_in=Wh.u)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.q8_decode_layer(Wh.x, Wh.xo, Wh.g, 1e-6, Wh.mats, u_in=Wh.u)
    dt = (time.perf_counter() - t0) / args.steps
    v = Wh.nbytes / dt / 1e9
    sample = (f"1/8 of the rows of each q8 matrix of the decode layer ({Wh.nbytes} weight bytes) per step; "
              "numpy f64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": Q8DecodeLayer.name, "B": 1},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": os.cpu_count(), "threads": os.cpu_count(),
                         "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    del torch


if __name__ == "__main__":
    main()
