#!/usr/bin/env python3
"""Benchmark of the attention-block library on the 8-layer SSSL stack.

Workload (one "step"): the attention blocks of an 8-layer GPT with window
pattern "SSSL" at B=16, T=2048, Hq=6, Hkv=3, d=128: forward of layers 0..7,
then backward of layers 7..0. Layers 0,1,2,4,5,6 use a causal window of
T/2 = 1024, layers 3 and 7 full causal attention; layers 1,3,5,7 add
0.5 * VE[token] to v (VE table 8192 x 384 bf16 per layer). QK-RMSNorm gains
~ 1 + 0.1 N(0,1). Seeded synthetic inputs (no dataset).

Metric: masked (in-band) TFLOP/s of fwd + bwd, counting 4 d P B Hq FLOPs for
the forward and 10 d P B Hq for the backward (the flash-attention convention,
S recomputed), where P = sum_i (min(i, W) + 1) is the number of visible
(query, key) pairs of one head.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) each rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sliding_window_gqa_qk_gb300.inputs import Problem, make_inputs  # noqa: E402

N_LAYER, PATTERN = 8, "SSSL"
B, T, HQ, HKV, D = 16, 2048, 6, 3, 128
VOCAB, VE_SCALE = 8192, 0.5
METRIC = "masked TFLOP/s fwd+bwd, T=2048 SSSL layers; % of GB300 bf16 tensor-core peak"
WORKLOAD = "8-layer SSSL stack (B=16, T=2048, Hq=6, Hkv=3, d=128, W=1024 on S layers, VE on odd layers)"

# Counters of the dominant kernel (bwd_tc128_kernel) from one ncu capture of
# an S-layer launch (6 of the stack's 8 layers are S layers), summarised in
# profiles/bwd_tc128_s_layer.md: DRAM traffic (dram__bytes_read.sum +
# dram__bytes_write.sum) per launch, tensor-pipe activity
# (sm__pipe_tensor_cycles_active, % of elapsed cycles) and DRAM throughput.
# "source_sha" is kernel_source_sha() of the build that was captured: when
# the kernel's sources have changed since, the bench line reports these as
# null.
NCU_CAPTURE = {
    "source_sha": "ebd410cd4fe49928",
    "traffic_bytes": 429_616_896,
    "tensor_pipe_pct": 39.9,
    "dram_gbs": 1909.5,
    "summary": "profiles/bwd_tc128_s_layer.md (S-layer launch)",
}
KERNEL_SOURCES = ("tc_bwd128.cuh", "tc_bwd.cuh", "tc_fwd.cuh", "ptx.cuh", "common.cuh")


def kernel_source_sha() -> str:
    """SHA-256 (first 16 hex digits) of the dominant kernel's source files."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sliding_window_gqa_qk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_evidence():
    """The captured counters when they belong to the current build, else nulls."""
    ok = NCU_CAPTURE["source_sha"] is not None and NCU_CAPTURE["source_sha"] == kernel_source_sha()
    keys = ("traffic_bytes", "tensor_pipe_pct", "dram_gbs")
    out = {k: (NCU_CAPTURE[k] if ok else None) for k in keys}
    out["summary"] = NCU_CAPTURE["summary"] if ok else None
    return out


def layer_schedule(window_fn, ve_fn):
    return [(window_fn(i, N_LAYER, PATTERN, T), bool(ve_fn(i, N_LAYER))) for i in range(N_LAYER)]


def pairs(Tn: int, W: int) -> int:
    """Visible (query, key) pairs of one head, causal, window W (-1: none)."""
    if W < 0 or W >= Tn - 1:
        return Tn * (Tn + 1) // 2
    # rows i <= W see i + 1 keys, rows beyond see W + 1
    return (W + 1) * (W + 2) // 2 + (Tn - W - 1) * (W + 1)


def flops(Bn, Tn, Hq, d, W):
    P = pairs(Tn, W)
    return 4 * d * P * Bn * Hq, 10 * d * P * Bn * Hq


def block_gemm_flops(rows, C, nq, nkv):
    """FLOPs of one block layer's projections, forward and backward: the
    forward's q, k, v and output projections (2 rows C (nq + 2 nkv) and
    2 rows nq C), twice that in the backward (each weight's gradient and
    each input's gradient)."""
    fwd = 2 * rows * C * (nq + 2 * nkv) + 2 * rows * nq * C
    return 3 * fwd


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in samples taken
        between t0 and t1 (wall clock; all samples when not given)."""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if t0 is not None and not (t0 <= ts <= t1 + 0.25):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax = float(parts[3])
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Oracle leg (CPU baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample(schedule, layers=None, batch=1, kv_heads=1, Tn=T, G=HQ // HKV, d=D, gain_std=0.1):
    """Runs the float64 oracle on a slice of a workload's layers: `batch`
    sequences of Tn positions and `kv_heads` kv heads (G query heads each).
    Returns (seconds, masked FLOPs of the sample, description)."""
    import numpy as np  # noqa: F401
    import oracle
    from sliding_window_gqa_qk_gb300.inputs import as_f64
    layers = list(range(len(schedule))) if layers is None else layers
    total_t, total_f = 0.0, 0
    for li in layers:
        W, ve = schedule[li]
        p = Problem(B=batch, T=Tn, Hq=kv_heads * G, Hkv=kv_heads, d=d, window=W,
                    gain_std=gain_std, ve=ve, vocab=VOCAB)
        x = make_inputs(p, layer=li, seed=4242)
        f = {k: as_f64(t) for k, t in x.items()}
        tok = x["tok"].numpy() if x["tok"] is not None else None
        kw = dict(window=W, eps=p.eps, ve=f["ve"], tok=tok, ve_scale=VE_SCALE)
        t0 = time.perf_counter()
        oracle.attention_forward(f["q"], f["k"], f["v"], f["gq"], f["gk"], **kw)
        oracle.attention_backward(f["q"], f["k"], f["v"], f["gq"], f["gk"], f["dO"], **kw)
        total_t += time.perf_counter() - t0
        ff, fb = flops(batch, Tn, kv_heads * G, d, W)
        total_f += ff + fb
    desc = (f"float64 oracle fwd+bwd of layers {layers} of the workload on a slice of "
            f"B={batch}, T={Tn}, Hq={kv_heads * G}, Hkv={kv_heads}, d={d}")
    return total_t, total_f, desc


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

WORKLOADS = {
    "stack": WORKLOAD,
    "s_layer": "one S layer (B=16, T=2048, Hq=6, Hkv=3, d=128, window 1024, no VE)",
    "l_layer": "one L layer (B=16, T=2048, Hq=6, Hkv=3, d=128, full causal, no VE)",
    "stack_rope": WORKLOAD[:-1] + ", rotary tables (base 10000) fused before the QK-norm)",
    "stack_full": WORKLOAD[:-1] + ", rotary tables, learned VE gate 2 sigmoid(W x[:32]) on the VE layers)",
    "stack_mha": WORKLOAD.replace("Hkv=3", "Hkv=6") + " with Hkv = Hq (the Guide's default n_kv_head = n_head)",
    "long": ("long context: one S layer (window 8192) and one L layer (full causal), B=2, T=16384, "
             "Hq=16, Hkv=4, d=128, QK-RMSNorm gains 1+0.1N, no VE"),
    "tiny": ("tiny: one layer B=1, T=256, Hq=2, Hkv=1, d=64, window 128, unit gains, no VE "
             "(latency-bound: 3 query tiles)"),
    "block_stack": ("8 whole attention blocks (pre-norm, c_q / c_k / c_v, attention, c_proj, "
                    "residual) at C=768: B=16, T=2048, Hq=6, Hkv=3, d=128, SSSL windows, rotary "
                    "tables, VE with the learned gate on odd layers"),
    "block_layer": ("one whole attention block (layer 1 of the block stack: window 1024, rotary, "
                    "VE with the learned gate) at C=768, B=16, T=2048, Hq=6, Hkv=3, d=128 (profiling)"),
}

# (B, T, Hq, Hkv) of each workload; d = 128 throughout
LONG_SHAPE = (2, 16384, 16, 4)


def shape_for(workload):
    if workload == "long":
        return LONG_SHAPE
    if workload == "tiny":
        return (1, 256, 2, 1)
    return (B, T, HQ, HQ if workload == "stack_mha" else HKV)


def head_dim_for(workload):
    """(head dim, gain std: None for unit gains) of a workload."""
    return (64, None) if workload == "tiny" else (D, 0.1)


def schedule_for(workload, window_fn, ve_fn):
    if workload == "s_layer":
        return [(T // 2, False)]
    if workload == "l_layer":
        return [(-1, False)]
    if workload == "tiny":
        return [(128, False)]
    if workload == "long":
        # one layer of each kind of the SSSL pattern at T = 16384
        t_long = LONG_SHAPE[1]
        return [(window_fn(0, N_LAYER, PATTERN, t_long), False),
                (window_fn(N_LAYER - 1, N_LAYER, PATTERN, t_long), False)]
    return layer_schedule(window_fn, ve_fn)


class Stack:
    def __init__(self, swa, dev, workload="stack"):
        self.swa = swa
        self.dev = dev
        Bn, Tn, hq, hkv = shape_for(workload)
        self.B, self.T, self.hq, self.hkv = Bn, Tn, hq, hkv
        d, gain_std = head_dim_for(workload)
        self.d = d
        # inputs smaller than L2: flush it before every timed step
        self.small = workload == "tiny"
        self.rope = None
        self.learned_gate = workload == "stack_full"
        if workload in ("stack_rope", "stack_full"):
            # standard rotary tables: angle t * 10000^(-2c/d), positions 0..T-1
            inv = 10000.0 ** (-torch.arange(D // 2, dtype=torch.float64) * 2.0 / D)
            ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
            self.rope_t = (torch.cos(ang).float().to(dev).contiguous(),
                           torch.sin(ang).float().to(dev).contiguous())
            self.rope = swa.make_extras(rope=self.rope_t)
        self.sched = schedule_for(workload, swa.swa_sssl_window, swa.swa_has_ve)
        self.layers = []
        for li, (W, ve) in enumerate(self.sched):
            p = Problem(B=Bn, T=Tn, Hq=hq, Hkv=hkv, d=d, window=W, gain_std=gain_std, ve=ve,
                        vocab=VOCAB)
            x = make_inputs(p, layer=li)
            g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
            prm = swa.make_params(Bn, Tn, hq, hkv, d, W, True, 0.0, p.eps, VE_SCALE,
                                  VOCAB if ve else 0)
            ws = swa.new_workspace(prm, True, dev, "bf16")
            L = dict(p=p, prm=prm, x=x, g=g, ws=ws)
            L["o"] = torch.empty_like(g["q"])
            L["lse"] = torch.empty(Bn, hq, Tn, dtype=torch.float32, device=dev)
            L["dq"], L["dk"], L["dv"] = (torch.empty_like(g["q"]), torch.empty_like(g["k"]),
                                         torch.empty_like(g["v"]))
            L["dgq"] = torch.empty(d, dtype=torch.float32, device=dev)
            L["dgk"] = torch.empty(d, dtype=torch.float32, device=dev)
            L["dve"] = (torch.empty(g["ve"].shape, dtype=torch.float32, device=dev) if ve else None)
            L["ex"] = self.rope
            if self.learned_gate and ve:
                # block input rows [B, T, 768] (the gate reads 32 channels) and
                # gate weights [Hkv, 32], seeded per layer
                gen = torch.Generator().manual_seed(1000 + li)
                L["gx"] = torch.randn(B, T, 768, generator=gen).to(torch.bfloat16).to(dev)
                L["gw"] = (0.1 * torch.randn(hkv, 32, generator=gen)).to(dev)
                L["dgw"] = torch.empty(hkv, 32, dtype=torch.float32, device=dev)
                L["dgx"] = torch.empty(B, T, 32, dtype=torch.float32, device=dev)
                L["ex"] = swa.make_extras(rope=self.rope_t, gate_x=L["gx"], gate_w=L["gw"],
                                          d_gate_w=L["dgw"], d_gate_x=L["dgx"])
            self.layers.append(L)
        self.flops_fwd = sum(flops(Bn, Tn, hq, d, W)[0] for W, _ in self.sched)
        self.flops_bwd = sum(flops(Bn, Tn, hq, d, W)[1] for W, _ in self.sched)

    def layer_gb(self):
        """Device bytes of one layer's tensors (inputs, outputs, gradients,
        workspace), in GB."""
        L = self.layers[0]
        n = L["ws"].numel() * L["ws"].element_size()
        for k in ("o", "lse", "dq", "dk", "dv"):
            n += L[k].numel() * L[k].element_size()
        for t in L["g"].values():
            if t is not None:
                n += t.numel() * t.element_size()
        return n / 1e9

    def fwd(self, L):
        g = L["g"]
        if L["ex"] is not None:
            st = self.swa.swa_attn_fwd_ex(L["prm"], L["ex"], g["q"], g["k"], g["v"], g["gq"], g["gk"],
                                          g["ve"], g["tok"], None, L["o"], L["lse"], L["ws"])
        else:
            st = self.swa.swa_attn_fwd(L["prm"], g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"],
                                       g["tok"], None, L["o"], L["lse"], L["ws"])
        if st != 0:
            raise self.swa.SwaError(st, "swa_attn_fwd")

    def bwd(self, L, stage):
        g = L["g"]
        args = (g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"], g["tok"], None, L["o"], L["lse"],
                g["dO"], L["dq"], L["dk"], L["dv"], L["dgq"], L["dgk"], L["dve"], L["ws"])
        if L["ex"] is not None:
            st = self.swa.swa_attn_bwd_ex(L["prm"], L["ex"], *args,
                                          flags=self.swa.SWA_REUSE_PROLOGUE | stage)
        else:
            st = self.swa.swa_attn_bwd(L["prm"], *args, flags=self.swa.SWA_REUSE_PROLOGUE | stage)
        if st != 0:
            raise self.swa.SwaError(st, "swa_attn_bwd")

    def step(self, ev=None):
        """One fwd+bwd pass over the 8 layers. With ev (a list of CUDA-event
        pairs per stage) the stages are bracketed for per-kernel timing."""
        swa = self.swa
        for L in self.layers:
            if ev is not None:
                ev["fwd"].append(_ev_pair())
                ev["fwd"][-1][0].record()
            self.fwd(L)
            if ev is not None:
                ev["fwd"][-1][1].record()
        for L in reversed(self.layers):
            for name, stage in (("bwd_pre", swa.SWA_BWD_STAGE_PRE),
                                ("bwd_main", swa.SWA_BWD_STAGE_MAIN),
                                ("bwd_post", swa.SWA_BWD_STAGE_POST)):
                if ev is not None:
                    ev[name].append(_ev_pair())
                    ev[name][-1][0].record()
                self.bwd(L, stage)
                if ev is not None:
                    ev[name][-1][1].record()

    # launches of our kernels per layer and step: fwd = prologue + attention;
    # bwd = pre + main + post + gain sum (+ the learned gate's backward and
    # its weight-gradient sum on VE layers)
    LAUNCHES_PER_LAYER = 2 + 4

    def launches_per_step(self):
        return sum(self.LAUNCHES_PER_LAYER + (2 if (self.learned_gate and ve) else 0)
                   for _, ve in self.sched)


class BlockStack:
    """The stack of whole attention blocks: per layer the block forward
    (pre-norm, projections, attention, output projection, residual), then
    the block backwards in reverse layer order, through swa_block_fwd /
    swa_block_bwd."""

    C = 768

    def __init__(self, swa, dev, only_layer=None):
        from sliding_window_gqa_qk_gb300.inputs import make_block_inputs
        self.swa = swa
        C = self.C
        self.sched = layer_schedule(swa.swa_sssl_window, swa.swa_has_ve)
        if only_layer is not None:
            self.sched = [self.sched[only_layer]]
        inv = 10000.0 ** (-torch.arange(D // 2, dtype=torch.float64) * 2.0 / D)
        ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
        self.rope = (torch.cos(ang).float().to(dev).contiguous(),
                     torch.sin(ang).float().to(dev).contiguous())
        f32 = dict(dtype=torch.float32, device=dev)
        self.layers = []
        for li, (W, ve) in enumerate(self.sched):
            p = Problem(B=B, T=T, Hq=HQ, Hkv=HKV, d=D, window=W, gain_std=0.1, ve=ve, vocab=VOCAB)
            x = make_block_inputs(p, C, layer=li if only_layer is None else only_layer,
                                  gate_ch=32 if ve else None)
            g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
            prm = swa.make_params(B, T, HQ, HKV, D, W, True, 0.0, p.eps, VE_SCALE, VOCAB if ve else 0)
            n = swa.swa_block_workspace_size(prm, C, 1)
            ws = torch.empty(n, dtype=torch.uint8, device=dev)
            if swa.swa_attn_workspace_init(ws, n) != 0:
                raise RuntimeError("workspace init")
            L = dict(prm=prm, g=g, ws=ws, out=torch.empty_like(g["x"]), dx=torch.empty_like(g["x"]))
            for k in ("wq", "wk", "wv", "wo"):
                L["d" + k] = torch.empty(g[k].shape, **f32)
            L["dgq"], L["dgk"] = torch.empty(D, **f32), torch.empty(D, **f32)
            L["dve"] = torch.empty(g["ve"].shape, **f32) if ve else None
            L["dgate_w"] = torch.empty(g["gate_w"].shape, **f32) if ve else None
            L["ex"] = swa.make_block_extras(rope=self.rope, gate_w=g["gate_w"], d_gate_w=L["dgate_w"])
            L["w"] = swa.make_block_weights(g["wq"], g["wk"], g["wv"], g["wo"])
            self.layers.append(L)
        self.flops_attn = sum(sum(flops(B, T, HQ, D, W)) for W, _ in self.sched)
        self.flops_gemm = len(self.sched) * block_gemm_flops(B * T, C, HQ * D, HKV * D)
        self.flops = self.flops_attn + self.flops_gemm

    def fwd(self, L):
        g = L["g"]
        st = self.swa.swa_block_fwd(L["prm"], L["ex"], L["w"], g["x"], g["gq"], g["gk"], g["ve"],
                                    g["tok"], L["out"], L["ws"])
        if st != 0:
            raise self.swa.SwaError(st, "swa_block_fwd")

    def bwd(self, L):
        g = L["g"]
        st = self.swa.swa_block_bwd(L["prm"], L["ex"], L["w"], g["x"], g["gq"], g["gk"], g["ve"],
                                    g["tok"], g["dout"], L["dx"], L["dwq"], L["dwk"], L["dwv"],
                                    L["dwo"], L["dgq"], L["dgk"], L["dve"], L["ws"])
        if st != 0:
            raise self.swa.SwaError(st, "swa_block_bwd")

    def step(self, ev=None):
        for L in self.layers:
            if ev is not None:
                ev["fwd"].append(_ev_pair())
                ev["fwd"][-1][0].record()
            self.fwd(L)
            if ev is not None:
                ev["fwd"][-1][1].record()
        for L in reversed(self.layers):
            if ev is not None:
                ev["bwd"].append(_ev_pair())
                ev["bwd"][-1][0].record()
            self.bwd(L)
            if ev is not None:
                ev["bwd"][-1][1].record()


def run_block_stack(args, rank, world, dev):
    """Times the block stack (or one block layer): one step's launches
    captured in a CUDA graph and replayed."""
    import sliding_window_gqa_qk_gb300 as swa
    swa.load("bf16")
    stack = BlockStack(swa, dev, only_layer=1 if args.workload == "block_layer" else None)
    start, stop = _ev_pair()
    ev = {"fwd": [], "bwd": []}
    with ClockSampler(_physical_index(torch.cuda.current_device())) as clocks:
        for _ in range(args.warmup):
            stack.step()
        for L in stack.layers:
            st = swa.swa_attn_check_status(L["ws"])
            if st != swa.SWA_OK:
                raise swa.SwaError(st, "device status after warm-up")
        graph = None
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                stack.step()
            graph.replay()
        torch.cuda.synchronize()
        _barrier(world)
        t0 = clocks.mark()
        start.record()
        for _ in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                stack.step()
        stop.record()
        torch.cuda.synchronize()
        t1 = clocks.mark()
        for _ in range(args.steps):
            stack.step(ev)
        torch.cuda.synchronize()
    _barrier(world)
    ms = _max_over_ranks(start.elapsed_time(stop), world) / args.steps
    stage_ms = {k: sum(a.elapsed_time(b) for a, b in v) / args.steps for k, v in ev.items()}
    value = _aggregate(stack.flops, world, ms)
    peaks, peak_kind = load_peaks()
    peak = peaks["bf16_tflops"]
    return {
        "metric": "TFLOP/s fwd+bwd of the whole attention block (masked attention + projections)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "global_batch": B * world, "seq_len": T,
                   "parallelism": "single GPU" if world == 1 else f"replicas over batch x{world}",
                   "l2": "inputs larger than L2", "flops_per_step": stack.flops,
                   "attention_flops_per_step": stack.flops_attn,
                   "projection_flops_per_step": stack.flops_gemm,
                   "attention_only_tflops": round(stack.flops_attn * world / (ms * 1e-3) / 1e12, 2),
                   "pct_of_peak": round(100 * value / world / peak, 2), "peak_tflops": peak,
                   "peak_source": f"{peak_kind} bf16_tflops (burst)",
                   "launch": ("one step's launches captured in a CUDA graph, replayed per step"
                              if graph is not None else "eager launches"),
                   "stage_ms_per_step": {k: round(v, 4) for k, v in stage_ms.items()},
                   "projections": "the library's tcgen05 GEMM (bf16 operands, fp32 accumulation)"},
        "clocks": clocks.summary(t0, t1),
    }


def _ev_pair():
    return (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))


def run_ours(args, rank, world, dev):
    import sliding_window_gqa_qk_gb300 as swa
    swa.load("bf16")
    stack = Stack(swa, dev, args.workload)
    n_layer = len(stack.sched)
    torch.cuda.synchronize()
    ev = {k: [] for k in ("fwd", "bwd_pre", "bwd_main", "bwd_post")}
    start, stop = _ev_pair()
    gpu_index = torch.cuda.current_device()
    # The clock sampler runs from the warm-up on; only samples taken inside
    # the timed region are summarised.
    with ClockSampler(_physical_index(gpu_index)) as clocks:
        for _ in range(args.warmup):
            stack.step()
        for L in stack.layers:
            st = swa.swa_attn_check_status(L["ws"])
            if st != swa.SWA_OK:
                raise swa.SwaError(st, "device status after warm-up")
        graph = None
        if not args.no_graph:
            # one step's launches captured once, replayed per timed step
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                stack.step()
            graph.replay()
        # inputs smaller than L2: a 256 MB write before each step, outside
        # the events, and the steps timed one by one
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if stack.small else None
        per_step = []
        torch.cuda.synchronize()
        _barrier(world)
        t0 = clocks.mark()
        start.record()
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 255)
                per_step.append(_ev_pair())
                per_step[-1][0].record()
            if graph is not None:
                graph.replay()
            else:
                stack.step(ev)
            if flush is not None:
                per_step[-1][1].record()
        stop.record()
        torch.cuda.synchronize()
        t1 = clocks.mark()
        if graph is not None:
            # per-stage split from eager steps bracketed by events
            for _ in range(args.steps):
                stack.step(ev)
            torch.cuda.synchronize()
    _barrier(world)
    for L in stack.layers:
        st = swa.swa_attn_check_status(L["ws"])
        if st != swa.SWA_OK:
            raise swa.SwaError(st, "device status after the timed steps")
    ms_total = (sum(a.elapsed_time(b) for a, b in per_step) if per_step
                else start.elapsed_time(stop))
    ms = _max_over_ranks(ms_total, world) / args.steps
    stage_ms = {k: sum(a.elapsed_time(b) for a, b in v) / args.steps for k, v in ev.items()}
    flops_step = stack.flops_fwd + stack.flops_bwd
    value = _aggregate(flops_step, world, ms)

    # dominant kernel: the backward main kernel (per launch = one layer). The
    # timed region is well under a second at full clock, so the denominator
    # is the measured burst bf16 peak; the sustained one is reported beside it.
    peaks, peak_kind = load_peaks()
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    ncu = ncu_evidence() if args.workload == "stack" else {
        "traffic_bytes": None, "tensor_pipe_pct": None, "dram_gbs": None, "summary": None}
    bwd_main_launch_ms = stage_ms["bwd_main"] / n_layer
    achieved = stack.flops_bwd / n_layer / (bwd_main_launch_ms * 1e-3) / 1e12
    fwd_launch_tflops = stack.flops_fwd / (stage_ms["fwd"] * 1e-3) / 1e12

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/dO, gains 1+0.1N, VE N(0,0.02), tokens U[0,8192))",
        "config": {"workload": WORKLOADS[args.workload], "global_batch": stack.B * world,
                   "head_dim": stack.d,
                   "seq_len": stack.T,
                   "parallelism": f"replicas over batch x{world}" if world > 1 else "single GPU",
                   "l2": (f"inputs larger than L2: {n_layer} layer(s) x {stack.layer_gb():.1f} GB of "
                          "tensors per step" if flush is None else
                          "inputs smaller than L2: L2 flushed by a 256 MB write before every "
                          "timed step, steps timed one by one with CUDA events"),
                   "flops_per_step": flops_step,
                   "pct_of_peak": round(100 * value / world / peak, 2),
                   "pct_of_sustained_peak": round(100 * value / world / peak_sus, 2),
                   "strict_tflops": round(value * 12 / 14, 2),
                   "strict_count": "forward 4 d P + backward 8 d P per head (no S recompute): "
                                   "12/14 of the flash-attention count",
                   "peak_tflops": peak, "peak_source": f"{peak_kind} bf16_tflops (burst)",
                   "sustained_peak_tflops": peak_sus,
                   "launch": ("one step's launches captured in a CUDA graph, replayed per step"
                              if graph is not None else "eager launches"),
                   "stage_ms_per_step": {k: round(v, 4) for k, v in stage_ms.items()},
                   "stage_split": "CUDA events around each stage of eager steps",
                   "fwd_tflops": round(fwd_launch_tflops, 1)},
        "roofline": {"kernel": ("bwd_tc128_kernel (backward main, d=128; one launch per layer)"
                                if stack.d == 128 else
                                "bwd_tc_kernel<64> (backward main, d=64; one launch per layer)"),
                     "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "traffic": ncu["traffic_bytes"],
                     "tensor_pipe_pct": ncu["tensor_pipe_pct"],
                     "dram_gbs": ncu["dram_gbs"],
                     "ncu_summary": ncu["summary"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, burst)"},
        "gpu_launches": stack.launches_per_step() * args.steps,
        "clocks": clocks.summary(t0, t1),
    }
    if not args.skip_e2e:
        out["e2e"] = run_e2e(args, stack, world)
    if rank == 0 and world == 1 and not args.skip_cpu:
        if args.workload == "stack":
            if args.quick_cpu:
                t, f, desc = oracle_sample(stack.sched, layers=[0, 3])
            else:
                t, f, desc = oracle_sample(stack.sched, batch=2, kv_heads=HKV)
        else:
            # one sequence and one kv-head group of the workload (the whole
            # problem for tiny); at T = 16384 its first layer only (the oracle
            # forms the full T x T logits of every head)
            g = stack.hq // stack.hkv
            layers = [0] if stack.T > 4096 else None
            t = f = 0
            reps = 0
            while t < 5.0:   # repeated to at least 5 s for a stable rate
                dt, df, desc = oracle_sample(stack.sched, layers=layers, Tn=stack.T, G=g, d=stack.d,
                                             gain_std=head_dim_for(args.workload)[1])
                t, f, reps = t + dt, f + df, reps + 1
            desc += f", {reps} time(s)"
        out["cpu_baseline"] = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s",
                               "cores": cores(), "kind": "oracle", "sample": desc,
                               "seconds": round(t, 2)}
    return out


def run_e2e(args, stack, world):
    """Same metric through the library's host-buffer entry point
    (swa_attn_step_host): per layer one C-ABI call that copies the layer's
    inputs from pinned host memory to the device, runs its forward and
    backward, and copies o, lse and every gradient back, all on one stream.
    The layers go round args.e2e_streams streams, each with its own device
    buffer, so that one layer's uploads, another's kernels and a third's
    downloads run at once; stream order keeps each buffer safe across layers
    and steps."""
    swa = stack.swa
    host_in, host_out = [], []
    h2d = d2h = 0
    for L in stack.layers:
        hin = {}
        for k in ("q", "k", "v", "dO", "gq", "gk", "ve", "tok"):
            t = L["x"][k]
            hin[k] = t.contiguous().pin_memory() if t is not None else None
            if t is not None:
                h2d += t.numel() * t.element_size()
        host_in.append(hin)
        hout = {}
        for k in ("o", "lse", "dq", "dk", "dv", "dgq", "dgk", "dve"):
            t = L[k]
            hout[k] = torch.empty(t.shape, dtype=t.dtype).pin_memory() if t is not None else None
            if t is not None:
                d2h += t.numel() * t.element_size()
        host_out.append(hout)
    n_st = max(1, args.e2e_streams)
    streams = [torch.cuda.Stream() for _ in range(n_st)]
    size = max(swa.swa_attn_step_host_size(L["prm"], "bf16") for L in stack.layers)
    bufs = []
    for s_ in streams:
        b = torch.empty(size, dtype=torch.uint8, device=stack.dev)
        if swa.swa_attn_workspace_init(b, size, s_.cuda_stream, "bf16") != swa.SWA_OK:
            raise RuntimeError("step buffer init failed")
        bufs.append(b)

    def step():
        for i, (L, hin, hout) in enumerate(zip(stack.layers, host_in, host_out)):
            st = swa.swa_attn_step_host(
                L["prm"], L["ex"], hin["q"], hin["k"], hin["v"], hin["gq"], hin["gk"], hin["ve"],
                hin["tok"], None, hin["dO"], hout["o"], hout["lse"], hout["dq"], hout["dk"], hout["dv"],
                hout["dgq"], hout["dgk"], hout["dve"], bufs[i % n_st], size, streams[i % n_st].cuda_stream,
                kind="bf16")
            if st != swa.SWA_OK:
                raise RuntimeError(f"step_host failed: {swa.swa_strerror(st)}")

    comp = torch.cuda.current_stream()
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    _barrier(world)
    a, b = _ev_pair()
    a.record()
    for s_ in streams:
        s_.wait_stream(comp)
    for _ in range(args.steps):
        step()
    for s_ in streams:
        comp.wait_stream(s_)
    b.record()
    torch.cuda.synchronize()
    for s_, buf in zip(streams, bufs):
        st = swa.swa_attn_check_status(buf, s_.cuda_stream, "bf16")
        if st != swa.SWA_OK:
            raise RuntimeError(f"device check: {swa.swa_strerror(st)}")
    ms = _max_over_ranks(a.elapsed_time(b), world) / args.steps
    value = _aggregate(stack.flops_fwd + stack.flops_bwd, world, ms)
    return {"value": round(value, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "pinned host buffers through swa_attn_step_host (one C-ABI call per layer: "
                      "upload, forward, backward, download on one stream); layers go round "
                      f"{n_st} streams"}


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    same workload per step (layers 0 and 3 of one batch/kv-head slice)."""
    import sliding_window_gqa_qk_gb300.inputs  # noqa: F401
    from oracle import sssl_window, has_ve
    sched = layer_schedule(sssl_window, has_ve)
    for _ in range(args.warmup):
        oracle_sample(sched, layers=[0])
    times, fl, desc = [], 0, ""
    for _ in range(args.steps):
        t, fl, desc = oracle_sample(sched, layers=[0, 3])
        times.append(t)
    sec = sum(times) / len(times)
    value = fl / sec / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": B, "seq_len": T,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# Process group plumbing (barrier and max over ranks only)
# ---------------------------------------------------------------------------

def _physical_index(i):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [x for x in vis.split(",") if x.strip()]
        if i < len(parts) and parts[i].strip().isdigit():
            return int(parts[i])
    return i


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world):
    """The maximum of x over the ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _aggregate(flops_per_rank_step, world, ms_per_step):
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="stack",
                    help="stack (the headline); one S / L layer (profiling); the stack with "
                         "rotary, learned gate or Hkv = Hq; long context; the stack of whole "
                         "blocks (projections included)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=4,
                    help="streams (each with its own device buffer) the e2e layers go round")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of replaying a CUDA graph of one step")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--quick-cpu", action="store_true", help="oracle sample of 2 layers only")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if args.workload in ("block_stack", "block_layer"):
        out = run_block_stack(args, rank, world, dev)
    else:
        out = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
