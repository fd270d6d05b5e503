"""Benchmark of the routed-expert FFN decode step on GB300 (and of decode GQA attention).

One step = one pass of the whole path (route -> gather -> gate+up -> down -> combine)
through the C ABI over one decode batch of synthetic tokens. Default workload: the largest
of the expert shapes, DeepSeek-V3 (H=7168, I=2048, E=256, top-8, BF16 weights, 22.5 GB per
layer) at T=512 tokens (16 tokens per expert). The metric is the weight-stream bandwidth:
bytes of the active experts' weights (each read once) per second; tokens/s is reported
beside it. The same JSON line carries a sweep over every (config, T) point of the five
expert workloads (Mixtral-8x7B, Mixtral-8x22B and its skewed variant, DeepSeek-V3, Qwen3-235B
INT8), each with its GB/s, % of peak, tokens/s and the expert call's roofline fraction.

`--op attention` measures decode-phase GQA attention instead (moe_gqa_decode, one new
token per sequence against its key/value cache): one step = one call over the batch;
the metric is the bandwidth of the key/value rows read (each once) per second, with
sequences/s beside it. Default workload: Qwen3-30B-A3B-shaped heads (32 query heads,
4 key/value heads, d = 128), 64 sequences of 512..8192 tokens.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]
        [--config NAME] [--T T] [--no-sweep] [--sweep-configs A,B] [--no-cpu-baseline]
        [--op attention [--attn-config NAME]]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path is not sharded); value = all ranks' bytes / the slowest rank's time.
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_workloads as mw  # noqa: E402

METRIC = "expert-FFN decode weight-stream HBM GB/s (% of peak) and tokens/s, 1 GB300"
METRIC_HOST = ("expert-FFN decode weight-stream GB/s with the expert weights in Grace LPDDR5X, read over "
               "NVLink-C2C (% of the measured host->device copy rate) and tokens/s, 1 GB300")
METRIC_ATTN = "decode GQA attention key/value-cache read GB/s (% of peak) and sequences/s, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def kernels_per_step(cfg, T: int, moe=None) -> int:
    """Launches of one moe_ffn_forward under the library's current policy: 1 for the one-launch decode
    step; otherwise routing (one fused launch for T <= 64 and T*k <= 1024, else top-k and scan), gather
    (INT8: straight into the fp16 copy), the expert kernels (INT8 adds the fp16 copy of h), combine."""
    if moe is not None and cfg.wtype != "int8_residual":
        return moe.moe_ffn_forward_launches(T, cfg.H, cfg.I, cfg.E, cfg.top_k, 0 if cfg.wtype == "bf16" else 1)
    route = 1 if (T <= 64 and T * cfg.top_k <= 1024) else 2
    experts = 2 if cfg.wtype == "bf16" else 3
    return route + 1 + experts + 1


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(total_ms: float, bytes_per_rank: float, tokens_per_rank: float, ws_n: int, device):
    """Whole-job throughput of ws_n independent replicas: every rank's bytes and tokens over the
    slowest rank's time (max over ranks; a collective when ws_n > 1). Returns
    (time_ms, GB/s, tokens/s)."""
    if ws_n > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return (total_ms, ws_n * bytes_per_rank / (total_ms * 1e-3) / 1e9, ws_n * tokens_per_rank / (total_ms * 1e-3))


def c2c_copy_peak(device, gbytes: float = 2.0) -> float:
    """GB/s of a pinned host -> device copy (the copy engines over NVLink-C2C), measured here:
    the ceiling for kernels that read weights in host memory."""
    n = int(gbytes * 1e9)
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device=device)
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    reps = 5
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    gbs = reps * n / (a.elapsed_time(b) * 1e-3) / 1e9
    del src, dst
    return gbs


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s sustained under the power cap (a kernel timed inside back-to-back steps)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (bf16_tflops_sustained)"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback (sustained)"


# the sources of the roofline kernels and of their launches: the expert kernels (all of them, and
# the BF16 family alone, whose captures an INT8-only change leaves valid), the attention kernel
EXPERT_SOURCES = ("expert_tc.cuh", "expert_pair.cuh", "moe_device.cuh", "expert_launch.cu")
BF16_SOURCES = ("expert_tc.cuh", "moe_device.cuh", "expert_launch.cu")
DECODE_SOURCES = ("decode_step.cu", "decode_device.cuh", "route_topk.cuh", "moe_device.cuh")
ATTN_SOURCES = ("gqa_decode.cu", "moe_device.cuh")


def expert_sources(wtype: str):
    """The sources a workload's expert kernels are built from."""
    return BF16_SOURCES if wtype == "bf16" else EXPERT_SOURCES


def _code_only(text: str) -> str:
    """Source text without // and /* */ comments, with each line's whitespace runs collapsed and
    empty lines dropped (the sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    lines = (re.sub(r"\s+", " ", re.sub(r"//.*$", "", ln)).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(sources=EXPERT_SOURCES) -> str:
    """Hash of a kernel's sources, comments left out; a recorded DRAM-traffic figure is used only
    while it matches (a change of code, not of comments, voids it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "routed_expert_ffn_softmax_gb300", "csrc")
    for n in sources:
        with open(os.path.join(csrc, n), encoding="utf-8") as f:
            h.update((n + "\n" + _code_only(f.read())).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, sources=EXPERT_SOURCES):
    """DRAM bytes per launch from a committed ncu capture, if it matches the current kernels."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("kernel_source_hash") == kernel_source_hash(sources):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def run_pipelined(n_steps, h2d_fn, compute_fn, d2h_fn, stream, dev):
    """n_steps end-to-end steps through the C ABI: step i's inputs are copied in from pinned host
    memory (h2d_fn(i, b), on a copy stream), the step runs (compute_fn(i, b), on `stream`) and its
    result is copied back (d2h_fn(i, b), on a second copy stream). Two buffer sets, b = i % 2, so
    that a step's copies overlap its neighbours' compute, as a serving loop overlaps them; every
    copy of every step lies between the two returned events."""
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(h2d)
    for i in range(n_steps):
        b = i & 1
        if i >= 2:
            h2d.wait_event(done[b])  # step i - 2 has read this input buffer
        with torch.cuda.stream(h2d):
            h2d_fn(i, b)
        in_ready[b].record(h2d)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_read[b])  # step i - 2's result has been read back
        compute_fn(i, b)
        done[b].record(stream)
        d2h.wait_event(done[b])
        with torch.cuda.stream(d2h):
            d2h_fn(i, b)
        out_read[b].record(d2h)
    end.record(d2h)  # after the last read-back, which waited for the last step and its inputs
    return start, end


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def per_step_times(step, n, stream):
    """ms of n single steps, each between its own two events (after the timed region: the events
    themselves cost the overlap between steps)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    for i in range(n):
        evs[i].record(stream)
        step(i)
    evs[-1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]


def ffn_forward(moe, cfg, L, x, lg, out, ws, stream):
    """moe_ffn_forward, or moe_ffn_forward_residual for residual-split INT8 weights."""
    if cfg.wtype == "int8_residual":
        moe.moe_ffn_forward_residual(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                                     L["Wr_gate"], L["Wr_up"], L["sr_gate"], L["sr_up"], cfg.top_k, out, ws, stream)
    else:
        moe.moe_ffn_forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                            cfg.top_k, out, ws, stream)


def expert_ffn(moe, cfg, L, xg, r, Y, ws, stream):
    """moe_expert_ffn, or moe_expert_ffn_residual for residual-split INT8 weights."""
    if cfg.wtype == "int8_residual":
        moe.moe_expert_ffn_residual(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"],
                                    L["s_gate"], L["s_up"], L["s_down"], L["Wr_gate"], L["Wr_up"], L["sr_gate"],
                                    L["sr_up"], Y, ws, stream)
    else:
        moe.moe_expert_ffn(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"], L["s_gate"],
                           L["s_up"], L["s_down"], Y, ws, stream)


# ------------------------------------------------------------------ workload
# The (config, T) points of the sweep: every expert shape and token count of the five workloads.
SWEEP_CONFIGS = ("mixtral8x7b", "mixtral8x22b", "mixtral8x22b_skew", "dsv3", "qwen3_int8", "mixtral8x7b_prefill",
                 "dsv3_prefill")
L2_BYTES = 129e6


def auto_copies(cfg: mw.MoEConfig, Ts, max_bytes: float = 120e9) -> int:
    """Distinct weight copies rotated across steps: enough that the active experts of all copies
    together exceed 4x L2 at the smallest T (so a step never finds the previous steps' experts in
    L2), at least 2, at most 8 and at most `max_bytes` of weights."""
    per_copy = min(mw.expected_active(cfg, T) for T in Ts) * cfg.weight_bytes_per_expert
    n = max(2, math.ceil(4 * L2_BYTES / per_copy))
    fit = int(max_bytes // (cfg.E * cfg.weight_bytes_per_expert))
    return max(2, min(n, 8, fit))


def weights_key(cfg: mw.MoEConfig):
    """Configs that differ only in their router logits (the skewed variant) share one set of weights."""
    return (cfg.H, cfg.I, cfg.E, cfg.wtype, cfg.seed)


class Layers:
    """Several distinct copies of one layer's expert weights (so that consecutive steps do not re-read
    the previous steps' experts from L2). The weights live in HBM, or with host_weights in pinned host
    memory (Grace LPDDR5X on a GB300 node), which the same kernels read over NVLink-C2C."""

    def __init__(self, cfg: mw.MoEConfig, copies: int, device, seed: int = 0, host_weights: bool = False):
        self.cfg, self.key, self.copies = cfg, weights_key(cfg), copies
        self.layers = []
        for c in range(copies):
            layer = mw.make_layer(cfg, seed=seed + 1000 * c, device=device)
            if host_weights:
                layer = {n: (torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) if v is not None
                             else None) for n, v in layer.items()}
                torch.cuda.synchronize()
            self.layers.append(layer)


class Workload:
    """One decode batch of T tokens per weight copy. The number of active experts per batch (which
    sets the weight bytes a step must stream) is read from the library's own routing kernel."""

    def __init__(self, cfg: mw.MoEConfig, T: int, layers: Layers, device, moe, seed: int = 0):
        self.cfg, self.T, self.device = cfg, T, device
        self.layers = layers.layers
        self.tokens = [mw.make_tokens(cfg, T, seed=seed + 1000 * c, device=device) for c in range(layers.copies)]
        self.active = []
        k = cfg.top_k
        for x, lg in self.tokens:
            i32 = dict(dtype=torch.int32, device=device)
            outs = [torch.empty(T, k, **i32), torch.empty(T, k, device=device), torch.empty(cfg.E, **i32),
                    torch.empty(cfg.E + 1, **i32), torch.empty(T * k, **i32), torch.empty(T, k, **i32),
                    torch.empty(cfg.E, **i32), torch.empty(1, **i32)]
            moe.moe_route_topk(lg, k, *outs)
            self.active.append(int(outs[-1].item()))
        self.wt = 0 if cfg.wtype == "bf16" else 1  # the residual split uses the INT8 workspace

    @property
    def copies(self) -> int:
        return len(self.layers)

    def weight_bytes(self, c: int) -> int:
        return self.active[c] * self.cfg.weight_bytes_per_expert

    def mean_weight_bytes(self) -> float:
        return sum(self.weight_bytes(c) for c in range(self.copies)) / self.copies

    def step_other_bytes(self) -> int:
        """Bytes of a whole step besides the weights: x and logits read, routing tables, the
        gathered block, h and Y written and read once, out written."""
        cfg, T = self.cfg, self.T
        P = T * cfg.top_k
        routing = 4 * (3 * P + 2 * cfg.E + 2)  # ids, w, sorted_token / inv_pos, counts, offsets, active
        return T * cfg.H * 2 + T * cfg.E * 4 + routing + 2 * P * cfg.H * 2 + 2 * P * cfg.I * 2 + 2 * P * cfg.H * 4 \
            + T * cfg.H * 2

    def act_bytes(self) -> int:
        """Token-side algorithmic bytes of the expert kernels: xg read, h write + read, Y write."""
        cfg, P = self.cfg, self.T * self.cfg.top_k
        return P * cfg.H * 2 + 2 * P * cfg.I * 2 + P * cfg.H * 4


def decode_step_roofline(moe, wl: Workload, ws, stream, n: int, peak: float):
    """The one-launch decode step is the whole step: its kernel timed per launch with events on the
    launching stream (an event pair around every call). Algorithmic bytes = every array of the step,
    each once. Returns (achieved GB/s, frac of peak, average ms per launch, algorithmic bytes)."""
    cfg, T = wl.cfg, wl.T
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=wl.device)
    evs, nbytes = [], []
    for i in range(n + 3):
        c = i % wl.copies
        x, lg = wl.tokens[c]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ffn_forward(moe, cfg, wl.layers[c], x, lg, out, ws, stream)
        b.record(stream)
        if i >= 3:
            evs.append((a, b))
            nbytes.append(wl.weight_bytes(c) + wl.step_other_bytes())
    torch.cuda.synchronize()
    if moe.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    t = [a.elapsed_time(b) for a, b in evs]
    avg_ms = sum(t) / len(t)
    alg = sum(nbytes) / len(nbytes)
    achieved = alg / (avg_ms * 1e-3) / 1e9
    return achieved, achieved / peak, avg_ms, alg


def roofline_for(moe, wl: Workload, ws, stream, n: int, peak: float):
    """(kernel description, achieved, frac, avg ms, algorithmic bytes) of the step's dominant kernel(s)."""
    if kernels_per_step(wl.cfg, wl.T, moe) == 1:
        return ("decode_step_kernel: the whole step in one launch (routing, gate+up with SiLU*up, down, "
                "combine), timed per launch",) + decode_step_roofline(moe, wl, ws, stream, n, peak)
    return ("expert FFN stream kernels (gate+up with SiLU*up, then down), timed together",) + \
        expert_call_roofline(moe, wl, ws, stream, n, peak)


def expert_call_roofline(moe, wl: Workload, ws, stream, n: int, peak: float):
    """The expert-FFN call (moe_expert_ffn: the expert kernels, which stream the weights) timed alone
    with events on the launching stream; routing and gather run outside the events. Returns
    (achieved GB/s of algorithmic bytes, frac of peak, average ms per call, algorithmic bytes)."""
    cfg, T, dev = wl.cfg, wl.T, wl.device
    r = {nm: torch.empty(sz, dtype=dt, device=dev) for nm, sz, dt in (
        ("ids", (T, cfg.top_k), torch.int32), ("w", (T, cfg.top_k), torch.float32), ("counts", (cfg.E,), torch.int32),
        ("offsets", (cfg.E + 1,), torch.int32), ("st", (T * cfg.top_k,), torch.int32),
        ("inv", (T, cfg.top_k), torch.int32), ("act", (cfg.E,), torch.int32), ("na", (1,), torch.int32))}
    xg = torch.empty(T * cfg.top_k, cfg.H, dtype=torch.bfloat16, device=dev)
    Y = torch.empty(T * cfg.top_k, cfg.H, dtype=torch.float32, device=dev)
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
    evs, nbytes = [], []
    for i in range(n + 3):
        c = i % wl.copies
        L = wl.layers[c]
        x, lg = wl.tokens[c]
        moe.moe_route_topk(lg, cfg.top_k, r["ids"], r["w"], r["counts"], r["offsets"], r["st"], r["inv"], r["act"],
                           r["na"], stream)
        moe.moe_gather(x, cfg.top_k, r["st"], xg, stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        expert_ffn(moe, cfg, L, xg, r, Y, ws, stream)
        b.record(stream)
        moe.moe_combine(Y, r["inv"], r["w"], cfg.top_k, out, stream)
        if i >= 3:
            evs.append((a, b))
            nbytes.append(wl.weight_bytes(c) + wl.act_bytes())
    torch.cuda.synchronize()
    if moe.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    t = [a.elapsed_time(b) for a, b in evs]
    avg_ms = sum(t) / len(t)
    alg = sum(nbytes) / len(nbytes)
    achieved = alg / (avg_ms * 1e-3) / 1e9
    return achieved, achieved / peak, avg_ms, alg


# ------------------------------------------------------------------ our implementation
def bench_ours(args, cfg, T):
    import routed_expert_ffn_softmax_gb300 as moe
    from routed_expert_ffn_softmax_gb300 import build as moe_build

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if rank == 0:
        moe_build.build()
    if ws_n > 1:
        dist.barrier()
    moe.load()
    moe.moe_set_decode_step_policy(args.decode_step_policy)

    host = args.weights == "host"
    copies = args.copies if args.copies > 0 else auto_copies(cfg, [T])
    layers = Layers(cfg, copies, dev, host_weights=host)
    wl = Workload(cfg, T, layers, dev, moe)
    stream = torch.cuda.current_stream()
    ws = moe.alloc_workspace(T, cfg.H, cfg.I, cfg.E, cfg.top_k, wl.wt, dev)
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)

    def step(c):
        x, lg = wl.tokens[c]
        ffn_forward(moe, cfg, wl.layers[c], x, lg, out, ws, stream)

    def barrier_sync():
        torch.cuda.synchronize()
        if ws_n > 1:
            dist.barrier()
        torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        for i in range(args.warmup):
            step(i % copies)
        barrier_sync()
        if moe.workspace_status(ws) != 0:
            raise RuntimeError("a kernel reported a timed-out wait during warm-up")
        # two events around the whole timed region: an event between steps would end the overlap
        # of one step's last kernel with the next step's first (programmatic dependent launch)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            step(i % copies)
        ev1.record(stream)
        barrier_sync()
    clocks = clk.summary()
    total_ms = ev0.elapsed_time(ev1)
    per_step = per_step_times(lambda i: step(i % copies), max(min(args.steps, 100), 20), stream)
    if moe.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    bytes_timed = sum(wl.weight_bytes(i % copies) for i in range(args.steps))
    total_ms, value, tokens_s = aggregate_over_ranks(total_ms, bytes_timed, T * args.steps, ws_n, dev)

    # ---- dominant kernels: the expert FFN pair (gate+up, down), timed alone with events
    if host:
        peak, peak_kind = round(c2c_copy_peak(dev), 1), "measured in this run (pinned host -> device copy, NVLink-C2C)"
    else:
        peak, peak_kind = hbm_peak()
        peak_kind = f"{peak_kind} (hbm_gbs, copy bandwidth)"
    roof_kernel, ffn_achieved, ffn_frac, ffn_avg_ms, ffn_alg = roofline_for(moe, wl, ws, stream,
                                                                             max(min(args.steps, 200), 20), peak)
    workload_name = f"{cfg.name}_T{T}" + ("_hostweights" if host else "")
    # the one-launch decode step's capture is keyed by its own sources
    traffic = recorded_traffic(workload_name, DECODE_SOURCES if kernels_per_step(cfg, T, moe) == 1
                               else expert_sources(cfg.wtype))

    # ---- end to end through the C ABI: host inputs in, host result out, every step (the copies
    # overlap the neighbouring steps' compute, double-buffered)
    x_h = [t[0].cpu().pin_memory() for t in wl.tokens]
    lg_h = [t[1].cpu().pin_memory() for t in wl.tokens]
    out_h = [torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(wl.tokens[0][0]) for _ in range(2)]
    lg_d = [torch.empty_like(wl.tokens[0][1]) for _ in range(2)]
    out_d = [out, torch.empty_like(out)]

    def e2e_in(i, b):
        x_d[b].copy_(x_h[i % copies], non_blocking=True)
        lg_d[b].copy_(lg_h[i % copies], non_blocking=True)

    def e2e_step(i, b):
        ffn_forward(moe, cfg, wl.layers[i % copies], x_d[b], lg_d[b], out_d[b], ws, stream)

    def e2e_out(i, b):
        out_h[b].copy_(out_d[b], non_blocking=True)

    run_pipelined(3, e2e_in, e2e_step, e2e_out, stream, dev)
    barrier_sync()
    a, b = run_pipelined(args.steps, e2e_in, e2e_step, e2e_out, stream, dev)
    barrier_sync()
    e2e_ms, e2e_value, _ = aggregate_over_ranks(a.elapsed_time(b), bytes_timed, T * args.steps, ws_n, dev)

    result = {
        "metric": METRIC_HOST if host else METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "ms_per_step_median": round(statistics.median(per_step), 5),
        "ms_per_step_geomean": round(statistics.geometric_mean(per_step), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE[cfg.wtype],
        "data": "synthetic (seeded N(0,1) tokens and logits, N(0,0.02) weights)",
        "pct_of_peak": round(100.0 * value / ws_n / peak, 2),
        "tokens_per_s": round(tokens_s, 1),
        # the routed work only: 2 flops per weight per token routed to its expert
        "tflops": round(2 * 3 * cfg.H * cfg.I * T * cfg.top_k / (total_ms / args.steps * 1e-3) / 1e12, 3),
        "config": {
            "workload": workload_name, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.top_k,
            "weights": cfg.wtype, "T": T, "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU",
            "weights_memory": "pinned host memory (Grace LPDDR5X), read by the kernels over NVLink-C2C" if host
                              else "HBM",
            "active_experts_mean": round(sum(wl.active) / len(wl.active), 2),
            "tokens_per_expert_mean": round(T * cfg.top_k * len(wl.active) / sum(wl.active), 2),
            "weight_bytes_per_step_mean": int(wl.mean_weight_bytes()),
            # every array of the step (weights, x, logits, routing tables, xg, h, Y, out), each once
            "algorithmic_bytes_per_step_mean": int(wl.mean_weight_bytes() + wl.step_other_bytes()),
            "l2": f"inputs larger than L2: each step streams >= "
                  f"{min(wl.weight_bytes(c) for c in range(copies)) / 1e6:.0f} MB of expert weights, "
                  f"rotating over {copies} distinct weight copies",
        },
        "roofline": {
            "kernel": roof_kernel,
            "bound": "c2c" if host else "hbm",
            "achieved": round(ffn_achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(ffn_frac, 4),
            "traffic": traffic,
            "avg_launch_ms": round(ffn_avg_ms, 5),
            "algorithmic_bytes_per_launch": int(ffn_alg),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": T * cfg.H * 2 + T * cfg.E * 4, "d2h_bytes_per_step": T * cfg.H * 2},
        "gpu_launches": kernels_per_step(cfg, T, moe) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, T, wl, budget_s=args.cpu_budget)
    held = [layers]  # the sweep reuses these weights for its points of the same config, then frees them
    del x_h, lg_h, out_h, x_d, lg_d, out_d, ws, wl, layers
    if rank == 0 and not args.no_sweep and not host:
        result["sweep"] = sweep(moe, dev, peak, held, args.sweep_configs.split(","))
    held.clear()
    if ws_n > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result if rank == 0 else None


DTYPE = {"bf16": "bf16", "int8": "int8 weights, bf16 activations",
         "int8_residual": "int8 + int8 residual gate/up, int8 down, bf16 activations"}


def measure_point(moe, cfg, T, layers: Layers, dev, peak, steps=60, warmup=5, n_roof=40):
    """GB/s and tokens/s of whole steps at one (config, T) point (two events around `steps` steps),
    and the expert call's roofline fraction."""
    wl = Workload(cfg, T, layers, dev, moe)
    ws = moe.alloc_workspace(T, cfg.H, cfg.I, cfg.E, cfg.top_k, wl.wt, dev)
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream()

    def step(c):
        x, lg = wl.tokens[c]
        ffn_forward(moe, cfg, wl.layers[c], x, lg, out, ws, s)
    for i in range(warmup):
        step(i % wl.copies)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for i in range(steps):
        step(i % wl.copies)
    b.record(s)
    torch.cuda.synchronize()
    if moe.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    ms = a.elapsed_time(b) / steps
    wb = sum(wl.weight_bytes(i % wl.copies) for i in range(steps)) / steps
    gbs = wb / (ms * 1e-3) / 1e9
    kernel, ach, frac, avg_ms, _ = roofline_for(moe, wl, ws, s, n_roof, peak)
    flops = 2 * 3 * cfg.H * cfg.I * T * cfg.top_k  # routed work: 2 flops per weight per token routed to it
    row = {"workload": f"{cfg.name}_T{T}", "weights": cfg.wtype, "T": T,
           "active_experts": round(sum(wl.active) / len(wl.active), 2),
           "tokens_per_expert": round(T * cfg.top_k * len(wl.active) / sum(wl.active), 2),
           "us_per_step": round(ms * 1e3, 2), "GB_s": round(gbs, 1), "pct_of_peak": round(100 * gbs / peak, 2),
           "tokens_per_s": round(T / (ms * 1e-3), 1), "launches_per_step": kernels_per_step(cfg, T, moe),
           "roofline": {"kernel": kernel, "achieved": round(ach, 1),
                        "frac": round(frac, 4), "avg_launch_us": round(avg_ms * 1e3, 2)},
           "copies": wl.copies,
           "tflops": round(flops / (ms * 1e-3) / 1e12, 2)}
    if cfg.wtype == "bf16" and T * cfg.top_k >= 32 * cfg.E:  # a real contraction: the tensor-core roofline
        tp, kind = tensor_peak()
        call = flops / (avg_ms * 1e-3) / 1e12
        row["tensor_roofline"] = {"kernel": "expert FFN (gate+up, down), timed together", "achieved": round(call, 1),
                                  "peak": tp, "peak_kind": kind, "unit": "TFLOP/s", "frac": round(call / tp, 4)}
    del wl, ws
    return row


def sweep(moe, dev, peak, held, names):
    """Every (config, T) point of the named workloads, measured the same way as the headline with
    fewer steps (weights rotate over distinct copies at every point). `held` may hold the headline's
    Layers; configs sharing its weights go first and reuse them."""
    have = held.pop() if held else None
    if have is not None:
        names = sorted(names, key=lambda n: weights_key(mw.CONFIGS[n]) != have.key)
    rows = []
    with ClockSampler(dev.index or 0) as clk:
        for name in names:
            cfg = mw.CONFIGS[name]
            if have is None or have.key != weights_key(cfg):
                have = None
                torch.cuda.empty_cache()
                have = Layers(cfg, auto_copies(cfg, cfg.T), dev)
            for T in cfg.T:
                rows.append(measure_point(moe, cfg, T, have, dev, peak))
                torch.cuda.empty_cache()
    have = None
    torch.cuda.empty_cache()
    return {"points": rows, "peak_gbs": peak, "clocks": clk.summary(),
            "method": "per point: 5 warm-up steps, 60 timed steps between two events (GB/s = active-expert "
                      "weight bytes / time), then the dominant kernel(s) for 40 calls with an event pair around "
                      "each: the expert call (moe_expert_ffn) for the staged path, the whole step for the "
                      "one-launch decode step (roofline frac = algorithmic bytes / time / peak); weights rotate "
                      "over distinct copies"}


# ------------------------------------------------------------------ CPU oracle (baseline leg)
def oracle_rate(cfg, T, budget_s, experts, x, lg):
    """Run the oracle token by token over the batch's first tokens (cycling) until the time budget is
    spent, at least one token. `experts` maps an expert id to its CPU weights (W_gate, W_up, W_down,
    s_*). Returns (weight GB/s for the whole batch, tokens/s, tokens run, seconds)."""
    import oracle
    ro = oracle.route(lg, cfg.top_k)
    full_bytes = ro["num_active"] * cfg.weight_bytes_per_expert
    sample = sample_tokens(ro, T, cfg.top_k, len(experts))
    t0 = time.perf_counter()
    n = 0
    while True:
        t = sample[n % len(sample)]
        ys = []
        for j in range(cfg.top_k):
            W = experts[int(ro["ids"][t, j])]
            if cfg.wtype == "int8_residual":
                h, _, _ = oracle.gateup_token_residual(x[t], W["W_gate"], W["s_gate"], W["Wr_gate"], W["sr_gate"],
                                                       W["W_up"], W["s_up"], W["Wr_up"], W["sr_up"])
                ys.append(oracle.down_token(h, W["W_down"], W["s_down"], "int8"))
            else:
                h, _, _ = oracle.gateup_token(x[t], W["W_gate"], W["W_up"], W["s_gate"], W["s_up"], cfg.wtype)
                ys.append(oracle.down_token(h, W["W_down"], W["s_down"], cfg.wtype))
        oracle.combine_token(np.stack(ys), ro["w"][t])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    per_token = dt / n
    # the oracle's cost is linear in tokens: the whole batch takes T * per_token
    return full_bytes / (T * per_token) / 1e9, 1.0 / per_token, n, dt


def sample_tokens(ro, T, k, max_experts):
    """The batch's first tokens whose experts together number at most max_experts (at least one)."""
    seen, out = set(), []
    for t in range(T):
        e = set(int(v) for v in ro["ids"][t])
        if out and len(seen | e) > max_experts:
            break
        seen |= e
        out.append(t)
    return out


def sample_experts(cfg, ro, T, max_experts, fetch):
    """CPU weights of the experts of sample_tokens(...): fetch(e) returns one expert's tensors."""
    need = sorted({int(v) for t in sample_tokens(ro, T, cfg.top_k, max_experts) for v in ro["ids"][t]})
    return {e: fetch(e) for e in need}


def cores_used():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    omp = os.environ.get("OMP_NUM_THREADS")
    return int(omp) if omp and omp.isdigit() else n


CPU_SAMPLE_EXPERTS = 32


def cpu_baseline(cfg, T, wl, budget_s):
    import oracle
    x, lg = (t.cpu() for t in wl.tokens[0])
    ro = oracle.route(lg, cfg.top_k)
    L = wl.layers[0]
    experts = sample_experts(cfg, ro, T, CPU_SAMPLE_EXPERTS,
                             lambda e: {n: (v[e].cpu() if v is not None else None) for n, v in L.items()})
    gbs, tok_s, n, dt = oracle_rate(cfg, T, budget_s, experts, x, lg)
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "tokens_per_s": round(tok_s, 3),
            "sample": f"{n} token evaluations cycling over the batch's first tokens whose experts number at most "
                      f"{CPU_SAMPLE_EXPERTS} ({dt:.1f} s of CPU time); the oracle's time is linear in tokens and the "
                      f"same for every token, so GB/s = active-expert weight bytes of the {T}-token batch / "
                      f"({T} x time per token)"}


def cpu_expert(cfg, e, seed=0):
    """One expert's weights drawn on the CPU (the same draws make_layer makes for it)."""
    L = mw.make_layer(cfg, seed=seed, device="cpu", experts=[e])
    return {n: (v[0] if v is not None else None) for n, v in L.items()}


def bench_reference(args, cfg, T):
    """The CPU oracle on the host cores, same metric and config (rank 0 only)."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    x, lg = mw.make_tokens(cfg, T, device="cpu")
    ro = oracle.route(lg, cfg.top_k)
    experts = sample_experts(cfg, ro, T, CPU_SAMPLE_EXPERTS, lambda e: cpu_expert(cfg, e))
    nsteps = args.steps + args.warmup
    per_step_budget = max(0.02, args.cpu_budget * 4 / nsteps)
    vals, times = [], []
    for i in range(nsteps):
        gbs, tok_s, n, dt = oracle_rate(cfg, T, per_step_budget, experts, x, lg)
        if i >= args.warmup:
            vals.append(gbs)
            times.append(T / tok_s)
    value = statistics.mean(vals)
    ms_step = 1e3 * statistics.mean(times)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 accumulate, bf16 inputs (CPU oracle)",
        "data": "synthetic (seeded N(0,1) tokens and logits, N(0,0.02) weights)",
        "tokens_per_s": round(T / (ms_step * 1e-3), 3),
        "config": {"workload": f"{cfg.name}_T{T}", "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.top_k,
                   "weights": cfg.wtype, "T": T, "active_experts": ro["num_active"]},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
                         "sample": f"each step runs the oracle token by token over the batch's first tokens whose "
                                   f"experts number at most {CPU_SAMPLE_EXPERTS} (cycling) for about "
                                   f"{per_step_budget:.2f} s (at least one token) and scales to the whole {T}-token "
                                   f"batch (time is linear in tokens and the same for every token)"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------------ decode GQA attention
class AttnWorkload:
    """One decode batch: queries, key/value caches (device-resident decode state, larger than L2 for
    the bench's workloads, so every call streams them from HBM) and the sequence lengths."""

    def __init__(self, acfg: mw.AttnConfig, device, seed: int = 0):
        self.acfg = acfg
        self.q, self.k, self.v, self.lens = mw.make_attention(acfg, seed=seed, device=device)
        self.L_cap = self.k.shape[2]
        self.kv_bytes = mw.attention_kv_bytes(self.lens, acfg.h_kv, acfg.d)
        self.io_bytes = 2 * self.q.numel() * 2  # query in, output out (bf16)


def bench_attention_ours(args, acfg):
    import routed_expert_ffn_softmax_gb300 as moe
    from routed_expert_ffn_softmax_gb300 import build as moe_build

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if rank == 0:
        moe_build.build()
    if ws_n > 1:
        dist.barrier()
    moe.load()
    wl = AttnWorkload(acfg, dev)
    stream = torch.cuda.current_stream()
    ws = moe.alloc_gqa_workspace(acfg.B, acfg.h_q, acfg.h_kv, acfg.d, wl.L_cap, dev)
    out = torch.empty(acfg.B, acfg.h_q, acfg.d, dtype=torch.bfloat16, device=dev)

    def step():
        moe.moe_gqa_decode(wl.q, wl.k, wl.v, wl.lens, acfg.scale, out, ws, stream)

    def barrier_sync():
        torch.cuda.synchronize()
        if ws_n > 1:
            dist.barrier()
        torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step()
        barrier_sync()
        if moe.workspace_status(ws) != 0:
            raise RuntimeError("the attention kernel reported a nonzero status during warm-up")
        # two events around the whole timed region (see bench_ours)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier_sync()
    clocks = clk.summary()
    total_ms = ev0.elapsed_time(ev1)
    per_step = per_step_times(lambda i: step(), min(args.steps, 100), stream)
    if moe.workspace_status(ws) != 0:
        raise RuntimeError("the attention kernel reported a nonzero status")
    total_ms, value, seq_s = aggregate_over_ranks(total_ms, wl.kv_bytes * args.steps, acfg.B * args.steps, ws_n, dev)
    # the one kernel of a step is the roofline's kernel: its average launch is the timed region / steps
    avg_ms = total_ms / args.steps
    achieved = (wl.kv_bytes + wl.io_bytes) / (avg_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    workload_name = acfg.name

    # ---- end to end through the C ABI: query and lengths in from pinned host memory, output back
    # (the copies overlap the neighbouring calls' compute, double-buffered)
    q_h = wl.q.cpu().pin_memory()
    lens_h = wl.lens.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(wl.q) for _ in range(2)]
    lens_d = [torch.empty_like(wl.lens) for _ in range(2)]
    out_d = [out, torch.empty_like(out)]

    def e2e_in(i, b):
        q_d[b].copy_(q_h, non_blocking=True)
        lens_d[b].copy_(lens_h, non_blocking=True)

    def e2e_step(i, b):
        moe.moe_gqa_decode(q_d[b], wl.k, wl.v, lens_d[b], acfg.scale, out_d[b], ws, stream)

    def e2e_out(i, b):
        out_h[b].copy_(out_d[b], non_blocking=True)

    run_pipelined(3, e2e_in, e2e_step, e2e_out, stream, dev)
    barrier_sync()
    a, b = run_pipelined(args.steps, e2e_in, e2e_step, e2e_out, stream, dev)
    barrier_sync()
    _, e2e_value, _ = aggregate_over_ranks(a.elapsed_time(b), wl.kv_bytes * args.steps, acfg.B * args.steps, ws_n,
                                           dev)
    lens = wl.lens.cpu()
    result = {
        "metric": METRIC_ATTN,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "ms_per_step_median": round(statistics.median(per_step), 5),
        "ms_per_step_geomean": round(statistics.geometric_mean(per_step), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (fp32 scores, softmax and accumulation)",
        "data": "synthetic (seeded N(0,1) queries, keys and values; lengths uniform in the stated range)",
        "pct_of_peak": round(100.0 * value / ws_n / peak, 2),
        "sequences_per_s": round(seq_s, 1),
        "config": {
            "workload": workload_name, "h_q": acfg.h_q, "h_kv": acfg.h_kv, "group": acfg.group, "d": acfg.d,
            "B": acfg.B, "seq_len_range": [acfg.len_lo, acfg.len_hi], "L_cap": wl.L_cap,
            "seq_len_mean": round(float(lens.float().mean()), 1),
            "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU",
            "kv_bytes_per_step": wl.kv_bytes,
            "l2": f"inputs larger than L2: each step reads {wl.kv_bytes / 1e6:.0f} MB of keys and values",
        },
        "roofline": {
            "kernel": "gqa_decode_kernel (the step's only kernel)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (hbm_gbs, copy bandwidth)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(workload_name, ATTN_SOURCES),
            "avg_launch_ms": round(avg_ms, 5),
            "algorithmic_bytes_per_launch": wl.kv_bytes + wl.io_bytes,
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": wl.q.numel() * 2 + acfg.B * 4, "d2h_bytes_per_step": out.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = attention_cpu_baseline(acfg, wl, budget_s=args.cpu_budget)
    if ws_n > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result if rank == 0 else None


def attention_oracle_rate(acfg, q, k, v, lens, budget_s):
    """The oracle over the batch's sequences one at a time (cycling) until the budget is spent, at
    least one; returns (key/value GB/s, sequences/s, sequences run, seconds)."""
    import oracle
    t0 = time.perf_counter()
    n = done_bytes = 0
    while True:
        b = n % q.shape[0]
        ln = int(lens[b])
        oracle.gqa_decode(q[b:b + 1], k[b:b + 1, :, :ln], v[b:b + 1, :, :ln], lens[b:b + 1], acfg.scale)
        done_bytes += ln * acfg.h_kv * acfg.d * 4
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done_bytes / dt / 1e9, n / dt, n, dt


def attention_cpu_baseline(acfg, wl, budget_s):
    q, lens = wl.q.cpu(), wl.lens.cpu()
    nseq = min(acfg.B, 8)
    k, v = wl.k[:nseq].cpu(), wl.v[:nseq].cpu()
    gbs, seq_s, n, dt = attention_oracle_rate(acfg, q[:nseq], k, v, lens[:nseq], budget_s)
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "sequences_per_s": round(seq_s, 3),
            "sample": f"{n} sequence evaluations cycling over the first {nseq} sequences of the batch "
                      f"({dt:.1f} s); GB/s = key/value bytes those sequences read / time"}


def bench_attention_reference(args, acfg):
    """The CPU oracle on the host cores, same metric and config (rank 0 only)."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    nseq = min(acfg.B, 8)
    lens_all = mw.draw_seq_lens(acfg.B, acfg.len_lo, acfg.len_hi, acfg.seed)
    q, k, v, lens = mw.make_attention(acfg, seq_lens=lens_all[:nseq])
    nsteps = args.steps + args.warmup
    per_step_budget = max(0.02, args.cpu_budget * 4 / nsteps)
    vals, times = [], []
    kv_full = mw.attention_kv_bytes(lens_all, acfg.h_kv, acfg.d)
    for i in range(nsteps):
        gbs, seq_s, n, dt = attention_oracle_rate(acfg, q, k, v, lens, per_step_budget)
        if i >= args.warmup:
            vals.append(gbs)
            times.append(kv_full / (gbs * 1e9))
    value = statistics.mean(vals)
    ms_step = 1e3 * statistics.mean(times)
    return {
        "impl": "reference",
        "metric": METRIC_ATTN,
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (CPU oracle), bf16 inputs",
        "data": "synthetic (seeded N(0,1) queries, keys and values; lengths uniform in the stated range)",
        "sequences_per_s": round(acfg.B / (ms_step * 1e-3), 3),
        "config": {"workload": acfg.name, "h_q": acfg.h_q, "h_kv": acfg.h_kv, "group": acfg.group, "d": acfg.d,
                   "B": acfg.B, "seq_len_range": [acfg.len_lo, acfg.len_hi]},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
                         "sample": f"each step runs the oracle over the first {nseq} sequences of the batch (cycling) "
                                   f"for about {per_step_budget:.2f} s and scales to the whole batch's key/value bytes"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="dsv3", choices=sorted(mw.CONFIGS))
    ap.add_argument("--T", type=int, default=512)
    ap.add_argument("--copies", type=int, default=0,
                    help="distinct weight copies rotated across steps (0: enough to exceed 4x L2, at least 2)")
    ap.add_argument("--weights", choices=("device", "host"), default="device",
                    help="where the expert weights live: HBM, or pinned host memory read over NVLink-C2C")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sweep over every (config, T) point of the expert workloads")
    ap.add_argument("--sweep-configs", default=",".join(SWEEP_CONFIGS),
                    help="comma-separated workloads the sweep covers (every T of each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--decode-step-policy", type=int, choices=(0, 1, 2), default=0,
                    help="moe_ffn_forward's path: 0 by batch shape (default), 1 never the one-launch decode step, "
                         "2 the one-launch decode step whenever the sizes allow")
    ap.add_argument("--op", choices=("ffn", "attention"), default="ffn",
                    help="ffn: the routed-expert FFN (default); attention: decode GQA attention")
    ap.add_argument("--attn-config", default="qwen3_30b_attn",
                    choices=sorted(n for n in mw.ATTN_CONFIGS if n != "attn_tiny"))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op == "attention":
        acfg = mw.ATTN_CONFIGS[args.attn_config]
        res = bench_attention_reference(args, acfg) if args.impl == "reference" else bench_attention_ours(args, acfg)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    cfg = mw.CONFIGS[args.config]
    if args.impl == "reference":
        res = bench_reference(args, cfg, args.T)
    else:
        res = bench_ours(args, cfg, args.T)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
