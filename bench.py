#!/usr/bin/env python3
"""Benchmark of the MoE layer forward (router -> dispatch -> grouped SwiGLU FFN + shared
expert -> combine) on GB300, through the C ABI.

Default workload: the DeepSeek-V3-shaped decode step, T = 128 tokens (64 requests x query
length 2), H = 7168, E = 256 routed experts, top-8, I = 2048, one shared expert I = 2048,
bf16 weights (22.5 GB of routed experts) and activations, fp32 output.  Inputs are seeded
synthetic tensors already resident in HBM; the activated experts' weights (13.2 GB per
step at T=128) are far larger than L2, so every step streams them from HBM.

One JSON line on rank 0.  Beside the decode headline, the same line carries a `workloads`
table measured in the same process on the same weights: the batch sweep T = 2 ... 256
(memory-bound: target >= 70% of 8 TB/s up to 64 tokens), the skewed 8192-token batch and
the 16384-token prefill (tensor-bound: target >= 60% of the bf16 burst rate).  Each row is
timed like the headline (bare calls between CUDA events) and gets its per-stage times from
a separate instrumented pass.  `--impl reference` times the fp64 CPU oracle instead (the
reference arm), on a bounded sample of the same workload.
Multi-GPU (torchrun): independent replicas, one per GPU, each with its own tokens; no
collective on the data path (the timing is reduced with a max over ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300 (DeepSeek-V3 shape)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# stage events: before the router, after the router, after dispatch, after the FFN launch
# (its up and down projections are one launch: the next mark is the same point, and
# "ffn_down" reads ~0), after the FFN, after combine
STAGES = ("router", "dispatch", "ffn_up", "ffn_down", "combine")
# routing options of other MoE families (moe_routing_t); "default" is the plain router
ROUTINGS = {
    "default": None,
    "groups_top2": dict(scoring="sigmoid", n_group=8, topk_group=4, group_top=2),
    "softmax_groups_max": dict(scoring="softmax", n_group=8, topk_group=3, group_top=1,
                               renorm=False),
    "softmax": dict(scoring="softmax"),
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    @staticmethod
    def _stats(win):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        pw = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons,
                "samples": len(win)}

    def summary(self, t0: float, t1: float, b0: float | None = None, b1: float | None = None):
        """Clocks over the timed region [t0, t1] and, when given, over the busy window
        [b0, b1] around it (warm-up, timed and instrumented passes of the same workload):
        a timed region of a few tens of milliseconds holds one or two 20 ms samples."""
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        timed = [p for (t, p) in self.samples if t0 <= t <= t1]
        out = self._stats(timed) if timed else {"samples": 0}
        if b0 is not None:
            busy = [p for (t, p) in self.samples if b0 <= t <= b1]
            if busy:
                wb = self._stats(busy)
                out = {**wb, "timed_region": out, "window": "busy window of this workload "
                       f"({b1 - b0:.2f} s: warm-up, timed and instrumented passes)"}
        return out


# ------------------------------------------------------------------------ accounting
TRAFFIC_MAX_TOKENS = 256


def ffn_traffic(w, fp8: bool, alg_bytes: int, path: str | None = None):
    """DRAM bytes per step of the FFN launches (bf16 weights: the routed launch; FP8: the up
    and the down launch) for batches of up to TRAFFIC_MAX_TOKENS tokens, where every
    activated expert is one token tile that streams its weights once: the step's
    algorithmic bytes times the DRAM / algorithmic ratio ncu measured on small cases of the
    same regime (profiles/ffn_traffic.json, taken on the current FFN sources).  None for
    larger batches (their token tiles' L2 reuse depends on the routing, so the small cases
    do not scale to them), or when the FFN sources changed since the record was taken."""
    if w.T > TRAFFIC_MAX_TOKENS:
        return None
    path = path or os.path.join(ROOT, "profiles", "ffn_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return int(round(rec["ratio"]["fp8" if fp8 else "bf16"] * alg_bytes))
    except (OSError, KeyError, ValueError, TypeError):
        return None


def workload_desc(w) -> str:
    """The config's workload string, the same on both arms."""
    dsv3 = (w.H, w.E, w.K, w.I, w.Is) == (7168, 256, 8, 2048, 2048)
    return (f"{w.name}: {'DeepSeek-V3-shaped ' if dsv3 else ''}MoE layer forward, T={w.T} "
            f"tokens, H={w.H}, E={w.E}, top-{w.K}, I={w.I}, shared I={w.Is}")


def shared_on_side(w, fp8: bool = False) -> bool:
    """moe_layer_forward runs the shared expert as its own launch on a side stream (bf16
    weights, up to 128 tokens); otherwise it is a second problem of the routed FFN launch."""
    return bool(w.Is) and not fp8 and w.T <= 128


def algorithmic(w, n_act: int, wbytes: int = 2, side: bool = False):
    """Per-launch algorithmic bytes and FLOPs of each stage (what the method must move or
    compute: the weights of the activated experts, the activations in and out).  wbytes:
    bytes per expert weight (2 bf16, 1 FP8; the FP8 tile scales add 1 byte per 16384).
    side: the shared expert is its own launch ("ffn_shared"), not part of "ffn"."""
    T, H, E, K, I, Is = w.T, w.H, w.E, w.K, w.I, w.Is
    TK = T * K
    # weights, token rows in and fp32 outputs of the shared expert
    sh_bytes = 3 * H * Is * wbytes + T * H * 2 + T * H * 4 if Is else 0
    sh_flops = 2 * T * 3 * H * Is
    b = {
        "router": E * H * 2 + T * H * 2 + T * K * 8,
        "dispatch": T * H * 2 + TK * H * 2 + T * K * 4 * 3,
        # weights of the activated experts (+ shared), token rows in, outputs out; the
        # intermediate h stays on chip or in L2 between the two projections and is not
        # counted
        "ffn": n_act * 3 * H * I * wbytes + TK * H * 2 + TK * H * 2 + (0 if side else sh_bytes),
        "combine": TK * H * 2 + (T * H * 4 if Is else 0) + T * H * 4 + T * K * 8,
    }
    f = {
        "router": 2 * T * E * H,
        "dispatch": 0,
        "ffn": 2 * TK * 3 * H * I + (0 if side else sh_flops),
        "combine": 2 * TK * H,
    }
    if side:
        b["ffn_shared"], f["ffn_shared"] = sh_bytes, sh_flops
    layer_bytes = ((n_act + (1 if Is else 0)) * 3 * H * I * wbytes + E * H * 2 + T * H * 2
                   + T * H * 4)
    layer_flops = 2 * T * (K * 3 * H * I + 3 * H * Is) + 2 * T * E * H
    return b, f, layer_bytes, layer_flops


def launches_per_step(w, with_affinity: bool, fp8: bool = False) -> int:
    """Kernels moe_layer_forward launches: router (GEMM + finalise for 16 <= T <= 2048
    and T > 4096, else one fused launch), dispatch (for T <= 256 one launch whose CTAs each form the bookkeeping and
    then compute the affinity matrix, gather the rows and zero the FFN's counters; else
    masks, scan, scatter and one launch for the affinity, the gather and the zeroing), the
    FFN (up and down projections in one persistent launch), combine.  On
    bf16 weights up to 128 tokens the shared expert is a second FFN launch, on a side
    stream beside the router and the dispatch.  FP8 experts quantise the permuted rows (and
    the token rows for the shared expert), split the FFN into its up and down launches and
    quantise h (and the shared expert's h) between them."""
    T = w.T
    router = 2 if (16 <= T <= 2048 or T > 4096) else 1
    dispatch = 1 if T <= 256 else 4
    ffn = 1 if not fp8 else 2 + (4 if w.Is else 2)
    side = 1 if shared_on_side(w, fp8) else 0
    return router + dispatch + ffn + side + 1


# ------------------------------------------------------------------- replica helpers
def replica_workload(name: str, rank: int):
    """The workload a replica runs: rank 0 runs the canonical batch, rank r > 0 the same
    shapes and weights with its own tokens (X seed shifted by 7919 r)."""
    from expert_routed_ffn_router_gb300 import synth
    w = synth.workload(name)
    return w if rank == 0 else synth.workload(name, x_seed=w.x_seed + 7919 * rank)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank timing over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- our arm
# Workloads measured beside the headline in the same process (same expert weights): the
# batch sweep of the memory-bound regime and the two tensor-bound batches.
SIDE_WORKLOADS = ("sweep2", "sweep4", "sweep8", "sweep16", "sweep32", "sweep64", "sweep256",
                  "skewed", "prefill")
HBM_TARGET = 0.70      # of 8 TB/s, batches of up to 64 tokens
# dense FP8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s nominal): FP8 contractions are measured
# against the measured bf16 peak times this ratio
FP8_OVER_BF16 = 2.0
TENSOR_TARGET = 0.60   # of the bf16 burst rate, batches of 8192 tokens and more


def _layer_for(w, routing, weights, dev, opts, fp8, weights8=None):
    import numpy as np
    import torch

    from expert_routed_ffn_router_gb300 import binding as B
    wts = dict(weights)
    wts["W_gate"] = torch.from_numpy(routing["W_gate"].view(np.int16)).view(torch.bfloat16).to(dev)
    wts["bias"] = torch.from_numpy(routing["bias"]).to(dev)
    X_host = torch.from_numpy(routing["X"].view(np.int16)).view(torch.bfloat16)
    if weights8 is not None:
        # pre-quantised experts: this workload's gate rows and bias (the router is bf16)
        weights8 = {**weights8, "W_gate": wts["W_gate"], "bias": wts["bias"]}
    layer = B.MoELayer(wts, w.T, w.K, with_affinity=True, routing=opts, fp8=fp8,
                       weights8=weights8)
    return layer, wts, X_host, X_host.to(dev)


def _timed(layer, X, K, stream, barrier):
    """Device time per step of K bare layer calls (CUDA events on the launching stream)."""
    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev0.record(stream)
    for _ in range(K):
        layer.forward(X)
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    return ev0.elapsed_time(ev1) / K, t0, t1


def _stage_pass(layer, X, K, stream):
    """Per-stage device times: a separate pass of K calls that record the library's stage
    events (the headline's timed region runs the bare call)."""
    import torch

    from expert_routed_ffn_router_gb300 import binding as B
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for evs in stage_ev:
        for ev in evs:
            ev.record(stream)          # materialise the handles
    torch.cuda.synchronize()
    for k in range(K):
        B.moe_debug_set_stage_events(stage_ev[k])
        layer.forward(X)
    torch.cuda.synchronize()
    B.moe_debug_set_stage_events(None)
    stage_ms = {name: statistics.fmean(stage_ev[k][i].elapsed_time(stage_ev[k][i + 1])
                                       for k in range(K))
                for i, name in enumerate(STAGES)}
    stage_ms["ffn"] = stage_ms["ffn_up"] + stage_ms["ffn_down"]
    return stage_ms


def dominant_roofline(w, n_act, stage_ms, peaks, peak_src, fp8):
    b, f, _, _ = algorithmic(w, n_act, 1 if fp8 else 2, shared_on_side(w, fp8))
    dom = max(("ffn", "router", "combine", "dispatch"), key=lambda s: stage_ms[s])
    t_dom = stage_ms[dom] / 1e3
    tpeak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if fp8 else 1.0)   # the FFN's own dtype
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor = f[dom] / max(b[dom], 1) > ridge and dom.startswith("ffn")
    if tensor:
        ach = f[dom] / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": round(tpeak, 1),
                "unit": "TFLOP/s"}
    else:
        ach = b[dom] / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = ffn_traffic(w, fp8, b[dom]) if dom == "ffn" else None
    if roof["traffic"] is not None:
        roof["traffic_source"] = ("algorithmic bytes x the DRAM / algorithmic ratio of ncu "
                                  "captures of small weight-streaming cases "
                                  "(profiles/ffn_traffic.json)")
    roof["kernel"] = dom
    roof["peak_source"] = (f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured"
                           else "fallback")
    if tensor and fp8:
        roof["peak_source"] += f": bf16 x {FP8_OVER_BF16:g}, the nominal dense FP8 / bf16 ratio"
    roof["algorithmic_bytes_per_launch"] = int(b[dom])
    roof["algorithmic_flops_per_launch"] = int(f[dom])
    roof["launch_ms"] = round(stage_ms[dom], 4)
    return roof


def layer_roofline(w, n_act, ms, peaks, fp8=False):
    """The whole layer against the measured copy bandwidth, 8 TB/s and the tensor rate of
    the expert GEMMs' dtype (bf16, or for FP8 experts bf16 x FP8_OVER_BF16; the layer's
    flops are counted alike whatever units run them)."""
    _, _, layer_bytes, layer_flops = algorithmic(w, n_act, 1 if fp8 else 2, shared_on_side(w, fp8))
    sec = ms / 1e3
    k = FP8_OVER_BF16 if fp8 else 1.0
    return {"algorithmic_bytes": int(layer_bytes), "algorithmic_flops": int(layer_flops),
            "hbm_gbs": round(layer_bytes / sec / 1e9, 1),
            "hbm_frac": round(layer_bytes / sec / 1e9 / peaks["hbm_gbs"], 4),
            "hbm_frac_of_8TBs": round(layer_bytes / sec / 8e12, 4),
            "tensor_tflops": round(layer_flops / sec / 1e12, 2),
            "tensor_frac": round(layer_flops / sec / 1e12 / (k * peaks["bf16_tflops"]), 4),
            "tensor_frac_sustained": round(layer_flops / sec / 1e12 /
                                           (k * peaks["bf16_tflops_sustained"]), 4),
            "tensor_dtype": "fp8" if fp8 else "bf16"}


def target_of(w):
    """The layer-level target of a DeepSeek-V3-shaped batch: >= 70% of 8 TB/s up to 64
    tokens, >= 60% of the bf16 burst rate from 8192 tokens; none in between."""
    if w.T <= 64:
        return "hbm_frac_of_8TBs", HBM_TARGET
    if w.T >= 8192:
        return "tensor_frac", TENSOR_TARGET
    return None, None


def measure_tiny(dev, steps: int, flush_bytes: int = 512 << 20) -> dict:
    """The tiny configuration (T=16, H=256, E=16, top-2, I=Is=128; 3.3 MB of expert
    weights): microseconds a layer call, warm (weights and activations left in L2 by the
    previous call) and cold (L2 flushed before every call by writing a buffer larger than
    it, the call alone timed with events around it)."""
    import torch

    from expert_routed_ffn_router_gb300 import binding as B
    from expert_routed_ffn_router_gb300 import synth
    w = synth.workload("tiny")
    routing = synth.routing_inputs(w)
    weights = {k: (None if v is None else torch.from_numpy(v.view("int16")).view(torch.bfloat16).to(dev))
               for k, v in synth.expert_weights_host(w).items()}
    layer, _, _, X = _layer_for(w, routing, weights, dev, None, False)
    stream = torch.cuda.current_stream()
    for _ in range(10):
        layer.forward(X)
    torch.cuda.synchronize()
    ms_warm, _, _ = _timed(layer, X, steps, stream, lambda: None)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush.fill_(1)                       # evicts the layer's data from the 129 MB L2
        e0.record(stream)
        layer.forward(X)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_cold = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    if layer.status() != 0:
        raise RuntimeError("device status word reported an error (tiny)")
    return {"T": w.T, "shape": {"H": w.H, "E": w.E, "K": w.K, "I": w.I, "I_shared": w.Is},
            "us_per_call_warm": round(ms_warm * 1e3, 2),
            "us_per_call_cold_l2": round(ms_cold * 1e3, 2),
            "l2": f"cold: a {flush_bytes >> 20} MB buffer written before every call",
            "gpu_launches_per_call": launches_per_step(w, with_affinity=True)}


def measure_side_workload(name, weights, dev, args, sampler, peaks, peak_src, barrier,
                          weights8=None):
    """One row of the workloads table: the same call as the headline on another batch (with
    weights8, the FP8 layer on those pre-quantised experts)."""
    import torch

    from expert_routed_ffn_router_gb300 import synth
    fp8 = weights8 is not None
    w = synth.workload(name)
    routing = synth.routing_inputs(w)
    layer, _, _, X = _layer_for(w, routing, weights, dev, None, fp8, weights8)
    stream = torch.cuda.current_stream()
    t_busy0 = time.time()
    for _ in range(args.warmup):
        layer.forward(X)
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError(f"device status word reported an error during warm-up ({name})")
    ms, t0, t1 = _timed(layer, X, args.steps, stream, barrier)
    stage_ms = _stage_pass(layer, X, args.steps, stream)
    t_busy1 = time.time()
    if layer.status() != 0:
        raise RuntimeError(f"device status word reported an error ({name})")
    counts = layer.counts.cpu().numpy()
    n_act = int((counts > 0).sum())
    lr = layer_roofline(w, n_act, ms, peaks, fp8)
    key, tgt = target_of(w) if not fp8 else (None, None)
    row = {"T": w.T, "ms_per_step": round(ms, 4), "tokens_per_s": round(w.T / (ms / 1e3), 1),
           "n_active_experts": n_act, **lr,
           "dominant_kernel": dominant_roofline(w, n_act, stage_ms, peaks, peak_src, fp8),
           "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
           "gpu_launches": args.steps * launches_per_step(w, with_affinity=True, fp8=fp8),
           "clocks": sampler.summary(t0, t1, t_busy0, t_busy1)}
    if fp8:
        row["precision"] = ("FP8 E4M3 experts, 128 x 128 weight / 1 x 128 activation block "
                            "scales, on the FP8 tensor cores")
    if key:
        row["target"] = {"metric": key, "min": tgt, "met": bool(lr[key] >= tgt)}
    if name == "skewed":
        row["routing_stats"] = skew_stats(counts, layer.affinity.cpu().numpy(), w.T)
    del layer
    torch.cuda.empty_cache()
    return row


def skew_stats(counts, affinity, T: int, cluster: int = 32) -> dict:
    """What the skewed recipe aims at, read off the layer's own counts and co-activation
    matrix: the log-log slope of count against popularity rank (ranks >= 3, the two
    capped at T left out) and the share of co-activations inside a cluster of 32 experts."""
    import numpy as np
    c = np.sort(np.asarray(counts, dtype=np.float64))[::-1]
    r = np.arange(1, c.size + 1)
    m = (c > 0) & (r >= 3)
    slope = float(np.polyfit(np.log(r[m]), np.log(c[m]), 1)[0]) if m.sum() >= 2 else None
    A = np.asarray(affinity, dtype=np.int64)
    g = np.arange(A.shape[0]) // cluster
    tot = int(A.sum())
    within = float(A[g[:, None] == g[None, :]].sum() / tot) if tot else None
    return {"zipf_slope": None if slope is None else round(slope, 3),
            "within_cluster_coactivation": None if within is None else round(within, 4),
            "top_counts": [int(x) for x in c[:3]], "cap": int(T)}


def run_ours(args, rank, world, local_rank):
    import torch

    from expert_routed_ffn_router_gb300 import binding as B
    from expert_routed_ffn_router_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    B.load()
    w = replica_workload(args.workload, rank)
    routing = synth.routing_inputs(w)
    weights = synth.expert_weights_device(w, dev)
    opts = ROUTINGS[args.routing]
    fp8 = args.precision == "fp8"
    layer, wts, X_host, X = _layer_for(w, routing, weights, dev, opts, fp8)
    peaks, peak_src = load_peaks()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    sampler.start()
    stream = torch.cuda.current_stream()
    t_busy0 = time.time()
    for _ in range(args.warmup):
        layer.forward(X)
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError("device status word reported an error during warm-up")

    # ---- device-resident timed region: the bare layer call, inputs already in HBM
    K = args.steps
    ms_rank, t_wall0, t_wall1 = _timed(layer, X, K, stream, barrier)
    ms = max_over_ranks(ms_rank, dev)
    if layer.status() != 0:
        raise RuntimeError("device status word reported an error in the timed region")
    # ---- per-stage times (a separate, instrumented pass)
    stage_ms = _stage_pass(layer, X, K, stream)

    # ---- end to end: pinned host input -> layer -> pinned host output, every step.  The
    # copies run on their own stream and overlap the neighbouring steps' compute: step k's
    # input is copied in while step k - 1 computes, its output copied out while step k + 1
    # computes (two sets of device inputs, outputs and workspaces alternate).
    Xh = X_host.pin_memory()
    Yh = [torch.empty(w.T, w.H, dtype=torch.float32).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(X) for _ in range(2)]
    layers = [layer, B.MoELayer(wts, w.T, w.K, with_affinity=True, routing=opts, fp8=fp8,
                                weights8=layer.w8)]
    copy_s = torch.cuda.Stream(device=dev)

    def e2e_steps(n):
        ev_x = [torch.cuda.Event() for _ in range(2)]
        ev_y = [torch.cuda.Event() for _ in range(2)]
        with torch.cuda.stream(copy_s):
            Xd[0].copy_(Xh, non_blocking=True)
            ev_x[0].record(copy_s)
        for k in range(n):
            b = k & 1
            stream.wait_event(ev_x[b])
            layers[b].forward(Xd[b])
            ev_y[b].record(stream)
            with torch.cuda.stream(copy_s):
                if k + 1 < n:
                    # buffer 1 - b was last read by step k - 1, whose output copy (queued
                    # on this stream before) waited for that step
                    Xd[1 - b].copy_(Xh, non_blocking=True)
                    ev_x[1 - b].record(copy_s)
                copy_s.wait_event(ev_y[b])
                Yh[b].copy_(layers[b].Y, non_blocking=True)
        stream.wait_stream(copy_s)

    e2e_steps(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_s.wait_event(e0)
    e2e_steps(K)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_busy1 = time.time()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / K, dev)
    if any(l.status() != 0 for l in layers):
        raise RuntimeError("device status word reported an error in the end-to-end region")
    del layers[1]
    clocks = sampler.summary(t_wall0, t_wall1, t_busy0, t_busy1)

    counts = layer.counts.cpu().numpy()
    n_act = int((counts > 0).sum())
    # GRACE-MoE placement for expert parallelism over 8 GPUs (4 per node), planned on the
    # host from this step's counts and co-activation matrix (outside the timed regions)
    A = layer.affinity.cpu().numpy()
    t_plan = time.perf_counter()
    plan = B.moe_grace_choose_r(A, 8, [0.0, 0.125, 0.25, 0.375, 0.5])
    rep = B.moe_grace_replicate(counts, plan["group_of"], 8)
    B.moe_grace_route_table(rep, 4)
    ms_plan = (time.perf_counter() - t_plan) * 1e3
    roof = dominant_roofline(w, n_act, stage_ms, peaks, peak_src, fp8)
    lr = layer_roofline(w, n_act, ms, peaks, fp8)

    total_tokens = w.T * world
    value = total_tokens / (ms / 1e3)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 experts (128x128 / 1x128 block scales), bf16 activations" if fp8 else "bf16",
        "data": "synthetic (seeded; random-init weights of the DeepSeek-V3 MoE shape)",
        "config": {"workload": workload_desc(w),
                   "tokens_per_gpu": w.T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: the activated experts' weights "
                         f"({lr['algorithmic_bytes'] / 1e9:.1f} GB) stream from HBM every step",
                   "n_active_experts": n_act,
                   "shared_expert": ("own FFN launch on a side stream beside the router and "
                                     "the dispatch" if shared_on_side(w, fp8) else
                                     "second problem of the routed FFN launch")},
        **({"routing": {"name": args.routing, **opts}} if opts else {}),
        "e2e": {"value": round(total_tokens / (ms_e2e / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size()),
                "d2h_bytes_per_step": int(Yh[0].numel() * Yh[0].element_size()),
                "copies": "own stream, overlapping the neighbouring steps' compute"},
        "gpu_launches": K * launches_per_step(w, with_affinity=True, fp8=fp8),
        "roofline": roof,
        "layer_roofline": lr,
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stages_note": "from a separate pass of the same calls with the library's stage "
                       "events recorded; the timed region runs the bare call",
        "grace_plan": {"gpus": 8, "gpus_per_node": 4, "r": plan["r"],
                       "U": round(float(plan["U"][plan["knee"]]), 4),
                       "S": round(float(plan["S"][plan["knee"]]), 4),
                       "rho": round(rep["rho"], 4), "n_replica": rep["n_replica"],
                       "n_hot": len(rep["hot"]), "planner_ms": round(ms_plan, 1)},
        "clocks": clocks,
    }
    del layer
    torch.cuda.empty_cache()
    if (world == 1 and args.workload == "decode" and not fp8 and opts is None
            and not args.no_workloads):
        rows = {}
        for name in SIDE_WORKLOADS:
            rows[name] = measure_side_workload(name, weights, dev, args, sampler, peaks,
                                               peak_src, barrier)
        rows["decode"] = {"T": w.T, "ms_per_step": round(ms, 4),
                          "tokens_per_s": round(value, 1), "n_active_experts": n_act, **lr,
                          "note": "the headline above"}
        # the same decode step with FP8 experts (the pages' serving precision; the experts
        # quantised once, outside every timed region)
        weights8 = B.quantize_expert_weights_fp8({**weights, "W_gate": None, "bias": None})
        torch.cuda.synchronize()
        rows["decode_fp8"] = measure_side_workload("decode", weights, dev, args, sampler, peaks,
                                                   peak_src, barrier, weights8=weights8)
        del weights8
        torch.cuda.empty_cache()
        rows["tiny"] = measure_tiny(dev, args.steps)
        out["workloads"] = rows
        out["targets"] = {n: r["target"] for n, r in rows.items() if "target" in r}
    sampler.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not fp8:
        out["cpu_baseline"] = cpu_baseline(w, routing, weights, budget_s=args.cpu_budget,
                                           opts=opts)
    return out


# --------------------------------------------------------------------- oracle (CPU)
def _oracle_route(w, routing, X, opts):
    import oracle
    if opts:
        return oracle.router_ex(X, routing["W_gate"], routing["bias"], w.K, **opts)
    return oracle.router(X, routing["W_gate"], routing["bias"], w.K)


def _oracle_step(w, routing, weights, tokens, host_cache, opts=None):
    """One oracle pass over `tokens`: router for those tokens + their experts + shared."""
    from expert_routed_ffn_router_gb300 import synth
    X = routing["X"][tokens]
    idx, wt = _oracle_route(w, routing, X, opts)
    used = sorted({int(e) for e in idx.ravel()})
    for e in used:
        if e not in host_cache:
            host_cache[e] = tuple(synth.bf16_tensor_to_bits(weights[n][e]) for n in ("W1", "W3", "W2"))
    if "shared" not in host_cache and w.Is:
        host_cache["shared"] = tuple(synth.bf16_tensor_to_bits(weights[n]) for n in ("W1s", "W3s", "W2s"))
    return X, idx, wt, used


def _oracle_timed(w, routing, weights, tokens, host_cache, opts=None):
    import numpy as np

    import oracle
    X, idx, wt, used = _oracle_step(w, routing, weights, tokens, host_cache, opts)
    t0 = time.perf_counter()
    idx, wt = _oracle_route(w, routing, X, opts)
    sh = host_cache.get("shared", (None, None, None))
    oracle.layer_tokens(X, idx, wt, {e: host_cache[e][0] for e in used},
                        {e: host_cache[e][1] for e in used}, {e: host_cache[e][2] for e in used},
                        *sh, np.arange(len(tokens)), w.I, w.Is)
    return time.perf_counter() - t0


def cpu_baseline(w, routing, weights, budget_s=12.0, opts=None):
    import numpy as np

    import oracle
    cores = oracle.num_threads()
    cache = {}
    n1 = cores
    t1 = _oracle_timed(w, routing, weights, np.arange(n1) % w.T, cache, opts)
    per_tok = t1 / n1
    # about budget_s of work: the workload's tokens in order, wrapping around for small
    # batches (at most 8 passes)
    n = int(min(8 * w.T, max(n1, round(budget_s / max(per_tok, 1e-6)))))
    tokens = np.arange(n) % w.T
    t = _oracle_timed(w, routing, weights, tokens, cache, opts)
    def sample_of(m):
        return (f"first {m} of the {w.T} tokens of the workload" if m <= w.T else
                f"{m} tokens: the workload's {w.T} tokens, {m / w.T:.1f} passes")
    which = sample_of(n)
    out = {"value": round(n / t, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{which}: fp64 router over all {w.E} experts + the {w.K} routed "
                     f"experts and the shared expert of each token ({t:.1f} s)"}
    # the same on one core, a smaller sample (about a tenth of the budget)
    n_one = int(max(1, min(n, round(0.1 * budget_s / max(per_tok * cores, 1e-6)))))
    prev = oracle.set_num_threads(1)
    try:
        t_one = _oracle_timed(w, routing, weights, np.arange(n_one) % w.T, cache, opts)
    finally:
        oracle.set_num_threads(prev)
    out["one_core"] = {"value": round(n_one / t_one, 3), "unit": UNIT, "cores": 1,
                       "sample": f"{sample_of(n_one)} ({t_one:.1f} s)"}
    return out


def run_reference(args):
    import numpy as np
    import torch

    import oracle
    from expert_routed_ffn_router_gb300 import synth
    w = synth.workload(args.workload)
    routing = synth.routing_inputs(w)
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    weights = synth.expert_weights_device(w, dev)
    cores = oracle.num_threads()
    cache = {}
    # size each step so that warm-up + timed steps take about two minutes
    opts = ROUTINGS[args.routing]
    t1 = _oracle_timed(w, routing, weights, np.arange(cores) % w.T, cache, opts)
    per_tok = t1 / cores
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.T, round(budget / max(per_tok, 1e-6)))))
    rng = np.random.default_rng(0)
    steps_tok = [rng.choice(w.T, size=n, replace=False) for _ in range(args.warmup + args.steps)]
    for k in range(args.warmup):
        _oracle_timed(w, routing, weights, steps_tok[k], cache, opts)
    tt = 0.0
    for k in range(args.steps):
        tt += _oracle_timed(w, routing, weights, steps_tok[args.warmup + k], cache, opts)
    value = n * args.steps / tt
    return {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": workload_desc(w), "tokens_per_gpu": w.T,
                   **({"routing": {"name": args.routing, **opts}} if opts else {})},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} random tokens of the {w.T}-token workload per step"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="decode",
                    help="decode (default), tiny, sweep2..sweep256, prefill, skewed")
    ap.add_argument("--routing", choices=sorted(ROUTINGS), default="default",
                    help="routing options of other MoE families (default: the plain router)")
    ap.add_argument("--precision", choices=("bf16", "fp8"), default="bf16",
                    help="expert weights: bf16 (default) or FP8 E4M3 with 128x128 block scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure the headline workload only (skip the sweep, skewed and "
                         "prefill rows measured beside the decode headline)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        # one process per GPU: N GPUs need N ranks (torch.distributed.run --nproc-per-node N)
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one process per "
                 "GPU with torch.distributed.run --nproc-per-node N")

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
