#!/usr/bin/env python
"""Benchmark of the MoE expert layer (moe_forward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--only]
                    [--impl ours|reference] [--weights fp4|bfp8]

One step = one moe_forward (activation cast, routing, counting-sort permute,
GEMM1 + SwiGLU (.) weight + FP8 requantisation, GEMM2, combine) over the
workload's T tokens, replayed from a CUDA graph.  The headline workload
(--workload, default: the skewed prefill, T=8192, H=7168, I=2048, E=256,
top-8, the largest configuration) gives `value`; the other four workloads
follow under `per_workload` (--only skips them).  Inputs are seeded synthetic
tensors (workloads/), resident in HBM when timing starts.  L2 is flushed
between timed steps (512 MiB written, then 512 MiB read, so no dirty flush
lines are written back inside the timed step).  Each step is bracketed by CUDA
events on the launching stream; the headline's timed region is bracketed by
a barrier and torch.cuda.synchronize(), with nvidia-smi sampling the clocks.

`roofline` describes the layer's dominant GEMM launch, timed alone on the
state a whole-layer call left (moe_forward's `phases`): the single launch of
GEMM1 + GEMM2 + combine for small problems, else the longer of the GEMM1 and
GEMM2 launches.

Multi-GPU: the layer does not shard across GPUs here (replicas only): with N
ranks each GPU runs its own independent replica, value = all ranks' tokens /
max-over-ranks time, "scaling": "weak".

`cpu_baseline` times the CPU oracle (oracle/, float64) on this host's cores on
a bounded sample: one token for the large workloads, every token of the small
decode.  --impl reference times the oracle alone as the reference arm (rank 0
only): one token per step for small workloads, one (token, slot) pair per step
for the large ones.

--weights bfp8 times the block-FP8 variant instead (moe_forward_bfp8: E4M3
weights with 128 x 128 block scales, per-128 token scales), on the same
workload shapes and inputs.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; % of roofline (FP8 tensor peak or HBM GB/s)"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# GEMM launches, from one-pass ncu captures (ncu flushes the caches before
# each captured launch) of the kernels built from sources whose SHA-256 is
# `src_sha256` (commands and figures in profiles/dram_traffic_gemm.md).  The
# prefills were captured on smaller cases with the same per-expert shapes
# (workloads.PROFILE_WORKLOADS) and enter as the ratio of measured to
# algorithmic bytes of that case, applied to the full workload's algorithmic
# bytes; the small decode was captured at full size.  `traffic` is reported
# as null once those sources change or for launches not captured.
PAIR_SOURCES = ("gemm2sm.cu", "gemm_common.cuh", "ptx.cuh", "layer_blocks.cuh", "host_common.h")
ONE_CTA_SOURCES = ("gemm.cu", "gemm_common.cuh", "ptx.cuh", "layer_blocks.cuh", "host_common.h")
TRAFFIC = {
    # the CTA-pair kernel (208-token tiles)
    "pair": {
        "sources": PAIR_SOURCES,
        "src_sha256": "06266b645b27a68e982d192fe8a19bf1f49d5f3aeaba799c6f018472937ddf9d",
        "prefill": {"gemm1": {"ratio": (533650944 + 8379392) / 511557632, "from": "prefill_e32"},
                    "gemm2": {"ratio": (258542592 + 38111744) / 316932096, "from": "prefill_e32"}},
        "skewed_prefill": {"gemm1": {"ratio": (1188315136 + 33220864) / 1047986176, "from": "skewed_e64"},
                           "gemm2": {"ratio": (535210240 + 196240896) / 768606208, "from": "skewed_e64"}},
    },
    # the one-CTA kernel (small tiles; the small decode's fused launch)
    "one_cta": {
        "sources": ONE_CTA_SOURCES,
        "src_sha256": "00bb534b5938cedf0335fbbd77d700aa126883961cdaf1ab36e8a59c9fa53683",
        "small_decode": {"fused": {"bytes": 94067968 + 1623040, "from": "small_decode (full size)"}},
    },
}
# the same for the block-FP8 variant's GEMMs (csrc/bfp8.cu)
BFP8_SOURCES = ("bfp8.cu", "ptx.cuh", "layer_blocks.cuh", "host_common.h")
TRAFFIC_BFP8 = {
    "src_sha256": "79311228cdde91d3cbb71523b34469c098f4a6b51a34adabb51fdec33e737862",
    "small_decode": {"gemm1": 117678592 + 65280, "gemm2": 58821888 + 25856},
}
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="skewed_prefill")
    ap.add_argument("--only", action="store_true", help="measure only --workload (no per_workload entries)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--schedule", type=int, default=0, choices=[0, 1, 2],
                    help="large CTA-pair problems: 0 library default, 1 separate launches, 2 expert waves (one launch)")
    ap.add_argument("--weights", default="fp4", choices=["fp4", "bfp8"],
                    help="fp4: FP8 x FP4 with UE8M0 per 32 (moe_forward); bfp8: block-FP8 weights (moe_forward_bfp8)")
    ap.add_argument("--no-flush", action="store_true", help="skip the L2 flush (for profiler launch lists)")
    ap.add_argument("--quick", action="store_true", help="skip the CPU-baseline and e2e legs")
    ap.add_argument("--launch-list", action="store_true",
                    help="profiler mode: only warm-up + timed graph replays, no flush, soak or extra legs")
    return ap.parse_args()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler running while the GPU is busy."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(dev) -> str:
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev.index or 0] if vis else str(dev.index or 0)


# ---------------------------------------------------------------- roofline bookkeeping

def gemm_sources_sha256(sources):
    import hashlib
    h = hashlib.sha256()
    base = os.path.join(os.path.dirname(os.path.abspath(__file__)), "moe_expert_layer_counting_gb300", "csrc")
    for name in sources:
        with open(os.path.join(base, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload, phase, alg_bytes, bfp8=False):
    """(bytes per launch, how) from the ncu tables above, or (None, why) if stale or not captured."""
    if bfp8:
        table, sources = TRAFFIC_BFP8, BFP8_SOURCES
    else:
        table = next((f for f in TRAFFIC.values() if phase in f.get(workload, {})), None)
        if table is None:
            return None, "not captured"
        sources = table["sources"]
    if table.get("src_sha256") != gemm_sources_sha256(sources):
        return None, "kernel sources changed since the capture"
    entry = table.get(workload, {}).get(phase)
    if entry is None:
        return None, "not captured"
    if isinstance(entry, dict) and "ratio" in entry:
        return int(round(entry["ratio"] * alg_bytes)), f"scaled from {entry['from']} (measured / algorithmic = {entry['ratio']:.4f})"
    if isinstance(entry, dict):
        return entry["bytes"], f"measured on {entry['from']}"
    return entry, "measured at full size"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def algorithmic(wl, counts):
    """Algorithmic bytes / flops of the layer and of each GEMM (one launch)."""
    touched = int((counts > 0).sum())
    P = wl.T * wl.k
    w1 = 2 * wl.I * (wl.H // 2 + wl.H // 32)           # per expert
    w2 = wl.H * (wl.I // 2 + wl.I // 32)
    x_q = wl.T * (wl.H + wl.H // 32)                   # FP8 activations + scales
    h_q = P * (wl.I + wl.I // 32)
    y_pairs = P * wl.H * 2
    return {
        "touched_experts": touched,
        "layer_bytes": wl.T * wl.H * 2 + wl.T * wl.E * 4 + touched * (w1 + w2) + wl.T * wl.H * 2,
        "layer_flops": 2 * P * 3 * wl.H * wl.I,
        "gemm1_bytes": touched * w1 + x_q + h_q,
        "gemm1_flops": 2 * P * 2 * wl.I * wl.H,
        "gemm2_bytes": touched * w2 + h_q + y_pairs,
        "gemm2_flops": 2 * P * wl.H * wl.I,
        # GEMM1 + GEMM2 + combine in one launch: h and the per-pair rows stay on
        # chip / in L2, so the launch's algorithmic bytes are the weights, the
        # cast tokens and y
        "fused_bytes": touched * (w1 + w2) + x_q + wl.T * wl.H * 2,
        "fused_flops": 2 * P * 3 * wl.H * wl.I,
    }


def algorithmic_bfp8(wl, counts):
    """The same for the block-FP8 variant: one byte per weight plus one float32
    scale per 128 x 128 block; FP8 tokens and h with one float32 scale per 128;
    GEMM2 writes FP32 pair rows."""
    touched = int((counts > 0).sum())
    P = wl.T * wl.k
    w1 = 2 * wl.I * wl.H + (2 * wl.I // 128) * (wl.H // 128) * 4
    w2 = wl.H * wl.I + (wl.H // 128) * (wl.I // 128) * 4
    x_q = wl.T * (wl.H + wl.H // 128 * 4)
    h_q = P * (wl.I + wl.I // 128 * 4)
    y_pairs = P * wl.H * 4
    return {
        "touched_experts": touched,
        "layer_bytes": wl.T * wl.H * 2 + wl.T * wl.E * 4 + touched * (w1 + w2) + wl.T * wl.H * 2,
        "layer_flops": 2 * P * 3 * wl.H * wl.I,
        "gemm1_bytes": touched * w1 + x_q + h_q,
        "gemm1_flops": 2 * P * 2 * wl.I * wl.H,
        "gemm2_bytes": touched * w2 + h_q + y_pairs,
        "gemm2_flops": 2 * P * wl.H * wl.I,
    }


def layer_rates(alg, ms_per_step):
    """Whole-layer rates of one step: algorithmic GB/s and TFLOP/s."""
    sec = ms_per_step * 1e-3
    return {"gbs": round(alg["layer_bytes"] / sec / 1e9, 1), "tflops": round(alg["layer_flops"] / sec / 1e12, 3),
            "algorithmic_bytes": alg["layer_bytes"], "algorithmic_flops": alg["layer_flops"]}


# ---------------------------------------------------------------- ranks

def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of per-rank floats over the process group (the
    slowest rank decides a timed region); the values themselves for one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def replica_tokens_per_s(world, tokens, steps, total_ms):
    """Whole-job throughput of `world` independent replicas that each processed
    `tokens` per step for `steps` steps within the max-over-ranks `total_ms`."""
    return world * tokens * steps / (total_ms / 1e3)


# ---------------------------------------------------------------- our arm

ALL_WORKLOADS = ("tiny", "small_decode", "large_decode", "prefill", "skewed_prefill")


def timed_loop(stream, step_fn, steps, flush=None, pre=None):
    """CUDA-event time (ms) of each of `steps` calls of step_fn on `stream`;
    before each: flush (L2) and pre (untimed set-up), outside the events."""
    import torch
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            if flush:
                flush()
            if pre:
                pre()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_fn()
            b.record(stream)
            evs.append((a, b))
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def roofline_of(alg, key, ms, hbm, fp8_peak_tflops):
    """Roofline entry of one launch: algorithmic bytes and flops of `key`
    against the measured copy bandwidth / FP8 rate, whichever bound is higher."""
    nbytes, flops = alg[f"{key}_bytes"], alg[f"{key}_flops"]
    if nbytes / (hbm * 1e9) >= flops / (fp8_peak_tflops * 1e12):
        achieved = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "algorithmic_bytes": nbytes, "algorithmic_flops": flops}
    achieved = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": fp8_peak_tflops, "unit": "TFLOP/s",
            "frac": round(achieved / fp8_peak_tflops, 4), "algorithmic_bytes": nbytes, "algorithmic_flops": flops}


def measure(args, wl, dev, stream, world, rank, headline):
    """One workload: weights, the layer replayed from a CUDA graph (timed), its
    GEMM launch(es) timed alone, the roofline; for the headline also the
    clocks, the end-to-end leg and the CPU baseline."""
    import torch

    import workloads as W
    from moe_expert_layer_counting_gb300 import binding as B
    from moe_expert_layer_counting_gb300.layer import QuantizedExperts

    x_cpu, logits_cpu = W.tokens(wl)
    x = x_cpu.to(dev)
    logits = logits_cpu.to(dev)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    bfp8 = args.weights == "bfp8"
    if bfp8:
        w1q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        w1s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        w2q = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
        for e in range(E):
            l1, l2 = W.expert_weights(wl, e, dev)
            B.bfp8_quantize_weight(l1[None], w1q[e:e + 1], w1s[e:e + 1])
            B.bfp8_quantize_weight(l2[None], w2q[e:e + 1], w2s[e:e + 1])
        ws = torch.empty(B.moe_bfp8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    else:
        qe = QuantizedExperts(wl.E, wl.H, wl.I, device=dev)
        for e in range(wl.E):
            l1, l2 = W.expert_weights(wl, e, dev)
            qe.set_expert(e, l1, l2)
        ws = torch.empty(B.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    del l1, l2
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def forward(st, phases=0, xb=None, lb=None, yb=None):
        xb = x if xb is None else xb
        lb = logits if lb is None else lb
        yb = y if yb is None else yb
        if bfp8:
            B.moe_forward_bfp8(xb, lb, w1q, w1s, w2q, w2s, k, yb, ws, topk_idx_out=idx, topk_w_out=wts,
                               counts_out=counts, offsets_out=offsets, perm_out=perm, phases=phases, stream=st)
        else:
            B.moe_forward(xb, lb, qe.w1q, qe.w1s, qe.w2q, qe.w2s, k, yb, ws, topk_idx_out=idx, topk_w_out=wts,
                          counts_out=counts, offsets_out=offsets, perm_out=perm, tile_n=args.tile_n,
                          phases=phases, schedule=args.schedule, stream=st)

    def flush():
        if not args.no_flush:
            flush_w.zero_()
            flush_r.sum()

    with torch.cuda.stream(stream):
        forward(stream)                       # first call outside capture (sets kernel attributes)
    stream.synchronize()
    assert B.moe_get_device_status(ws, stream) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        forward(torch.cuda.current_stream())
    counts_np = counts.cpu().numpy()
    n_launch_forward = (launches_per_forward_bfp8(T, H, E, k) if bfp8 else
                        launches_per_forward(T, H, I, E, k, args.schedule))
    fused = (not bfp8) and single_gemm_launch(T, H, I, E, k, args.schedule)   # GEMM1 + GEMM2 + combine, one launch
    loop = lambda fn, n, **kw: timed_loop(stream, fn, n, flush=flush, **kw)  # noqa: E731

    if args.launch_list:
        loop(graph.replay, args.warmup + args.steps)
        # then one launch of the layer's GEMM launch(es) alone (the kernels the roofline figures describe)
        with torch.cuda.stream(stream):
            if fused:
                forward(stream, B.PHASE_RESET)
                forward(stream, B.PHASE_GEMM1 | B.PHASE_GEMM2)
            else:
                forward(stream, B.PHASE_GEMM1)
                forward(stream, B.PHASE_GEMM2)
        torch.cuda.synchronize()
        return {"launch_list": True, "workload": wl.describe(), "replays": args.warmup + args.steps}

    loop(graph.replay, args.warmup)
    clk = None
    if headline:
        # a short soak so that the clock sampler sees the GPU under load, then
        # the timed region bracketed by a barrier and a device synchronisation
        if world > 1:
            torch.distributed.barrier()
        with ClockSampler(gpu_id_for(dev)) as clk:
            t_soak = time.time()
            while time.time() - t_soak < 1.5:
                loop(graph.replay, 20)
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            t0 = time.time()
            times = loop(graph.replay, args.steps)
            torch.cuda.synchronize()
            wall = time.time() - t0
            if world > 1:
                torch.distributed.barrier()
        total_ms, mean_ms = max_over_ranks([sum(times), sum(times) / len(times)], world, dev)
    else:
        times = loop(graph.replay, args.steps)
        total_ms, mean_ms = sum(times), sum(times) / len(times)
    assert B.moe_get_device_status(ws, stream) == 0, "device status word reports an error"
    value = replica_tokens_per_s(world if headline else 1, T, args.steps, total_ms)

    # the layer's GEMM launch(es) alone, on the state the forward left
    nt = max(args.steps, 20)
    if fused:
        g_ms = statistics.mean(loop(lambda: forward(stream, B.PHASE_GEMM1 | B.PHASE_GEMM2), nt,
                                    pre=lambda: forward(stream, B.PHASE_RESET)))
        gemm_ms = {"gemm1_gemm2_combine": round(g_ms, 5)}
    else:
        g1 = statistics.mean(loop(lambda: forward(stream, B.PHASE_GEMM1), nt))
        g2 = statistics.mean(loop(lambda: forward(stream, B.PHASE_GEMM2), nt))
        gemm_ms = {"gemm1": round(g1, 5), "gemm2": round(g2, 5)}
    assert B.moe_get_device_status(ws, stream) == 0

    alg = algorithmic_bfp8(wl, counts_np) if bfp8 else algorithmic(wl, counts_np)
    hbm, bf16, peak_src = peaks()
    fp8_peak_tflops = 2 * bf16                      # FP8 dense = 2x BF16 dense (nominal ratio)
    kname = "bfp8_gemm_kernel" if bfp8 else "expert_gemm_kernel"
    if fused:
        dom, dom_ms = "fused", g_ms
        what = (f"{kname}<16, GEMM1 + GEMM2 + combine> (one launch)" if T <= 64 else
                "expert_gemm_pair_kernel<GEMM1 + GEMM2 + combine> (one launch, CTA pairs, expert waves)")
    else:
        dom = "gemm1" if g1 >= g2 else "gemm2"
        dom_ms = max(g1, g2)
        what = (f"expert_gemm_pair_kernel ({dom}, one launch, CTA pairs)" if (not bfp8 and pair_tiles(T, H, I, E, k))
                else f"{kname} ({dom}, one launch)")
    roof = roofline_of(alg, dom, dom_ms, hbm, fp8_peak_tflops)
    traffic, traffic_how = measured_traffic(wl.name, dom, roof["algorithmic_bytes"], bfp8)
    roof.update({"kernel": what, "ms": round(dom_ms, 5), "traffic": traffic, "traffic_source": traffic_how,
                 "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs; fp8 = 2 x bf16_tflops)"})
    layer_time_bound = max(alg["layer_bytes"] / (hbm * 1e9), alg["layer_flops"] / (fp8_peak_tflops * 1e12))
    out = {
        "value": round(value, 1), "ms_per_step": round(mean_ms, 5),
        "config": {"workload": wl.describe() + (" block-FP8 weights" if bfp8 else ""), "tokens_per_step": T,
                   "pairs": T * k, "weights": args.weights + (" (tile-contiguous codes)" if bfp8 else ""),
                   "touched_experts": alg["touched_experts"], "tile_n": args.tile_n or "auto",
                   "l2": "flushed between steps (512 MiB write + 512 MiB read)" if not args.no_flush else "not flushed",
                   "cuda_graph": True, "parallelism": "replicas" if world > 1 else "single GPU",
                   "schedule": {0: "default", 1: "separate", 2: "expert waves"}[args.schedule]},
        "layer_roofline_frac": round(layer_time_bound / (mean_ms * 1e-3), 4),
        "layer_rates": layer_rates(alg, mean_ms),
        "gemm_ms": gemm_ms,
        "roofline": roof,
        "gpu_launches": n_launch_forward * args.steps,
    }
    if headline:
        # context for the fraction: PyTorch kernels moving the same number of DRAM
        # bytes as the dominant kernel, cold L2 like the kernel -- a copy (half the
        # bytes read, half written) and a read-only reduction (sum)
        dom_bytes = roof["algorithmic_bytes"]
        half = max(dom_bytes // 8, 1)                   # float32 elements in half the bytes
        cp_src = torch.ones(half, dtype=torch.float32, device=dev)
        cp_dst = torch.empty_like(cp_src)
        copy_ms = statistics.median(loop(lambda: cp_dst.copy_(cp_src), nt))
        del cp_src, cp_dst
        read_buf = torch.ones(max(dom_bytes // 4, 1), dtype=torch.float32, device=dev)
        read_out = torch.empty((), dtype=torch.float32, device=dev)
        read_ms = statistics.median(loop(lambda: torch.sum(read_buf, dim=(0,), out=read_out), nt))
        del read_buf
        out["same_size_reference"] = {
            "bytes": dom_bytes, "copy_ms": round(copy_ms, 5),
            "copy_gbs": round(dom_bytes / (copy_ms * 1e-3) / 1e9, 1), "sum_ms": round(read_ms, 5),
            "sum_gbs": round(dom_bytes / (read_ms * 1e-3) / 1e9, 1),
            "what": "PyTorch copy_ of bytes/2 (bytes of DRAM traffic) and torch.sum over bytes, float32, "
                    "L2 flushed before each call (median)"}
        out["wall_s_timed_region"] = round(wall, 4)
        out["clocks"] = clk.summary()
        if not args.quick:
            # end to end through the public API with host buffers: H2D inputs, layer, D2H output
            x_h = x_cpu.pin_memory()
            l_h = logits_cpu.pin_memory()
            y_h = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

            def e2e_step():
                x.copy_(x_h, non_blocking=True)
                logits.copy_(l_h, non_blocking=True)
                graph.replay()
                y_h.copy_(y, non_blocking=True)

            # (a) one step at a time: copy in, layer, copy out, L2 flushed between steps
            serial_times = loop(e2e_step, args.steps)
            serial_total = max_over_ranks([sum(serial_times)], world, dev)[0]
            # (b) as a serving loop runs it: step s's inputs are copied in on one
            # copy stream while step s-1's layer runs, its output copied out on
            # another while step s+1's runs (two buffer sets, a graph for each);
            # every step's copies are inside the timed region, which spans all
            # steps (events on the first copy-in and after the last copy-out)
            bx = [x, torch.empty_like(x)]
            bl = [logits, torch.empty_like(logits)]
            by = [y, torch.empty_like(y)]
            byh = [y_h, torch.empty(T, H, dtype=torch.bfloat16).pin_memory()]
            graph2 = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                forward(stream, xb=bx[1], lb=bl[1], yb=by[1])
            stream.synchronize()
            with torch.cuda.graph(graph2, stream=stream):
                forward(torch.cuda.current_stream(), xb=bx[1], lb=bl[1], yb=by[1])
            graphs = [graph, graph2]
            cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

            def pipelined(nsteps):
                in_ready = [torch.cuda.Event() for _ in range(2)]
                done = [torch.cuda.Event() for _ in range(2)]
                out_done = [torch.cuda.Event() for _ in range(2)]
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                t0.record(cin)
                for s_ in range(nsteps):
                    b = s_ % 2
                    if s_ >= 2:
                        cin.wait_event(done[b])              # the layer of step s-2 has read bx[b], bl[b]
                    with torch.cuda.stream(cin):
                        bx[b].copy_(x_h, non_blocking=True)
                        bl[b].copy_(l_h, non_blocking=True)
                    in_ready[b].record(cin)
                    stream.wait_event(in_ready[b])
                    if s_ >= 2:
                        stream.wait_event(out_done[b])       # step s-2's output has left by[b]
                    with torch.cuda.stream(stream):
                        graphs[b].replay()
                    done[b].record(stream)
                    cout.wait_event(done[b])
                    with torch.cuda.stream(cout):
                        byh[b].copy_(by[b], non_blocking=True)
                    out_done[b].record(cout)
                t1.record(cout)
                t1.synchronize()
                return t0.elapsed_time(t1)

            pipelined(max(args.warmup, 3))
            pipe_ms = max_over_ranks([pipelined(args.steps)], world, dev)[0]
            wbytes = int(alg["layer_bytes"] - 2 * T * H * 2 - T * E * 4)
            out["e2e"] = {"value": round(replica_tokens_per_s(world, T, args.steps, pipe_ms), 1), "unit": UNIT,
                          "h2d_bytes_per_step": x_h.numel() * 2 + l_h.numel() * 4,
                          "d2h_bytes_per_step": y_h.numel() * 2,
                          "how": "moe_forward with host buffers as a serving loop: step s's H2D copies overlap "
                                 "step s-1's layer, its D2H copy step s+1's (two buffer sets, two copy streams); "
                                 f"timed over all {args.steps} steps; L2 not flushed (each step reads "
                                 f"{wbytes / 1e9:.2f} GB of expert weights, above the 129 MB L2)",
                          "serial": {"value": round(replica_tokens_per_s(world, T, args.steps, serial_total), 1),
                                     "how": "copy in, layer, copy out per step on one stream, L2 flushed "
                                            "between steps"}}
            del graph2
    del graph
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    import workloads as W
    wl = W.WORKLOADS.get(args.workload) or W.PROFILE_WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    head = measure(args, wl, dev, stream, world, rank, headline=True)
    if args.launch_list:
        return head
    result = {"metric": METRIC, "value": head.pop("value"), "unit": UNIT, "n_gpus": world, "steps": args.steps,
              "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"), "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None,
              "dtype": "fp8xfp8, 128x128 block scales (fp32 accumulate)" if args.weights == "bfp8"
              else "fp8xfp4 (fp32 accumulate)",
              "data": "synthetic (seeded, workloads/)"}
    result.update(head)
    torch.cuda.empty_cache()
    if not args.quick and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(wl, bfp8=args.weights == "bfp8")
    if not args.only and args.workload in ALL_WORKLOADS:
        per = {}
        for name in ALL_WORKLOADS:
            if name == args.workload:
                continue
            other = measure(args, W.WORKLOADS[name], dev, stream, world, rank, headline=False)
            if name == "small_decode" and not args.quick and rank == 0 and world == 1:
                other["cpu_baseline"] = cpu_baseline(W.WORKLOADS[name], bfp8=args.weights == "bfp8")
            per[name] = other
            torch.cuda.empty_cache()
        result["per_workload"] = per
    return result


# ---------------------------------------------------------------- CPU oracle

def _spawn_pool():
    import concurrent.futures as cf
    import multiprocessing as mp
    return cf.ProcessPoolExecutor(max_workers=max(1, min(16, len(os.sched_getaffinity(0)))),
                                  mp_context=mp.get_context("spawn"))


def _oracle_weights(wl, experts, bfp8):
    """The oracle's quantised weights of `experts` (untimed set-up), in arrays
    over all E experts (untouched experts stay zero, never read)."""
    import numpy as np
    import torch

    import workloads as W
    from oracle import bfp8 as OB
    from oracle import moe as O
    E, H, I = wl.E, wl.H, wl.I
    if bfp8:
        quant = OB.quantize_weight
        w = [np.zeros((E, 2 * I, H), np.uint8), np.zeros((E, 2 * I // 128, H // 128), np.float32),
             np.zeros((E, H, I), np.uint8), np.zeros((E, H // 128, I // 128), np.float32)]
    else:
        quant = O.quantize_weight
        w = [np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // 32), np.uint8),
             np.zeros((E, H, I // 2), np.uint8), np.zeros((E, H, I // 32), np.uint8)]
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)[None]  # noqa: E731
    big = len(experts) > 2 and 3 * H * I > (1 << 22)
    pool = _spawn_pool() if big else None
    try:
        jobs = []
        for e in experts:
            l1, l2 = W.expert_weights(wl, e, "cpu")
            if pool:
                jobs.append((e, pool.submit(quant, bits(l1)), pool.submit(quant, bits(l2))))
            else:
                jobs.append((e, quant(bits(l1)), quant(bits(l2))))
        for e, r1, r2 in jobs:
            (q1, s1), (q2, s2) = (r1.result(), r2.result()) if pool else (r1, r2)
            w[0][e], w[1][e], w[2][e], w[3][e] = q1[0], s1[0], q2[0], s2[0]
    finally:
        if pool:
            pool.shutdown()
    return w


def _oracle_sample(wl, n_tokens, bfp8):
    """The first `n_tokens` tokens of the workload and the oracle-quantised
    weights of the experts they route to."""
    import numpy as np
    import torch

    import workloads as W
    from oracle import moe as O
    x, logits = W.tokens(wl)
    idx, _ = O.route_topk(logits[:n_tokens].numpy(), wl.k)
    need = sorted(set(idx.reshape(-1).tolist()))
    xb = x[:n_tokens].view(torch.int16).numpy().view(np.uint16)
    return xb, logits[:n_tokens].numpy(), _oracle_weights(wl, need, bfp8), bfp8


def _oracle_tokens_step(wl, sample):
    """One step of the CPU baseline: the oracle's whole layer on the sample's tokens."""
    from oracle import bfp8 as OB
    from oracle import moe as O
    xb, lg, w, bfp8 = sample
    (OB if bfp8 else O).forward(xb, lg, *w, wl.k)


def _heavy(wl):
    """Per-token oracle cost is tens of seconds: sample pairs, not tokens."""
    return 3 * wl.H * wl.I > (1 << 24)


def cpu_baseline(wl, bfp8=False, steps=None):
    """The oracle timed on this host's cores (BLAS threads: all of them) on a
    bounded sample of the workload: every token for the small workloads,
    one token (its k experts) for the large ones."""
    n_tokens = 1 if _heavy(wl) else wl.T
    steps = steps or (1 if _heavy(wl) else 2)
    sample = _oracle_sample(wl, n_tokens, bfp8)
    if not _heavy(wl):
        _oracle_tokens_step(wl, sample)            # warm-up
    t0 = time.time()
    for _ in range(steps):
        _oracle_tokens_step(wl, sample)
    dt = (time.time() - t0) / steps
    what = "block-FP8 oracle" if bfp8 else "oracle"
    full = "all" if n_tokens == wl.T else f"the first {n_tokens}"
    return {"value": round(n_tokens / dt, 4), "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{full} token(s) of {wl.describe()} ({n_tokens * wl.k} pairs) per step through the "
                      f"float64 NumPy {what}'s whole layer (weights of the experts they route to quantised "
                      f"untimed), {steps} step(s), {dt:.2f} s per step"}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on this host's cores.
    Small workloads: one token through the oracle's whole layer per step.
    Large workloads (a token costs tens of seconds): one (token, slot) pair per
    step through the oracle's expert GEMMs (GEMM1 + SwiGLU + requantisation +
    GEMM2), i.e. 1/k token of work, with the token's cast and routing done
    once, untimed (microseconds at one token)."""
    import numpy as np

    import workloads as W
    from oracle import bfp8 as OB
    from oracle import moe as O
    wl = W.WORKLOADS.get(args.workload) or W.PROFILE_WORKLOADS[args.workload]
    bfp8 = args.weights == "bfp8"
    M = OB if bfp8 else O
    if _heavy(wl):
        x, logits = W.tokens(wl)
        import torch
        xb = x[:1].view(torch.int16).numpy().view(np.uint16)
        idx, w = M.route_topk(logits[:1].numpy(), wl.k)
        e = int(idx[0, 0])
        one = np.full_like(idx, -1)
        one[0, 0] = e
        weights = _oracle_weights(wl, [e], bfp8)
        xq, xs = M.quantize_act(xb)

        def step():
            M.expert_forward(xq, xs, *weights, one, w, wl.E, experts=[e])
        tokens_per_step = 1.0 / wl.k
        sample_txt = (f"one (token, slot) pair of {wl.describe()} per step (1/{wl.k} token): the float64 NumPy "
                      f"{'block-FP8 ' if bfp8 else ''}oracle's expert GEMMs for that pair (expert {e}); weights "
                      f"quantised, token cast and routed once, untimed")
    else:
        sample = _oracle_sample(wl, 1, bfp8)

        def step():
            _oracle_tokens_step(wl, sample)
        tokens_per_step = 1.0
        sample_txt = (f"one token of {wl.describe()} per step through the float64 NumPy "
                      f"{'block-FP8 ' if bfp8 else ''}oracle's whole layer (weights of its experts quantised "
                      f"untimed)")
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.time()
        step()
        times.append(time.time() - t0)
    total = sum(times)
    value = tokens_per_step * args.steps / total
    cores = len(os.sched_getaffinity(0))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, workloads/)",
            "config": {"workload": wl.describe() + (" block-FP8 weights" if bfp8 else ""),
                       "tokens_per_step": tokens_per_step, "weights": args.weights},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample_txt},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def pair_tiles(T, H, I, E, k):
    """Large problems whose GEMMs run on CTA pairs (208-token tiles; csrc/gemm2sm.cu)."""
    P = T * k
    if 1 <= T <= 64 and E <= 256 and P * H <= (4 << 20):
        return False                           # small-problem front kernel
    ne = min(E, P)
    return -(-P // ne) > 64 and (2 * I // 128) % 2 == 0 and (H // 128) % 2 == 0


def single_gemm_launch(T, H, I, E, k, schedule=0):
    """Whether the layer's GEMMs (and the combine) are one launch: small
    problems with 16-token tiles, or CTA-pair problems under the expert-wave
    schedule (moe_forward's `schedule` = 2)."""
    P = T * k
    if 1 <= T <= 64 and E <= 256 and P * H <= (4 << 20):
        return -(-P // min(E, P)) <= 16        # 16-token tiles after the front kernel
    return schedule == 2 and pair_tiles(T, H, I, E, k)


def launches_per_forward(T, H, I, E, k, schedule=0):
    """Kernels one moe_forward launches (the dispatch in csrc/api.cu)."""
    P = T * k
    permute = 1 if P <= 2048 else 2            # single-block permute, or count + scatter
    if 1 <= T <= 64 and E <= 256 and P * H <= (4 << 20):
        ne = min(E, P)
        if -(-P // ne) <= 16:                  # 16-token tiles
            return 2                           # front (route + permute + pool cast), GEMM1 + GEMM2 + combine
        return 4                               # front, GEMM1, GEMM2, combine
    cast = 1                                   # pool-order cast, or token-order cast (P*H > 16M)
    if single_gemm_launch(T, H, I, E, k, schedule):
        return 1 + permute + cast + 1          # route, permute, cast, GEMM1 + GEMM2 + combine
    return 1 + permute + cast + 3              # route, permute, cast, GEMM1, GEMM2, combine


def launches_per_forward_bfp8(T, H, E, k):
    """Kernels one moe_forward_bfp8 launches (csrc/bfp8.cu): small problems the
    front (routing + permute + pool cast) and one launch of GEMM1 + GEMM2 +
    combine; otherwise routing, permute, pool cast, GEMM1, GEMM2, combine."""
    P = T * k
    if 1 <= T <= 64 and E <= 256 and P * H <= (4 << 20):
        return 2
    permute = 1 if P <= 2048 else 2
    return 1 + permute + 1 + 3


def main():
    args = parse()
    if args.launch_list:
        args.no_flush = True
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    import __graft_entry__
    __graft_entry__.build()
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
