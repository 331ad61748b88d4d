#!/usr/bin/env python3
"""Benchmark of the KV-cache compression hot path on GB300.

One step = one pass of every hot-path row over one batch of synthetic input,
all inputs resident in HBM when the timed region starts:
  KIVI INT4 workload (batch 8, 8 KV heads, T 8192, head_dim 128, bf16):
    quantize K (per channel, groups of 64 tokens) and V (per token, groups of
    64 channels), asymmetric [0, 15], bf16 scale + zero, 128-token bf16
    residual window; dequantize both; error statistics of both;
  eviction workload (32 heads, history fp32 [64 steps, T 131072], B 2048,
    W 128): H2O select + compaction of K and V, SnapKV select (mean of the
    last 32 steps) + compaction of K and V.
The L2 is flushed (a 2x-L2 buffer is written) before every step, outside the
CUDA-event interval that times the step; the step's phases run back to back
(each also bracketed by events, for the per-phase breakdown).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line (rank 0).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV quant+dequant GB/s & % of GB300 HBM peak; H2O select+compact tokens/s"
UNIT = "GB/s"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# workload constants
KIVI = dict(batch=8, heads=8, T=8192, D=128, g=64, R=128)
EVICT = dict(heads=32, steps=64, T=131072, D=128, budget=2048, window=128, obs=32)
WORKLOAD_NAME = ("kivi_int4[b8,h8,T8192,d128,g64,R128] + h2o/snapkv[h32,S64,T131072,d128,B2048,W128,obs32]")
# Rows timed beside the step (their own events and rooflines; not in `value`):
# the largest quantize / dequantize workloads
FULLMODEL = dict(layers=32, T=8192, heads=32, D=128)
SWEEP = dict(batch=16, heads=8, T=32768, D=128)
EXTRA_ROWS_NAME = ("rows: fullmodel_int8_per_channel[L32,T8192,H32,d128] K+V quantize/dequantize/error_stats; "
                   "sweep_sym[b16,h8,T32768,d128] K+V int4 and int2 g64 per token quantize/dequantize")


# ---------------------------------------------------------------- algorithmic bytes

def kivi_bytes():
    """Per step, K and V together (read + write bytes the method must move)."""
    outer, T, D, g, R = KIVI["batch"] * KIVI["heads"], KIVI["T"], KIVI["D"], KIVI["g"], KIVI["R"]
    Tq = T - R
    x = outer * T * D * 2
    codes = outer * Tq * D // 2
    meta = (outer * (Tq // g) * D) * 2 * 2          # K: bf16 scale + zero per (group, channel)
    meta_v = (outer * Tq * (D // g)) * 2 * 2        # V: per (token, group)
    resid = outer * R * D * 2
    quant = x * 2 + codes * 2 + meta + meta_v + resid * 2
    dequant = quant                                                           # reverse direction
    stats = x * 2 + codes * 2 + meta + meta_v                                 # residual error is zero: not read
    return dict(quantize=quant, dequantize=dequant, error_stats=stats)


def evict_bytes():
    H, S, T, D, B, obs = (EVICT[k] for k in ("heads", "steps", "T", "D", "budget", "obs"))
    keep = H * B * 4
    compact = 2 * (2 * H * B * D * 2)                 # K and V: read kept rows + write them
    return dict(h2o_select=H * S * T * 4 + keep, h2o_compact=compact,
                snapkv_select=H * obs * T * 4 + keep, snapkv_compact=compact)


# ---------------------------------------------------------------- helpers

def rank_seed_offset(rank: int) -> int:
    """Seed offset of a rank's synthetic inputs: rank 0 keeps the workload's
    own seeds, every other rank draws a batch of its own."""
    return 1000 * rank


def reduce_max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank value over all ranks (the timing rule: the slowest
    rank decides); a no-op for one rank.  Uses the default process group."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: float, step_ms: float, world: int) -> float:
    """Whole-job throughput: every rank moved bytes_per_rank_step in step_ms."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources of the dominant call's kernels (colsum_bin1_kernel and
# gather_finish_kernel): a change to either invalidates its ncu traffic.
DOMINANT_SOURCES = ("select.cu", "kvq_device.cuh")


def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_quantization_kvq_gb300", "csrc")
    for f in DOMINANT_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the dominant call, from the committed ncu
    summary, if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("source_digest") == source_digest():
            return d.get("traffic_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
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
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the GPU step

class Step:
    """Device buffers and the launches of one step, through the C ABI."""

    def __init__(self, b, dev, stream, only="all", rank=0):
        import torch
        from kv_cache_quantization_kvq_gb300 import workloads as W
        self.b, self.dev, self.stream = b, dev, stream
        outer = KIVI["batch"] * KIVI["heads"]
        self.kshape = (outer, KIVI["T"], KIVI["D"])
        self.seed_off = rank_seed_offset(rank)     # every rank its own synthetic batch (weak scaling)
        if only in ("all", "kivi"):
            self._init_kivi(b, dev, W)
        if only in ("all", "evict"):
            self._init_evict(b, dev, W)
        torch.cuda.synchronize()

    def _init_kivi(self, b, dev, W):
        import torch
        self.K, self.V = W.kivi_kv(dev, seed=2 + self.seed_off, batch=KIVI["batch"], heads=KIVI["heads"], T=KIVI["T"], D=KIVI["D"])
        self.qpK = b.QParams.asym(4, 0, 15, axis=b.ALONG_T, group=KIVI["g"], residual=KIVI["R"],
                                  scale_dtype=b.BF16, zero_dtype=b.BF16)
        self.qpV = b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=KIVI["g"], residual=KIVI["R"],
                                  scale_dtype=b.BF16, zero_dtype=b.BF16)
        self.qK, self.wsK = b.alloc_quantized(self.kshape, b.BF16, self.qpK, dev)
        self.qV, self.wsV = b.alloc_quantized(self.kshape, b.BF16, self.qpV, dev)
        self.dK = torch.empty_like(self.K)
        self.dV = torch.empty_like(self.V)
        self.stK = torch.zeros(3, dtype=torch.float64, device=dev)
        self.stV = torch.zeros(3, dtype=torch.float64, device=dev)

    def _init_evict(self, b, dev, W):
        import torch
        H, S, T, D = EVICT["heads"], EVICT["steps"], EVICT["T"], EVICT["D"]
        self.hist, self.EK, self.EV = W.eviction_inputs(dev, seed=5 + self.seed_off, heads=H, steps=S, T=T, D=D,
                                                        window=EVICT["window"])
        self.keep = torch.empty((H, EVICT["budget"]), dtype=torch.int32, device=dev)
        self.skeep = torch.empty_like(self.keep)
        self.selB = b.kv_select_workspace(H, T)
        self.sel_ws = torch.empty(self.selB, dtype=torch.uint8, device=dev)
        self.sel_ws2 = torch.empty(self.selB, dtype=torch.uint8, device=dev)    # SnapKV's own
        self.cK = torch.empty((H, EVICT["budget"], D), dtype=torch.bfloat16, device=dev)
        self.cV = torch.empty_like(self.cK)
        self.scK = torch.empty_like(self.cK)
        self.scV = torch.empty_like(self.cK)

    # each phase returns the number of kernels it launched
    def quantize(self):
        b, s = self.b, self.stream
        b.kvq_quantize(self.K, b.BF16, self.kshape, self.qpK, self.qK.codes, self.qK.scale, self.qK.zero,
                       self.qK.resid, self.wsK, self.wsK.numel(), s)
        b.kvq_quantize(self.V, b.BF16, self.kshape, self.qpV, self.qV.codes, self.qV.scale, self.qV.zero,
                       self.qV.resid, self.wsV, self.wsV.numel(), s)
        return 2

    def dequantize(self):
        b, s = self.b, self.stream
        b.kvq_dequantize(self.qK.codes, self.qK.scale, self.qK.zero, self.qK.resid, self.kshape, self.qpK,
                         self.dK, b.BF16, s)
        b.kvq_dequantize(self.qV.codes, self.qV.scale, self.qV.zero, self.qV.resid, self.kshape, self.qpV,
                         self.dV, b.BF16, s)
        return 2

    def error_stats(self):
        b, s = self.b, self.stream
        b.kvq_error_stats(self.K, b.BF16, self.qK.codes, self.qK.scale, self.qK.zero, self.qK.resid,
                          self.kshape, self.qpK, self.stK, self.wsK, self.wsK.numel(), s)
        b.kvq_error_stats(self.V, b.BF16, self.qV.codes, self.qV.scale, self.qV.zero, self.qV.resid,
                          self.kshape, self.qpV, self.stV, self.wsV, self.wsV.numel(), s)
        return 4          # two stats kernels + two finalize kernels

    def h2o_select(self):
        b, H, S, T = self.b, EVICT["heads"], EVICT["steps"], EVICT["T"]
        b.kv_h2o_select(self.hist, H, S, T, EVICT["budget"], EVICT["window"], self.keep, None, self.sel_ws,
                        self.selB, self.stream)
        return 3          # column sums + candidate gather + finish (plus two memsets)

    def h2o_compact(self):
        b, H, T, D = self.b, EVICT["heads"], EVICT["T"], EVICT["D"]
        b.kv_compact_kv(self.EK, self.EV, b.BF16, H, T, D, self.keep, EVICT["budget"], self.cK, self.cV, self.stream)
        return 1

    def snapkv_select(self):
        b, H, S, T = self.b, EVICT["heads"], EVICT["steps"], EVICT["T"]
        b.kv_snapkv_select(self.hist, H, S, T, EVICT["obs"], EVICT["budget"], EVICT["window"], self.skeep, None,
                           self.sel_ws2, self.selB, self.stream)
        return 3

    def snapkv_compact(self):
        b, H, T, D = self.b, EVICT["heads"], EVICT["T"], EVICT["D"]
        b.kv_compact_kv(self.EK, self.EV, b.BF16, H, T, D, self.skeep, EVICT["budget"], self.scK, self.scV,
                        self.stream)
        return 1

    PHASES = ("quantize", "dequantize", "error_stats", "h2o_select", "h2o_compact", "snapkv_select",
              "snapkv_compact")


def run_ours(args, rank, world, local_rank):
    import torch
    from kv_cache_quantization_kvq_gb300 import build as build_lib
    build_lib()
    from kv_cache_quantization_kvq_gb300 import binding as b

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    if args.only == "attend":
        # the fused decode-attention rows alone (profiling)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        return {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "data": "synthetic",
                "config": {"workload": "kivi_int4 decode attention [b8,h8,T8192,d128,g64,R128]", "only": "attend"},
                "configs": run_configs(b, dev, stream, flush, only_attend=True)}
    if args.only == "mixed":
        # the mixed-precision rows alone (profiling)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        return {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "data": "synthetic",
                "config": {"workload": "kivi_int4 keys, per-token mixed precision [b8,h8,T8192,d128]", "only": "mixed"},
                "configs": run_configs(b, dev, stream, flush, only_mixed=True)}
    if args.only == "rotate":
        # the rotation rows alone (profiling)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        return {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "data": "synthetic",
                "config": {"workload": "kivi_int4 rotation [b8,h8,T8192,d128]", "only": "rotate"},
                "configs": run_configs(b, dev, stream, flush, only_rotate=True)}
    if args.only == "fullmodel":
        # the full-model INT8 rows alone (profiling; --fullmodel-layers shrinks the case)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        return {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "data": "synthetic",
                "config": {"workload": f"fullmodel_int8[L{args.fullmodel_layers},T8192,H32,d128]", "only": "fullmodel"},
                "configs": run_configs(b, dev, stream, flush, only_fullmodel=True, layers=args.fullmodel_layers)}
    with torch.cuda.stream(stream):
        st = Step(b, dev, stream, args.only, rank)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    kb, eb = kivi_bytes(), evict_bytes()
    pbytes = {**kb, **eb}
    phases = [ph for ph in Step.PHASES
              if args.only == "all" or (args.only == "kivi") == (ph in kb)]
    pbytes = {ph: pbytes[ph] for ph in phases}

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            for ph in phases:
                getattr(st, ph)()
    barrier()

    # Per-phase breakdown (not the headline): every phase bracketed by events,
    # the L2 flushed (a 2x-L2 buffer written) before every step.
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    Kb = max(3, min(args.steps, 200))
    ev = {ph: [mk() for _ in range(Kb)] for ph in phases}
    with torch.cuda.stream(stream):
        for i in range(Kb):
            flush.zero_()
            for ph in phases:
                a, z = ev[ph][i]
                a.record(stream)
                getattr(st, ph)()
                z.record(stream)
    torch.cuda.synchronize()
    ph_ms = {ph: statistics.fmean(a.elapsed_time(z) for a, z in ev[ph]) for ph in phases}

    # The step as one sequence: captured once as a CUDA graph (the same C-ABI
    # calls, recorded on the stream) unless --no-graph; launches counted once.
    per_step = 0
    graph = None
    # independent chains of rows (they share no buffer): KIVI, H2O, SnapKV
    chains = [c for c in ([ph for ph in phases if ph in kivi_bytes()],
                          [ph for ph in phases if ph.startswith("h2o")],
                          [ph for ph in phases if ph.startswith("snapkv")]) if c]
    overlap = (not args.serial_rows) and len(chains) > 1

    def capture(branches):
        nonlocal per_step
        per_step = 0
        g = torch.cuda.CUDAGraph()
        sides = [torch.cuda.Stream(device=dev) for _ in chains[1:]]
        with torch.cuda.graph(g, stream=stream):
            if branches:
                # one branch of the graph per chain, joined at the end of the step
                fork = torch.cuda.Event()
                fork.record(stream)
                for sd in sides:
                    sd.wait_event(fork)
                for chain, sd in zip(chains, [stream] + sides):
                    st.stream = sd
                    for ph in chain:
                        per_step += getattr(st, ph)()
                st.stream = stream
                for sd in sides:
                    join = torch.cuda.Event()
                    join.record(sd)
                    stream.wait_event(join)
            else:
                for ph in phases:
                    per_step += getattr(st, ph)()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize()
        return g

    def time_graph(g, n):
        evs = [mk() for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                flush.zero_()
                evs[i][0].record(stream)
                g.replay()
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.fmean(a.elapsed_time(z) for a, z in evs)

    serial_ms = None
    if not args.no_graph:
        if overlap:          # the rows in sequence, for reference (not the headline)
            serial_ms = time_graph(capture(False), max(3, min(args.steps, 200)))
        graph = capture(overlap)

    # Timed region: K steps; before each, the L2 is flushed outside the step's
    # event interval; the step replays the graph (the KIVI, H2O and SnapKV
    # rows as concurrent branches unless --serial-rows).  The K steps are
    # repeated (each repeat bracketed by a barrier and a synchronize) until
    # about --min-timed-seconds of steps have run; ms_per_step is the median
    # repeat's mean step time, so the number rests on many clock samples.
    K = args.steps
    launches = 0
    rep_ms = []
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        while True:
            ev_step = [mk() for _ in range(K)]
            barrier()
            with torch.cuda.stream(stream):
                for i in range(K):
                    flush.zero_()
                    ev_step[i][0].record(stream)
                    if graph is not None:
                        graph.replay()
                        launches += per_step
                    else:
                        for ph in phases:
                            launches += getattr(st, ph)()
                    ev_step[i][1].record(stream)
            barrier()
            rep_ms.append(statistics.fmean(a.elapsed_time(z) for a, z in ev_step))
            timed_s = sum(rep_ms) * K * 1e-3
            if len(rep_ms) >= args.max_repeats or (len(rep_ms) >= 3 and timed_s >= args.min_timed_seconds):
                break
        wall = time.perf_counter() - t0
    step_ms = reduce_max_over_ranks(statistics.median(rep_ms), world, dev)
    total_bytes = sum(pbytes.values())
    value = whole_job_gbs(total_bytes, step_ms, world)

    # sanity of the step's outputs (not timed): finite statistics
    torch.cuda.synchronize()
    if "error_stats" in phases:
        assert torch.isfinite(st.stK).all() and torch.isfinite(st.stV).all()

    result = None
    if rank == 0:
        peak, peak_kind = measured_peak()
        h2o_ms = ph_ms.get("h2o_select", float("nan")) + ph_ms.get("h2o_compact", float("nan"))
        tokens = EVICT["heads"] * EVICT["T"]
        sel_B = evict_bytes()["h2o_select"]
        sel_gbs = sel_B / (ph_ms["h2o_select"] * 1e-3) / 1e9 if "h2o_select" in ph_ms else None
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f32 in, int4 codes; f32 arithmetic",
            "data": "synthetic (seeded generators; shapes and distributions of the pages' workloads)",
            "config": {"workload": WORKLOAD_NAME,
                       "l2": "flushed (2x L2 written) before every step, outside the timed interval",
                       "inputs_resident_in_hbm": True, "parallelism": f"weak: {world} independent replica(s)",
                       "launch": ("CUDA graph of the step's C-ABI calls" if graph is not None else "C-ABI calls") +
                                 ("; the KIVI, H2O and SnapKV rows as concurrent branches" if graph is not None and overlap else "")},
            "hbm_frac_of_8TBs": round(value / world / SPEC_HBM_GBS, 4),
            "hbm_frac_of_measured": round(value / world / peak, 4),
            "h2o_tokens_per_s": round(world * tokens / (h2o_ms * 1e-3), 1) if h2o_ms == h2o_ms else None,
            "phases": {ph: {"ms": round(ph_ms[ph], 5), "GB/s": round(pbytes[ph] / (ph_ms[ph] * 1e-3) / 1e9, 1),
                            "bytes": pbytes[ph]} for ph in phases},
            "roofline": {"kernel": "kv_h2o_select (colsum_bin1_kernel + gather_finish_kernel)",
                         "bound": "hbm", "achieved": round(sel_gbs, 1) if sel_gbs else None, "peak": peak,
                         "unit": "GB/s", "frac": round(sel_gbs / peak, 4) if sel_gbs else None,
                         "peak_kind": f"of {peak_kind}",
                         "bytes_per_launch": sel_B, "traffic": ncu_traffic()},
            "ms_per_step_rows_in_sequence": round(serial_ms, 5) if serial_ms else None,
            "gpu_launches": launches,                    # all repeats of the timed region
            "gpu_launches_per_step": launches // max(1, K * len(rep_ms)),
            "timed_repeats": {"repeats": len(rep_ms), "steps_each": K,
                              "ms_per_step_min": round(min(rep_ms), 5),
                              "ms_per_step_median": round(statistics.median(rep_ms), 5),
                              "ms_per_step_max": round(max(rep_ms), 5),
                              "timed_s": round(sum(rep_ms) * K * 1e-3, 3)},
            "wall_s_timed_region": round(wall, 3),
            "clocks": clk.summary(),
        }
        if args.only == "all" and not args.no_extra_rows:
            # the largest quantize / dequantize workloads, each op its own row
            rows, rclk = run_extra_rows(b, dev, stream, flush, peak, runs=max(5, min(args.steps, 50)))
            result["phases"].update(rows)
            result["config"]["workload"] = WORKLOAD_NAME + "; " + EXTRA_ROWS_NAME
            result["clocks"] = {**result["clocks"], "extra_rows": rclk}
        result["wait_timeouts"] = b.kvq_wait_timeouts()    # bounded waits that gave up in this process: 0
        if args.only != "all":
            result["config"]["only"] = args.only
        if args.evict_tokens is not None:
            result["config"]["evict_tokens"] = args.evict_tokens
        if not args.no_e2e and args.only == "all":
            result["e2e"] = run_e2e(b, st, stream, dev, args, total_bytes, world)
        if not args.no_cpu_baseline and world == 1:
            result["cpu_baseline"] = cpu_baseline(min_seconds=args.cpu_seconds)
            try:                              # informational; keep the contract line whatever happens
                result["cpu_baseline_all_cores"] = cpu_baseline_all_cores(min_seconds=args.cpu_seconds)
            except Exception as exc:
                result["cpu_baseline_all_cores"] = {"error": f"{type(exc).__name__}: {exc}"}
        if args.configs:
            try:
                result["configs"] = run_configs(b, dev, stream, flush)
            except Exception as exc:          # the table is informational; keep the contract line
                result["configs"] = {"error": f"{type(exc).__name__}: {exc}"}
    return result


# ---------------------------------------------------------------- per-config table

def quant_bytes(shape, x_es, cB, sB, zB, rB):
    """Algorithmic bytes of one quantize (read x, write codes + metadata +
    residual) -- the same total for dequantize, reversed -- and of one
    error-statistics pass (read x + codes + metadata; the residual's error is
    zero by construction)."""
    outer, T, C = shape
    x = outer * T * C * x_es
    return x + cB + sB + zB + rB, x + cB + sB + zB


def run_configs(b, dev, stream, flush, runs=20, only_fullmodel=False, layers=32, only_attend=False,
                only_rotate=False, only_mixed=False):
    """Median over `runs` (L2 flushed before each) of every op of the large
    configurations: KIVI INT4 (2), full-model INT8 per channel (3), the
    group / bit-width sweep (4), H2O / SnapKV (5); the tiny one (1) in us.
    only_fullmodel: the full-model rows alone, with `layers` layers;
    only_attend: the fused decode attention over the KIVI cache alone;
    only_rotate: the rotation rows (stand-alone, and fused into the value
    cache's quantize / dequantize) alone; only_mixed: the per-token mixed
    precision rows alone."""
    import torch
    from kv_cache_quantization_kvq_gb300 import workloads as W
    peak, _ = measured_peak()
    out = {}

    def med(fn):
        ts = []
        with torch.cuda.stream(stream):
            fn()
            for _ in range(runs):
                flush.zero_()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                z.record(stream)
                ts.append((a, z))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(z) for a, z in ts)

    def entry(ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac_of_8TBs": round(gbs / SPEC_HBM_GBS, 3),
                "frac_of_measured": round(gbs / peak, 3), "bytes": nbytes}

    def qdq(tag, named, qp, stats=True):
        shape = tuple(named[0][1].shape)
        for name, x in named:
            qt, ws = b.alloc_quantized(shape, b.BF16, qp, dev)
            cB, sB, zB, rB = (t.numel() for t in (qt.codes, qt.scale, qt.zero, qt.resid))
            qb, sb = quant_bytes(shape, 2, cB, sB, zB, rB)
            outx = torch.empty_like(x)
            e = torch.zeros(3, dtype=torch.float64, device=dev)
            q_ms = med(lambda: b.quantize(x, qp, out=qt, workspace=ws, stream=stream))
            d_ms = med(lambda: b.dequantize(qt, out=outx, stream=stream))
            out[f"{tag}/{name}/quantize"] = entry(q_ms, qb)
            out[f"{tag}/{name}/dequantize"] = entry(d_ms, qb)
            if stats:
                s_ms = med(lambda: b.error_stats(x, qt, workspace=ws, stream=stream, out_dev=e))
                out[f"{tag}/{name}/error_stats"] = entry(s_ms, sb)
            out[f"{tag}/{name}/bytes_per_number"] = round((cB + sB) / (shape[0] * shape[1] * shape[2]), 6)
            del qt, ws, outx

    if only_fullmodel:
        K, V = W.fullmodel_kv(dev, seed=3, layers=layers)
        qdq(f"3_fullmodel_int8_L{layers}", [("K", K), ("V", V)], b.QParams.sym(8, axis=b.ALONG_T, group=0))
        return out
    # 2: KIVI INT4
    K, V = W.kivi_kv(dev, seed=2)

    def rotate_rows():
        # randomized Hadamard rotation of the key cache (bf16 -> bf16): read + write
        signs = torch.where(torch.rand(K.shape[-1], device=dev, generator=torch.Generator(device=dev).manual_seed(3)) < 0.5,
                            -1, 1).to(torch.int8)
        rot = torch.empty_like(K)
        out["2_kivi_int4/K/rotate"] = entry(med(lambda: b.rotate(K, signs, out=rot, stream=stream)), 2 * K.numel() * 2)
        # the rotation fused into the value cache's per-token quantize and dequantize
        # (the KIVI value format): the same bytes as the plain quantize / dequantize
        vqf = b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
        qvf, _ = b.alloc_quantized(tuple(V.shape), b.BF16, vqf, dev)
        fq_B, _ = quant_bytes(tuple(V.shape), 2, *(t.numel() for t in (qvf.codes, qvf.scale, qvf.zero, qvf.resid)))
        vout = torch.empty_like(V)
        out["2_kivi_int4/V/rotate_quantize"] = entry(med(lambda: b.rotate_quantize(V, signs, vqf, out=qvf, stream=stream)),
                                                     fq_B)
        out["2_kivi_int4/V/dequantize_rotate"] = entry(med(lambda: b.dequantize_rotate(qvf, signs, out=vout, stream=stream)),
                                                       fq_B)
        del rot, qvf, vout

    def mixed_rows():
        # per-token mixed precision of the key cache, the four levels in equal shares
        # (seeded tags): quantize reads K and writes the records, dequantize the reverse
        shp = tuple(K.shape)
        tags = torch.randint(0, 4, shp[:2], dtype=torch.uint8, device=dev, generator=torch.Generator(device=dev).manual_seed(4))
        sB, oB, tB = b.kvq_mixed_sizes(shp)
        mbuf = torch.empty(sB, dtype=torch.uint8, device=dev)
        moff = torch.empty(oB // 8, dtype=torch.int64, device=dev)
        mt2 = torch.empty(tB, dtype=torch.uint8, device=dev)
        mout = torch.empty_like(K)
        b.kvq_mixed_quantize(K, tags, shp, mbuf, moff, mt2, stream)
        torch.cuda.synchronize()
        used = int(moff.view(shp[0], shp[1] + 1)[:, -1].sum().item())      # record bytes of all slices
        mq_B = K.numel() * 2 + tags.numel() + used + oB + tB
        out["2_kivi_int4/K/mixed_quantize"] = entry(med(lambda: b.kvq_mixed_quantize(K, tags, shp, mbuf, moff, mt2, stream)), mq_B)
        out["2_kivi_int4/K/mixed_dequantize"] = entry(med(lambda: b.kvq_mixed_dequantize(mbuf, moff, mt2, shp, mout, stream)),
                                                      used + oB + tB + K.numel() * 2)
        out["2_kivi_int4/K/mixed_bytes_per_number"] = round((used + tB) / K.numel(), 6)
        del mbuf, moff, mt2, mout, tags

    if only_rotate:
        rotate_rows()
        return out
    if only_mixed:
        mixed_rows()
        return out
    if not only_attend:
        for axis, x, name in ((b.ALONG_T, K, "K"), (b.ALONG_C, V, "V")):
            qp = b.QParams.asym(4, 0, 15, axis=axis, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
            qdq("2_kivi_int4", [(name, x)], qp)
    # decode attention over the quantized KIVI cache (dequantization fused):
    # bytes = the quantized K and V caches read + queries + outputs + split partials
    kq = b.QParams.asym(4, 0, 15, axis=b.ALONG_T, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    vq = b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    qk, qv = b.quantize(K, kq, stream=stream), b.quantize(V, vq, stream=stream)
    torch.cuda.synchronize()
    cache_B = sum(t.numel() for t in (qk.codes, qk.scale, qk.zero, qk.resid, qv.codes, qv.scale, qv.zero, qv.resid))
    outer = K.shape[0]
    for G in (1, 4, 8):
        q = torch.randn((outer, G, K.shape[2]), device=dev, generator=torch.Generator(device=dev).manual_seed(G))
        o = torch.empty_like(q)
        ws = torch.empty(b.kvq_attend_workspace(tuple(K.shape), G), dtype=torch.uint8, device=dev)
        ms = med(lambda: b.attend_decode(q, qk, qv, out=o, workspace=ws, stream=stream))
        out[f"2_kivi_int4/attend_decode_G{G}"] = entry(ms, cache_B + 2 * q.numel() * 4 + 2 * ws.numel())
    del qk, qv
    if only_attend:
        return out
    # streaming append: 64 decode steps of one token into the KIVI key and value
    # caches of one layer (block 64: the 32nd step flushes one block of 64 tokens
    # of each cache), one kvq_append_kv call per step, microseconds per step
    kq_s = b.QParams.asym(4, 0, 15, axis=b.ALONG_T, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    vq_s = b.QParams.asym(4, 0, 15, axis=b.ALONG_C, group=64, residual=128, scale_dtype=b.BF16, zero_dtype=b.BF16)
    cap_shape = (K.shape[0], K.shape[1], K.shape[2])
    stores = {}
    for name, qp in (("K", kq_s), ("V", vq_s)):
        store_qp = b.QParams(qp.bits, qp.mode, qp.qmin, qp.qmax, qp.axis, qp.group, 0, qp.scale_dtype, qp.zero_dtype)
        cB, sB, zB, _, _ = b.kvq_quantized_sizes(cap_shape, b.BF16, store_qp)
        stores[name] = (torch.empty(cB, dtype=torch.uint8, device=dev), torch.empty(sB, dtype=torch.uint8, device=dev),
                        torch.empty(zB, dtype=torch.uint8, device=dev),
                        torch.empty(K.shape[0] * (128 + 64) * K.shape[2], dtype=torch.bfloat16, device=dev))
    wB = b.kvq_append_kv_workspace(cap_shape, b.BF16, kq_s, vq_s, 64)
    aws = torch.empty(wB, dtype=torch.uint8, device=dev)
    app = b.KVAppender(cap_shape, b.BF16, kq_s, vq_s, 64, stores["K"], stores["V"], aws, stream=stream)
    ksteps = [K[:, i:i + 1].contiguous() for i in range(64)]
    vsteps = [V[:, i:i + 1].contiguous() for i in range(64)]

    def decode_steps():
        app.set_counters(0, 160)                        # 160 of 192 buffered: the 32nd step flushes
        for k1, v1 in zip(ksteps, vsteps):
            app.append(k1, v1, 1)
    ms = med(decode_steps)
    out["2_kivi_int4/append_KV_one_token_us"] = round(1e3 * ms / 64, 2)
    del stores, aws, app, ksteps, vsteps
    mixed_rows()
    rotate_rows()
    del K, V
    # 3: full model INT8, per channel over all tokens
    K, V = W.fullmodel_kv(dev, seed=3)
    qdq("3_fullmodel_int8", [("K", K), ("V", V)], b.QParams.sym(8, axis=b.ALONG_T, group=0))
    del K, V
    # 4: sweep, per token, INT4 / INT2, g in {32, 64, 128}
    K, V = W.sweep_kv(dev, seed=4)
    for bits in (4, 2):
        for g in (32, 64, 128):
            qdq(f"4_sweep_int{bits}_g{g}", [("K", K), ("V", V)],
                b.QParams.sym(bits, axis=b.ALONG_C, group=g, scale_dtype=b.BF16), stats=False)
    del K, V
    torch.cuda.empty_cache()
    # 1: tiny (launch-bound: microseconds only)
    x, hist = W.tiny_inputs(0)
    xd = torch.from_numpy(x).reshape(1, 256, 128).to(dev)
    hd = torch.from_numpy(hist).to(dev)
    for qn, qp in (("int8_sym", b.QParams.sym(8, axis=b.ALONG_T, group=0)),
                   ("int8_asym", b.QParams.asym(8, -128, 127, axis=b.ALONG_T, group=0, zero_dtype=b.I8)),
                   ("int4_g32", b.QParams.sym(4, axis=b.ALONG_T, group=32))):
        qt, ws = b.alloc_quantized((1, 256, 128), b.F32, qp, dev)
        o = torch.empty_like(xd)
        e = torch.zeros(3, dtype=torch.float64, device=dev)
        out[f"1_tiny/{qn}/quantize_us"] = round(1e3 * med(lambda: b.quantize(xd, qp, out=qt, workspace=ws, stream=stream)), 2)
        out[f"1_tiny/{qn}/dequantize_us"] = round(1e3 * med(lambda: b.dequantize(qt, out=o, stream=stream)), 2)
        out[f"1_tiny/{qn}/error_stats_us"] = round(1e3 * med(lambda: b.error_stats(xd, qt, workspace=ws, stream=stream, out_dev=e)), 2)
    out["1_tiny/h2o_select_us"] = round(1e3 * med(lambda: b.h2o_select(hd, 64, 16, stream=stream)), 2)
    out["1_tiny/snapkv_select_us"] = round(1e3 * med(lambda: b.snapkv_select(hd, 32, 64, 16, stream=stream)), 2)
    return out


def fullmodel_bytes():
    """Symmetric INT8 per channel over all T, fp32 scale, K and V together:
    quantize reads x and writes codes + scales; dequantize the reverse; the
    statistics read x, codes and scales."""
    L, T, H, D = (FULLMODEL[k] for k in ("layers", "T", "heads", "D"))
    x = 2 * L * T * H * D * 2
    codes = 2 * L * T * H * D
    scales = 2 * L * H * D * 4
    return dict(quantize=x + codes + scales, dequantize=x + codes + scales, error_stats=x + codes + scales)


def sweep_bytes(bits, g):
    """Symmetric per token (groups of g channels), bf16 scale, K and V."""
    n = 2 * SWEEP["batch"] * SWEEP["heads"] * SWEEP["T"] * SWEEP["D"]
    q = n * 2 + n * bits // 8 + (n // g) * 2
    return dict(quantize=q, dequantize=q)


def run_extra_rows(b, dev, stream, flush, peak, runs=20):
    """Full-model INT8 (quantize, dequantize, statistics) and the per-token
    INT4 / INT2 g 64 sweep (quantize, dequantize), K and V inside one event
    pair per op; median of `runs` with the L2 flushed before each.  Returns
    the rows (with bytes and a roofline each) and the clock samples taken
    while they ran."""
    import torch
    from kv_cache_quantization_kvq_gb300 import workloads as W
    rows = {}

    def med(fn):
        ts = []
        with torch.cuda.stream(stream):
            fn()
            for _ in range(runs):
                flush.zero_()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                z.record(stream)
                ts.append((a, z))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(z) for a, z in ts)

    def add(name, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows[name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1), "bytes": nbytes,
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                   "frac": round(gbs / peak, 4)}}

    def qdq(tag, K, V, qp, nbytes, stats):
        shape = tuple(K.shape)
        qk, wk = b.alloc_quantized(shape, b.BF16, qp, dev)
        qv, wv = b.alloc_quantized(shape, b.BF16, qp, dev)
        ok, ov = torch.empty_like(K), torch.empty_like(V)
        ek = torch.zeros(3, dtype=torch.float64, device=dev)
        ev = torch.zeros(3, dtype=torch.float64, device=dev)

        def quant():
            b.quantize(K, qp, out=qk, workspace=wk, stream=stream)
            b.quantize(V, qp, out=qv, workspace=wv, stream=stream)

        def dequant():
            b.dequantize(qk, out=ok, stream=stream)
            b.dequantize(qv, out=ov, stream=stream)

        def errs():
            b.error_stats(K, qk, workspace=wk, stream=stream, out_dev=ek)
            b.error_stats(V, qv, workspace=wv, stream=stream, out_dev=ev)

        add(f"{tag}/quantize", med(quant), nbytes["quantize"])
        add(f"{tag}/dequantize", med(dequant), nbytes["dequantize"])
        if stats:
            add(f"{tag}/error_stats", med(errs), nbytes["error_stats"])
            assert torch.isfinite(ek).all() and torch.isfinite(ev).all()
        del qk, qv, wk, wv, ok, ov

    with ClockSampler(dev.index or 0) as clk:
        K, V = W.fullmodel_kv(dev, seed=3, **FULLMODEL)
        qdq("3_fullmodel_int8", K, V, b.QParams.sym(8, axis=b.ALONG_T, group=0), fullmodel_bytes(), True)
        del K, V
        K, V = W.sweep_kv(dev, seed=4, **SWEEP)
        for bits in (4, 2):
            qdq(f"4_sweep_int{bits}_g64", K, V, b.QParams.sym(bits, axis=b.ALONG_C, group=64, scale_dtype=b.BF16),
                sweep_bytes(bits, 64), False)
        del K, V
        torch.cuda.empty_cache()
    return rows, clk.summary()


def run_e2e(b, st, stream, dev, args, total_bytes, world):
    """Same step through the C ABI with host buffers: pinned host -> device
    copies of every input, the step, device -> host copies of the results."""
    import torch
    ins = [st.K, st.V, st.hist, st.EK, st.EV]
    host_in = [t.cpu().pin_memory() for t in ins]
    outs = [st.qK.codes, st.qK.scale, st.qK.zero, st.qK.resid, st.qV.codes, st.qV.scale, st.qV.zero,
            st.qV.resid, st.stK, st.stV, st.keep, st.skeep, st.cK, st.cV, st.scK, st.scV]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    n = max(3, min(args.steps, args.e2e_steps))

    def one():
        for d, h in zip(ins, host_in):
            d.copy_(h, non_blocking=True)
        for ph in Step.PHASES:
            getattr(st, ph)()
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            one()
        z.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(z) / n
    return {"value": round(world * total_bytes / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}


# ---------------------------------------------------------------- the oracle (CPU)

def oracle_sample(seed=0):
    """One [outer] slice of the KIVI workload and one head of the eviction
    workload, drawn on the host with the same recipes."""
    from kv_cache_quantization_kvq_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    T, D = KIVI["T"], KIVI["D"]
    xk = W.to_bf16_bits(W.random_kv(rng, (1, T, D), 0.02, 8.0))
    xv = W.to_bf16_bits(rng.standard_normal((1, T, D), dtype=np.float32))
    ET = EVICT["T"]
    hist = W.random_history(rng, 1, EVICT["steps"], ET, planted=256, window=EVICT["window"])
    ek = W.to_bf16_bits(rng.standard_normal((1, ET, D), dtype=np.float32))
    ev = W.to_bf16_bits(rng.standard_normal((1, ET, D), dtype=np.float32))
    return xk, xv, hist, ek, ev


def oracle_step(sample):
    import oracle as O
    xk, xv, hist, ek, ev = sample
    qk = O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=KIVI["g"], residual=KIVI["R"], scale_dtype=O.BF16,
                        zero_dtype=O.BF16)
    qv = O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=KIVI["g"], residual=KIVI["R"], scale_dtype=O.BF16,
                        zero_dtype=O.BF16)
    a, c = O.quantize(xk, O.BF16, qk), O.quantize(xv, O.BF16, qv)
    O.dequantize(a, xk.shape, qk, O.BF16)
    O.dequantize(c, xv.shape, qv, O.BF16)
    O.error_stats(xk, O.BF16, a, qk)
    O.error_stats(xv, O.BF16, c, qv)
    keep, _ = O.h2o_select(hist, EVICT["budget"], EVICT["window"])
    O.compact(ek, keep)
    O.compact(ev, keep)
    skeep, _ = O.snapkv_select(hist, EVICT["obs"], EVICT["budget"], EVICT["window"])
    O.compact(ek, skeep)
    O.compact(ev, skeep)
    outer = KIVI["batch"] * KIVI["heads"]
    kb, eb = kivi_bytes(), evict_bytes()
    return sum(kb.values()) / outer + sum(eb.values()) / EVICT["heads"]


SAMPLE_DESC = ("oracle (plain C, 1 thread) on 1 of 64 [batch*head] slices of the KIVI workload "
               "(quantize/dequantize/error stats of K and V) plus 1 of 32 heads of the eviction "
               "workload (H2O + SnapKV select, compaction of K and V); GB/s = the slice's algorithmic bytes / time")


def host_cpu():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = {line.split(":", 1)[0].strip(): line.split(":", 1)[1].strip()
                  for line in out.splitlines() if ":" in line}
        name = " ".join(v for v in (fields.get("Vendor ID"), fields.get("Model name")) if v and v != "-")
        if name:
            return name
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def cpu_baseline(min_seconds=10.0):
    import oracle as O
    O.build()
    sample = oracle_sample(1)
    oracle_step(sample)                     # warm
    done, nbytes, t0 = 0, 0.0, time.perf_counter()
    while True:
        nbytes += oracle_step(sample)
        done += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": round(nbytes / el / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "host_cpu": host_cpu(), "sample": f"{SAMPLE_DESC}; {done} repetitions in {el:.1f} s"}


def _oracle_worker(job):
    """One process of the all-cores oracle baseline: its own KIVI slice and
    eviction head (seed), the same loop as the one-core baseline."""
    seed, seconds = job
    sample = oracle_sample(seed)
    oracle_step(sample)                     # warm
    done, nbytes, t0 = 0, 0.0, time.perf_counter()
    while True:
        nbytes += oracle_step(sample)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return nbytes, el, done


def cpu_baseline_all_cores(min_seconds=10.0, processes=None):
    """The oracle as it stands on every host core: one process per core (spawn
    start, safe after CUDA is initialised), each on independent units -- its
    own KIVI slice and eviction head -- for about min_seconds.  GB/s = the
    algorithmic bytes of all processes / the longest process's loop time."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    import oracle as O
    O.build()
    n = processes or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)
    # a worker that dies raises BrokenProcessPool instead of blocking; every wait is bounded
    ex = ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
    try:
        futs = [ex.submit(_oracle_worker, (100 + i, min_seconds)) for i in range(n)]
        res = [f.result(timeout=10 * min_seconds + 300) for f in futs]
    finally:
        ex.shutdown(wait=False, cancel_futures=True)
    nbytes, el, done = sum(r[0] for r in res), max(r[1] for r in res), sum(r[2] for r in res)
    return {"value": round(nbytes / el / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{n} processes of the one-core sample, each on its own KIVI slice and eviction head; "
                      f"{done} repetitions in {el:.1f} s"}


def run_reference(args):
    import oracle as O
    O.build()
    sample = oracle_sample(1)
    for _ in range(args.warmup):
        oracle_step(sample)
    times, nbytes = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        nbytes += oracle_step(sample)
        times.append(time.perf_counter() - t0)
    el = sum(times)
    value = nbytes / el / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 arithmetic (CPU oracle)",
        "data": "synthetic (seeded generators, host)",
        "config": {"workload": WORKLOAD_NAME, "sample": "one KIVI slice + one eviction head per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": SAMPLE_DESC},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-rows", action="store_true",
                    help="skip the full-model INT8 and g/bit sweep rows timed beside the step")
    ap.add_argument("--min-timed-seconds", type=float, default=1.0,
                    help="repeat the K timed steps until about this much step time has run (at least 3 repeats)")
    ap.add_argument("--max-repeats", type=int, default=400)
    ap.add_argument("--configs", action="store_true",
                    help="add the per-configuration table (tiny, KIVI INT4, full-model INT8, g/bit sweep)")
    ap.add_argument("--serial-rows", action="store_true",
                    help="run the KIVI, H2O and SnapKV rows one after the other instead of as concurrent "
                         "branches of the step graph")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue the timed steps as plain C-ABI calls instead of replaying a captured CUDA graph")
    ap.add_argument("--only", choices=("all", "kivi", "evict", "fullmodel", "attend", "rotate", "mixed"), default="all",
                    help="time only the KIVI phases or only the eviction phases (profiling); "
                         "fullmodel / attend / rotate / mixed: only the full-model INT8 rows / the fused "
                         "decode-attention rows / the rotation rows / the mixed-precision rows of the "
                         "per-configuration table")
    ap.add_argument("--fullmodel-layers", type=int, default=32,
                    help="layers of the full-model INT8 workload with --only fullmodel (a smaller profiling case)")
    ap.add_argument("--evict-tokens", type=int, default=None,
                    help="context length T of the eviction workload (profiling of a smaller case; "
                         "the timed workload keeps the default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.evict_tokens is not None:
        if args.evict_tokens < EVICT["budget"] or args.evict_tokens % 4:
            ap.error("--evict-tokens must be a multiple of 4 and at least the budget")
        EVICT["T"] = args.evict_tokens

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
