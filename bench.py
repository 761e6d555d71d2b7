#!/usr/bin/env python3
"""Benchmark of the hybrid-attention forward (CSA + HCA + sliding window) on B300.

One step = one pass of the whole forward over one batch: for the default
workload (Pro-shaped 1M-token hybrid decode, batch 4) that is, per sequence,
a CSA layer (compress the completed block of the KV streams and of the
indexer keys, lightning-indexer scores over 262,144 entries, top-1024, sparse
MQA attention, sliding-window merge) and an HCA layer (compress, dense MQA
attention over 8,192 entries, sliding-window merge).

Prints ONE JSON line.  `value` is decode queries/s (or prefill tokens/s)
with inputs resident in HBM; `e2e` is the same metric through the public
API with the step's fresh inputs copied from pinned host memory and the
outputs read back inside the timed region.

Timing: W warm-up steps, then exactly K steps captured as one CUDA graph of
the library's launches and replayed once between CUDA events (the headline
time); inputs rotate over enough copies that one pass over them touches at
least 4x the L2 size.  A second graph of the same K steps with CUDA events
around every stage, and around the indexer's scoring kernel (recorded by the
library), gives each stage's and that kernel's average duration (the
roofline); its own step time is reported beside the headline.

`session` (hybrid decode, one GPU): the same layer pair decoded token by token
through the incremental session (caches, block tails and windows in rings) over
the 128 positions ending at the workload's query, one CUDA graph per token.
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
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "pro_1m_hybrid_decode"
METRIC = "hybrid-attn decode queries/s & prefill tok/s at 1M ctx; % HBM/TC roofline"


# ---------------------------------------------------------------- peaks


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# -------------------------------------------------------- algorithmic bytes


def stage_model(w, proj=None):
    """Algorithmic bytes / flops per stage per step (the minimum traffic the
    stage's definition needs: each input read once, each output written once).
    proj: the step's grouped output projection, {"g", "d_g", "in_heads", "calls"} (None: none)."""
    B, c, H = w.batch, w.c, w.n_h
    bf = 2 if w.dtype.itemsize == 2 else 4
    kb, qb = _index_row_bytes(w)
    m = {}
    if w.kind == "swa_decode":
        m["swa"] = dict(bytes=B * (w.n_win * c * bf + H * c * bf * 2), flops=B * w.n_win * H * c * 4,
                        flop_dtype="bf16")
    if w.kind in ("hybrid_decode", "csa_decode", "parallel_decode"):
        N = w.n_csa
        m["csa_compress"] = dict(bytes=B * (4 * 2 * w.m * (c + w.c_I) * bf + c * bf + kb), flops=0)
        m["csa_index_topk"] = dict(bytes=B * (N * kb + w.n_ih * (qb + 4) + w.k * 4),
                                   flops=B * N * w.n_ih * w.c_I * 2, flop_dtype="fp8")
        # attention over the selected entries with the window merge fused (one call)
        m["csa_attend"] = dict(bytes=B * ((w.k + w.n_win) * c * bf + w.k * 4 + H * c * bf + H * c * bf + H * 4),
                               flops=B * (w.k + w.n_win) * H * c * 4, flop_dtype="bf16")
    if w.kind in ("hybrid_decode", "hca_decode", "parallel_decode"):
        Nh = w.n_hca
        m["hca_compress"] = dict(bytes=B * (2 * w.m_hca * c * bf + c * bf), flops=0)
        m["hca_attend"] = dict(bytes=B * ((Nh + w.n_win) * c * bf + H * c * bf + H * c * bf + H * 4),
                               flops=B * (Nh + w.n_win) * H * c * 4, flop_dtype="bf16")
    if w.kind == "csa_prefill":
        n, N = w.n_ctx, w.n_csa
        pairs = sum(min(N, (t + 1) // w.m) for t in range(n))  # visible (query, entry) pairs
        sel = sum(min(w.k, (t + 1) // w.m) for t in range(n))
        win = sum(min(w.n_win, t + 1) for t in range(n))
        m["csa_compress"] = dict(bytes=n * 4 * (c + w.c_I) * bf + N * (c * bf + w.c_I + 4), flops=0)
        m["csa_index_topk"] = dict(bytes=n * w.n_ih * (w.c_I + 8) + N * (w.c_I + 4) + n * w.k * 4,
                                   flops=pairs * w.n_ih * w.c_I * 2, flop_dtype="fp8")
        m["csa_attend"] = dict(bytes=n * H * c * (bf + bf) + N * c * bf + n * w.k * 4 + n * c * bf,
                               flops=(sel + win) * H * c * 4, flop_dtype="bf16")
    if w.decode and "csa_compress" in m and "hca_compress" in m:
        # decode steps with both layers compress in one launch (hyb_compress_batch)
        cm = [m.pop(k) for k in ("csa_compress", "hca_compress") if k in m]
        m = dict(compress=dict(bytes=sum(v["bytes"] for v in cm), flops=0), **m)
    if proj is not None:
        rows = B * w.n_q
        K = proj["in_heads"] * c // proj["g"]
        m["proj"] = dict(bytes=proj["g"] * proj["d_g"] * K * 2 + rows * proj["in_heads"] * c * 2
                         + rows * proj["g"] * proj["d_g"] * 4,
                         flops=2 * rows * proj["g"] * proj["d_g"] * K, flop_dtype="bf16")
    return m


# DRAM bytes (read + write) of one launch of a kernel, counted by ncu
# (dram__bytes_read.sum + dram__bytes_write.sum) on a workload with the current
# build of that kernel; absent where no capture of the current kernel exists
KERNEL_NCU_TRAFFIC = {
    # index_tc_kernel<1>: 138.52 MB read (keys, scales, queries) + 6.60 MB written (scores, histograms)
    ("pro_1m_hybrid_decode", "index_scores"): 138_524_672 + 6_600_960,
    ("pro_1m_hybrid_decode", "csa_attend"): 5_348_096,
    ("pro_1m_hybrid_decode", "hca_attend"): 34_682_624 + 52_736,
    ("pro_1m_hybrid_decode", "topk"): 4_410_368,
    # the stage's two projections (one per layer), 137.9 MB each
    ("pro_1m_hybrid_decode", "proj"): 2 * (134_834_176 + 3_063_552),
}


def _index_row_bytes(w):
    """Bytes of one indexer key row (with its scales) and of one query head row (with its
    scales): FP8 c_I + 4 and c_I + 4; MXFP4 c_I/2 + c_I/32 for both."""
    if w.idx_fmt == "mxfp4":
        return w.c_I // 2 + w.c_I // 32, w.c_I // 2 + w.c_I // 32
    return w.c_I + 4, w.c_I + 4


def scoring_kernel_model(w):
    """Algorithmic bytes / flops of one launch of the indexer's scoring kernel (its
    inputs read once: the FP8 keys and scales, the queries, scales and head weights)."""
    if w.kind not in ("hybrid_decode", "csa_decode", "csa_prefill", "parallel_decode"):
        return None
    n_q = 1 if w.decode else w.n_ctx
    N = w.n_csa
    kb, qrow = _index_row_bytes(w)
    qb = w.n_ih * (qrow + 4)
    if w.decode:
        pairs = N
    else:
        pairs = sum(min(N, (t + 1) // w.m) for t in range(w.n_ctx))
    return dict(bytes=w.batch * (N * kb + n_q * qb), flops=w.batch * pairs * w.n_ih * w.c_I * 2,
                flop_dtype="fp8")


def topk_kernel_model(w):
    """Algorithmic bytes of the selection on its own: the float32 scores of the visible
    entries read once, the k indices written."""
    if w.decode:
        return dict(bytes=w.batch * (w.n_csa * 4 + w.k * 4), flops=0)
    pairs = sum(min(w.n_csa, (t + 1) // w.m) for t in range(w.n_ctx))
    return dict(bytes=w.batch * (pairs * 4 + w.n_ctx * w.k * 4), flops=0)


def stage_kernels(w):
    """The kernel of each timed stage, for the per-kernel roofline table (decode launches with
    128 heads run the 128-heads-per-CTA attention kernel, the others the 64-head one)."""
    att = "attend_h128_kernel" if (w.decode and w.n_h % 128 == 0) else "attend_tc_kernel"
    return {
        "swa": f"{att}<2> (swa_merge, window only)",
        "compress": "compress_batch_kernel (the step's compressions in one launch)",
        "proj": "out_proj_kernel (grouped output projection)",
        "csa_compress": "compress_kernel x2 (CSA entry bf16 + indexer key e4m3)",
        "csa_attend": f"{att}<0> (csa_attend, window fused)",
        "hca_compress": "compress_kernel (HCA entry)",
        "hca_attend": f"{att}<1> (hca_attend, window fused)",
    }


def kernel_roofline(name, model, ms, peaks, peak_kind, traffic=None):
    """Roofline entry of one kernel: algorithmic bytes (or flops, above the ridge) of one
    launch over its measured duration, against the measured peak."""
    if model["flops"] > 0 and model.get("flop_dtype") in ("bf16", "fp8") and \
            model["flops"] / max(model["bytes"], 1) > _ridge(peaks, model.get("flop_dtype")):
        peak = _tensor_peak(peaks, model["flop_dtype"])
        achieved = model["flops"] / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        peak = peaks["hbm_gbs"]
        achieved = model["bytes"] / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = achieved / peak
    roof["traffic"] = traffic
    roof["kernel"] = name
    roof["ms_per_launch"] = ms
    roof["algorithmic_bytes"] = model["bytes"]
    roof["algorithmic_flops"] = model["flops"]
    if roof["bound"] == "tensor" and model["flop_dtype"] == "fp8":
        roof["peak_source"] = peaks.get("fp8_source", "2 x the bf16 burst peak")
    else:
        roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    return roof


def _tensor_peak(peaks, dt):
    """Dense tensor peak (TFLOP/s) for a contraction of type dt.  The kernels here run
    at the maximum SM clock inside the step (no power cap seen), so the burst figures
    apply: bf16 from MEASURED_PEAKS.json, FP8 measured by this run (fp8_peak_probe)
    where it could be, else twice the bf16 figure."""
    if dt == "fp8":
        return peaks.get("fp8_tflops") or 2 * peaks["bf16_tflops"]
    return peaks["bf16_tflops"]


def fp8_peak_probe(device, n=8192, reps=10):
    """Dense FP8 (e4m3 x e4m3 -> bf16, cuBLASLt through torch._scaled_mm) n^3 GEMM: best of
    `reps` after warm-up, timed with CUDA events; 2 n^3 flops.  Timing only: no GPU setting
    is touched.  Returns TFLOP/s or None where the call is unavailable."""
    import torch

    try:
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=device)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2 * n ** 3 / (best / 1e3) / 1e12
    except Exception:  # noqa: BLE001 - the probe is optional
        return None


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- our arm


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x: the job's time is its slowest rank's."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the job's time."""
    return units_per_rank * world / (ms / 1e3)


def rank_seed(seed: int, rank: int) -> int:
    """Each rank decodes its own sequences (weak scaling): a distinct seed per rank."""
    return seed + 7919 * rank


def make_proj(w, spec, dev):
    """Seeded bf16 projection matrices for a step (HybridStep's proj argument) and the
    stage model's description of them.  spec: "per_layer" (each attention output of the
    step projected by its own [g][d_g][(n_h/g) c] set) or "concat" (one set over the 2 n_h
    concatenated heads of the parallel composition)."""
    import torch

    g_, d_g = w.out_groups, w.out_dim
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed + 31)
    heads = 2 * w.n_h if spec == "concat" else w.n_h
    K = heads * w.c // g_
    mk = lambda: (torch.randn((g_, d_g, K), generator=gen, device=dev) / math.sqrt(K)).to(torch.bfloat16)
    mats = {"w": mk()}
    calls = 2 if spec == "concat" else 1
    if spec == "per_layer" and w.kind == "hybrid_decode":
        mats["w_h"] = mk()
        calls = 2
    model = {"g": g_ * (2 if "w_h" in mats else 1), "d_g": d_g, "in_heads": heads * (2 if "w_h" in mats else 1),
             "calls": calls}
    return mats, model


def measure_workload(args, w, dev, dist=None, rank=0, world=1, steps_k=None, proj_spec=None, sample_clocks=True):
    """Time one workload: K steps captured as one CUDA graph of the library's launches
    (the step time), and the same K steps as a second graph with CUDA events around
    every stage and around the indexer's scoring kernel (stage and kernel times).
    Inputs rotate over enough copies that one pass streams at least 4x the L2 size.
    Returns (result dict, the step objects, the stream)."""
    import torch

    from sparse_attention_gated_b300 import pipeline, workloads

    K = steps_k or args.steps
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    mats, pmodel = make_proj(w, proj_spec, dev) if proj_spec else (None, None)
    model = stage_model(w, pmodel)
    step_bytes = sum(v["bytes"] for v in model.values())
    # each rank processes its own sequences (independent decode streams): different seeds
    wr = workloads.scaled(w, seed=rank_seed(w.seed, rank))
    copies = max(1, min(16, math.ceil(4 * l2 / max(step_bytes, 1))))
    if w.kind == "csa_prefill":
        copies = 1  # 17 GB per copy; one step streams >> L2
    steps = []
    for r in range(copies):
        x = workloads.make_inputs(workloads.scaled(wr, seed=wr.seed + 104729 * r), dev)
        steps.append(pipeline.HybridStep(w, x, proj=mats))
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    stages = list(model.keys())

    def run_step(st, ev=None):
        # one forward step; ev: dict stage -> (start, end) events recorded around each stage
        # (and "index_scores" -> the events the library records around its scoring kernel)
        def rec(name, which):
            if ev is not None and name in ev:
                ev[name][which].record(stream)

        if ev is None:  # the headline graph: the library's launches, as HybridStep.run issues them
            st.run(stream)
            return
        if st.swa_only:
            rec("swa", 0)
            st.run_swa(stream)
            rec("swa", 1)
        if "compress" in ev:
            rec("compress", 0)
            st.run_compress(stream)
            rec("compress", 1)
        if st.has_csa:
            rec("csa_compress", 0)
            _csa_parts(st, stream, rec, ev["index_scores"])
        if st.has_hca:
            rec("hca_compress", 0)
            _hca_parts(st, stream, rec)
        if st.proj is not None:
            rec("proj", 0)
            st.run_proj(stream)
            rec("proj", 1)

    # warm-up (eager), also the first-call setup of every kernel
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            run_step(steps[i % copies])
    stream.synchronize()
    if int(steps[0].dev_status.item()) != 0:
        raise RuntimeError(f"{w.name}: device status {int(steps[0].dev_status.item())}")

    ev = lambda: torch.cuda.Event(enable_timing=True, external=True)
    events = [{s_: (ev(), ev()) for s_ in stages + ["index_scores"]} for _ in range(K)]
    with torch.cuda.stream(stream):
        for e in events:  # create the events (the library records two of them itself)
            for pair in e.values():
                pair[0].record(stream), pair[1].record(stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    g_ev = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                run_step(steps[i % copies])
        with torch.cuda.graph(g_ev, stream=stream):
            for i in range(K):
                run_step(steps[i % copies], events[i])
    # warm the graphs (and the clocks) for about a second
    sampler = ClockSampler(dev.index or 0) if sample_clocks else None
    t_busy0 = time.time()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    # (replays until a second has passed, so that the clock samples cover the busy GPU)
    with torch.cuda.stream(stream):
        while time.time() - t_busy0 < 1.0:
            for _ in range(8):
                g.replay()
            stream.synchronize()
        g_ev.replay()
    stream.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t_timed1 = time.time()
    clocks = sampler.stop(t_busy0, t_timed1) if sampler else None
    ms_step = max_over_ranks(start.elapsed_time(end), dist, dev) / K
    # the evented graph, right after: per-stage and scoring-kernel times
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s0.record(stream)
        g_ev.replay()
        s1.record(stream)
    torch.cuda.synchronize()
    if int(steps[0].dev_status.item()) != 0:
        raise RuntimeError(f"{w.name}: device status {int(steps[0].dev_status.item())}")
    ms_step_ev = s0.elapsed_time(s1) / K
    has_scoring = "csa_index_topk" in stages
    timed = stages + (["index_scores"] if has_scoring else [])
    stage_ms = {s_: statistics.mean(events[i][s_][0].elapsed_time(events[i][s_][1]) for i in range(K))
                for s_ in timed}
    scoring_ms = stage_ms.pop("index_scores", None)
    units = w.batch if w.decode else w.n_ctx

    # roofline of every kernel (stage events; the indexer's scoring kernel by the events the
    # library records around it, the selection as the rest of its stage); the dominant kernel
    # is the one with the longest measured time
    peaks, peak_kind = args.peaks
    kern = {}
    if has_scoring:
        label = ("index_fp4_kernel (csa_index_topk scoring, MXFP4)" if w.idx_fmt == "mxfp4"
                 else "index_tc_kernel (csa_index_topk scoring)")
        kern["index_scores"] = (label, scoring_kernel_model(w), scoring_ms)
        kern["topk"] = ("topk_grid_kernel (csa_index_topk selection)", topk_kernel_model(w),
                        stage_ms["csa_index_topk"] - scoring_ms)
    for s_name, label in stage_kernels(w).items():
        if s_name in stage_ms:
            kern[s_name] = (label, model[s_name], stage_ms[s_name])
    kernels = {k: kernel_roofline(lbl, m_, ms_, peaks, peak_kind, KERNEL_NCU_TRAFFIC.get((w.name, k)))
               for k, (lbl, m_, ms_) in kern.items()}
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"])
    step_roof_s = step_bytes / (peaks["hbm_gbs"] * 1e9)
    # each stage at its own bound (bytes at the HBM peak or flops at the tensor peak)
    step_roof_any_s = sum(max(v["bytes"] / (peaks["hbm_gbs"] * 1e9),
                              v["flops"] / (_tensor_peak(peaks, v["flop_dtype"]) * 1e12) if v["flops"] else 0.0)
                          for v in model.values())
    config = {"workload": w.name, "batch": w.batch, "context": w.n_ctx, "n_h": w.n_h, "c": w.c, "m": w.m,
              "m_hca": w.m_hca, "top_k": w.k, "n_ih": w.n_ih, "c_I": w.c_I, "n_win": w.n_win,
              "l2_defeat": f"inputs rotate over {copies} copies (>= 4x L2 per pass)" if copies > 1 else
              "one step streams several times the L2 size", "graph": "K steps captured as one CUDA graph"}
    if pmodel:
        config["out_proj"] = {"spec": proj_spec, "groups": pmodel["g"], "d_g": pmodel["d_g"],
                              "weights": "seeded random bf16, resident"}
    res = {
        "value": job_rate(units, world, ms_step),
        "unit": "queries/s" if w.decode else "tokens/s",
        "ms_per_step": ms_step,
        "steps": K,
        "config": config,
        "clocks": clocks,
        "gpu_launches": _launches_per_step(w, pmodel) * K,
        "roofline": dict(kernels[dom]),
        "kernels": kernels,
        "stages_ms": stage_ms,
        "ms_per_step_with_stage_events": ms_step_ev,
        "step_hbm_roofline_frac": step_roof_s / (ms_step / 1e3),
        "step_roofline_frac": step_roof_any_s / (ms_step / 1e3),
    }
    return res, steps, stream


# the other workloads of the method's configurations, measured after the headline at N = 1:
# (workload, output projection, steps)
EXTRA_CONFIGS = (
    ("flash_csa_decode", None, 20),
    ("flash_hca_decode", None, 20),
    ("flash_swa_decode", None, 20),
    ("pro_1m_parallel_decode", "concat", 20),
    ("pro_1m_hybrid_decode", "per_layer", 20),
    ("pro_1m_hybrid_decode_fp4", None, 20),
    ("pro_1m_hybrid_decode_in_branch", None, 20),
    ("pro_csa_prefill", None, 3),
)


def run_ours(args, w):
    import torch

    from sparse_attention_gated_b300 import workloads

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    peaks, peak_kind = measured_peaks()
    fp8 = fp8_peak_probe(dev) if rank == 0 else None
    if fp8:
        peaks = dict(peaks, fp8_tflops=fp8, fp8_source="measured by this run: dense e4m3 8192^3 GEMM (cuBLASLt)")
    args.peaks = (peaks, peak_kind)

    res, steps, stream = measure_workload(args, w, dev, dist, rank, world)
    units = w.batch if w.decode else w.n_ctx
    # -------- e2e through the public API: fresh inputs from pinned host memory.  For the
    # hybrid decode: the session, one token per sequence per step (the serving loop); the
    # snapshot step with its whole block tails and windows re-sent is reported beside it.
    e2e_snap = run_e2e(args, w, steps[0], stream, units, world, dist)
    e2e = e2e_snap
    if w.kind == "hybrid_decode" and w.idx_fmt == "e4m3" and not w.in_branch:
        e2e = run_e2e_session(args, w, stream, world, dist)
    out = {
        "metric": METRIC,
        "value": res["value"],
        "unit": res["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16+fp8" if w.dtype != torch.float32 else "f32",
        "data": "synthetic",
        "config": res["config"],
        "clocks": res["clocks"],
        "e2e": e2e,
        "e2e_snapshot_step": e2e_snap if e2e is not e2e_snap else None,
        "gpu_launches": res["gpu_launches"],
        "roofline": res["roofline"],
        "kernels": res["kernels"],
        "fp8_tflops_measured": fp8,
        "stages_ms": res["stages_ms"],
        "ms_per_step_with_stage_events": res["ms_per_step_with_stage_events"],
        "step_hbm_roofline_frac": res["step_hbm_roofline_frac"],
        "step_roofline_frac": res["step_roofline_frac"],
    }
    if rank == 0 and world == 1 and w.kind == "hybrid_decode" and w.idx_fmt == "e4m3" and not args.no_session:
        out["session"] = run_session(w, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, steps[0])
    del steps
    if world == 1 and not args.no_configs:
        # the method's other configurations (context for the headline, same timing rules)
        out["configs"] = {}
        for name, spec, k in EXTRA_CONFIGS:
            torch.cuda.empty_cache()
            wx = workloads.WORKLOADS[name]
            key = name + ("+out_proj" if spec else "")
            try:
                r, st_x, _ = measure_workload(args, wx, dev, steps_k=min(args.steps, k), proj_spec=spec)
                if not args.no_cpu_baseline:
                    r["cpu_baseline"] = cpu_baseline(wx, st_x[0], budget_s=3.0, prefill_rows=4)
                del st_x
            except Exception as e:  # noqa: BLE001 - one failed extra config must not lose the headline
                r = {"error": f"{type(e).__name__}: {e}"}
            out["configs"][key] = r
    if dist is not None:
        dist.destroy_process_group()
    return out if rank == 0 else None


def _make_session(w, tokens, dev):
    """A DecodeSession at the workload's context, with the caches before the `tokens`
    positions ending at the workload's query position holding seeded random entries (as
    the decode workload's), and each of those tokens' rows and queries (device tensors)."""
    import math

    import torch

    from sparse_attention_gated_b300 import session

    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 7)
    Bq, c, cI = w.batch, w.c, w.c_I
    kv_std = 1.0 / math.sqrt(c)
    rn = lambda *shape, std=1.0: torch.randn(*shape, generator=g, device=dev).mul_(std)
    t0, t_end = w.n_ctx - tokens, w.n_ctx
    s = session.DecodeSession(batch=Bq, n_max=w.n_ctx, n_h=w.n_h, c=c, m=w.m, m_hca=w.m_hca, k=w.k, n_ih=w.n_ih,
                              c_I=cI, n_win=w.n_win, bias=rn(2 * w.m, c), biasI=rn(2 * w.m, cI),
                              bias_h=rn(w.m_hca, c), device=dev)
    nv, nvh = t0 // w.m, t0 // w.m_hca
    for i in range(0, nv, 16384):  # the entries before t0, in slices (bounded temporaries)
        j = min(nv, i + 16384)
        s.csa_kc[:, i:j] = rn(Bq, j - i, c, std=kv_std).to(s.dtype)
        s.csa_kI[:, i:j] = rn(Bq, j - i, cI).to(torch.float8_e4m3fn)
    s.csa_kIs[:, :nv] = torch.rand(Bq, nv, generator=g, device=dev) + 0.5
    s.hca_kc[:, :nvh] = rn(Bq, nvh, c, std=kv_std).to(s.dtype)
    for r in (s.rings, s.rings_I):
        r.copy_(rn(*r.shape, std=kv_std))
    width = {k: v[0].shape[-1] for k, v in s.token_slots(t0).items()}
    rows = [{k: rn(Bq, wd, std=kv_std).to(s.dtype) for k, wd in width.items()} for _ in range(tokens)]
    inp = [dict(q=rn(Bq, w.n_h, c).to(s.dtype), q_h=rn(Bq, w.n_h, c).to(s.dtype),
                qI=rn(Bq, w.n_ih, cI).to(torch.float8_e4m3fn),
                qI_scale=torch.rand(Bq, w.n_ih, generator=g, device=dev) + 0.5,
                w=torch.rand(Bq, w.n_ih, generator=g, device=dev)) for _ in range(tokens)]
    s.t = t0
    s.reserve(t_end - 1)
    return s, rows, inp, t0


def run_session(w, stream, tokens=128, reps=5):
    """Token-by-token decode through session.DecodeSession at the workload's context:
    the `tokens` positions ending at the workload's query position (every m-th token
    completes a CSA block, the last one an HCA block).  The caches before them hold
    seeded random entries (as the decode workload's), each token's appends and step are
    captured as one CUDA graph, and the graphs are replayed in order `reps` times
    between CUDA events.  The appends are torch copies into the rings (a model's
    projections would write there directly)."""
    import torch

    dev = torch.device("cuda")
    s, rows, inp, t0 = _make_session(w, tokens, dev)
    t_end = t0 + tokens
    Bq = w.batch
    with torch.cuda.stream(stream):
        for i in range(tokens):  # one eager pass (first launches, same writes as the replays)
            s.append(rows[i])
            s.step(**inp[i], stream=stream)
    stream.synchronize()
    if s.dev_status.item() != 0:
        raise RuntimeError(f"session decode: device status {s.dev_status.item()}")
    s.t = t0
    graphs = []
    for i in range(tokens):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            s.append(rows[i])
            s.step(**inp[i], stream=stream)
        graphs.append(gr)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for gr in graphs:
            gr.replay()
        stream.synchronize()
        e0.record(stream)
        for _ in range(reps):
            for gr in graphs:
                gr.replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / (reps * tokens)
    return {"tokens_per_s": Bq / (ms / 1e3), "ms_per_token_step": ms, "sequences": Bq,
            "positions": [t0, t_end - 1], "csa_blocks_completed": tokens // w.m,
            "hca_blocks_completed": tokens // w.m_hca, "reps": reps,
            "graph": "one CUDA graph per token (appends + step), replayed in order"}


def run_e2e_session(args, w, stream, world, dist, tokens=128):
    """The decode metric end to end through the public API as a serving loop runs it:
    DecodeSession token by token at the workload's context (4 sequences, positions
    n_ctx - tokens .. n_ctx - 1), every step copying in from pinned host memory only what
    one token brings (each sequence's raw rows of the token for every stream, its queries,
    indexer queries, scales and head weights: one packed buffer) and copying both layers'
    outputs back.  Host-to-device copies on one stream, device-to-host on another, two
    sets of step buffers, so that a token's copies overlap the neighbouring tokens'
    compute; the `tokens` steps are captured as one CUDA graph and replayed between CUDA
    events."""
    import torch

    dev = stream.device
    s, rows, inp, t0 = _make_session(w, tokens, dev)
    B = w.batch
    # the packed layout of one token's inputs (256-byte aligned fields)
    fields = [(k, v) for k, v in rows[0].items()] + [(k, inp[0][k]) for k in ("q", "q_h", "qI", "qI_scale", "w")]
    layout, off = [], 0
    for k, v in fields:
        n = v.numel() * v.element_size()
        layout.append((k, off, n, v.dtype, tuple(v.shape)))
        off = (off + n + 255) // 256 * 256
    nbytes = off
    host_in = torch.empty((tokens, nbytes), dtype=torch.uint8, pin_memory=True)
    for i in range(tokens):
        src = dict(rows[i], **inp[i])
        for k, o, n, dt, shp in layout:
            host_in[i, o:o + n].view(dt).copy_(src[k].reshape(-1).cpu())
    dev_in = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    view = [{k: d[o:o + n].view(dt).view(shp) for k, o, n, dt, shp in layout} for d in dev_in]
    out_shape = (2, B, 1, w.n_h, w.c)
    dev_out = [torch.empty(out_shape, dtype=s.dtype, device=dev) for _ in range(2)]
    host_out = [torch.empty(out_shape, dtype=s.dtype, pin_memory=True) for _ in range(2)]
    d2h = dev_out[0].numel() * dev_out[0].element_size()
    row_names = list(rows[0].keys())
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def steps(n):
        s.t = t0
        fork = torch.cuda.Event()
        fork.record(stream)
        s_h2d.wait_event(fork)
        s_d2h.wait_event(fork)
        freed = [None, None]
        for i in range(n):
            b = i % 2
            if freed[b] is not None:
                s_h2d.wait_event(freed[b])
                stream.wait_event(freed[b])
            with torch.cuda.stream(s_h2d):
                dev_in[b].copy_(host_in[i], non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_h2d)
            stream.wait_event(e_in)
            f = view[b]
            with torch.cuda.stream(stream):
                s.out, s.out_h = dev_out[b][0], dev_out[b][1]
                s.append({k: f[k] for k in row_names})
                s.step(q=f["q"], qI=f["qI"], qI_scale=f["qI_scale"], w=f["w"], q_h=f["q_h"], stream=stream)
            e_done = torch.cuda.Event()
            e_done.record(stream)
            s_d2h.wait_event(e_done)
            with torch.cuda.stream(s_d2h):
                host_out[b].copy_(dev_out[b], non_blocking=True)
            freed[b] = torch.cuda.Event()
            freed[b].record(s_d2h)
        for sx in (s_h2d, s_d2h):  # join
            j = torch.cuda.Event()
            j.record(sx)
            stream.wait_event(j)

    with torch.cuda.stream(stream):
        steps(tokens)  # eager pass: first launches and workspaces
    torch.cuda.synchronize()
    if s.dev_status.item() != 0:
        raise RuntimeError(f"session e2e: device status {s.dev_status.item()}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            steps(tokens)
        g.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, args.steps // tokens) if args.steps > tokens else 1
    with torch.cuda.stream(stream):
        s0.record(stream)
        for _ in range(reps):
            g.replay()
        s1.record(stream)
    torch.cuda.synchronize()
    if s.dev_status.item() != 0:
        raise RuntimeError(f"session e2e: device status {s.dev_status.item()}")
    ms = max_over_ranks(s0.elapsed_time(s1), dist, dev) / (reps * tokens)
    return {"value": job_rate(B, world, ms), "unit": "queries/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "path": "DecodeSession token by token (public API): per step one token's rows and queries per "
                    f"sequence in, both layers' outputs out; positions {t0}..{t0 + tokens - 1} "
                    f"({tokens // w.m} CSA and {tokens // w.m_hca} HCA blocks completed)",
            "graph": f"{tokens} token steps with their copies captured as one CUDA graph",
            "copies": "one H2D (packed token inputs) and one D2H (out, out_h) per step, on their own streams, "
                      "double-buffered so copies overlap the neighbouring steps' compute"}


def _ridge(peaks, dt):
    return _tensor_peak(peaks, dt) * 1e12 / (peaks["hbm_gbs"] * 1e9)


def _csa_parts(st, stream, rec, scoring_events=None):
    """The CSA layer's ABI calls with stage events between them (same calls as HybridStep.run
    issues; decode steps compressed before, in one launch); scoring_events: (begin, end)
    events the library records around its scoring kernel."""
    from sparse_attention_gated_b300 import ops

    w, x, b = st.w, st.x, st.buf
    kc, kI, kIs = st._csa_tensors()
    s = st.dev_status
    if w.decode and st.has_hca:
        pass  # compressed before, in one launch with the HCA entry
    elif w.decode:
        N = w.n_csa
        ops.hyb_compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True, first_block=N - 2,
                         out=kc, out_row0=N - 1, dev_status=s, stream=stream)
        ops.hyb_compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True,
                         first_block=N - 2, out=kI, out_scale=kIs, out_row0=N - 1, dev_status=s, stream=stream)
    else:
        ops.hyb_compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True, out=kc,
                         dev_status=s, stream=stream)
        ops.hyb_compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True, out=kI,
                         out_scale=kIs, dev_status=s, stream=stream)
    rec("csa_compress", 1)
    rec("csa_index_topk", 0)
    ops.csa_index_topk(x["qI"], x["w"], kI, m=w.m, k=w.k, q_pos0=w.q_pos0, qI_scale=x.get("qI_scale"), kI_scale=kIs,
                       idx=b["idx"], workspace=st.ws["index"], dev_status=s, stream=stream,
                       scores_events=scoring_events)
    rec("csa_index_topk", 1)
    rec("csa_attend", 0)
    # the in-branch RMSNorm + RoPE: both layers' in one launch when the step has both
    st.run_in_branch(stream, ("csa", "hca") if w.decode and st.has_hca else ("csa",))
    ops.csa_attend(x["q"], kc, kc, b["idx"], scale=w.scale, o=b["o"], lse=b["lse"], workspace=st.ws["csa"],
                   dev_status=s, stream=stream, window=st._win_csa(as_dict=True), sink=st.sink("csa"))
    rec("csa_attend", 1)


def _hca_parts(st, stream, rec):
    from sparse_attention_gated_b300 import ops

    w, x, b = st.w, st.x, st.buf
    s = st.dev_status
    kc = st._hca_cache()
    q = st._hca_q_kv()[0]
    if not st.has_csa:  # (with a CSA layer too, compressed before in one launch)
        Nh = w.n_hca
        ops.hyb_compress(x["ch"], x["zh"], x["bias_h"], w.m_hca, first_block=Nh - 1, out=kc, out_row0=Nh - 1,
                         dev_status=s, stream=stream)
    rec("hca_compress", 1)
    rec("hca_attend", 0)
    if not st.has_csa:
        st.run_in_branch(stream, ("hca",))
    ops.hca_attend(q, kc, kc, m=w.m_hca, q_pos0=w.q_pos0, scale=w.scale, o=b["o_h"], lse=b["lse_h"],
                   workspace=st.ws["hca"], dev_status=s, stream=stream, window=st._win_hca(as_dict=True),
                   sink=st.sink("hca"))
    rec("hca_attend", 1)


def _launches_per_step(w, proj=None):
    n = 0
    if w.kind == "swa_decode":
        n += 1
    if w.kind in ("hybrid_decode", "parallel_decode"):
        n += 1  # the step's three compressions, one launch
    if w.kind == "csa_decode":
        n += 2  # the entry and its indexer key
    if w.kind == "hca_decode":
        n += 1
    if w.kind in ("hybrid_decode", "csa_decode", "parallel_decode"):
        n += 2 + 1  # index scores + top-k, attention with the window merge fused
    if w.kind == "csa_prefill":
        n += 2 + 2 + 1  # compress x2, index scores + top-k, attention with the window merge fused
    if w.kind in ("hybrid_decode", "hca_decode", "parallel_decode"):
        n += 1
    if w.in_branch:
        # RMSNorm + RoPE of the queries and the completed entries (one launch); the sinks ride in
        # the 128-head attention launches, other head counts add a sink launch per layer
        n += 1
        if w.n_h % 128 != 0:
            n += (w.kind in ("hybrid_decode", "csa_decode")) + (w.kind in ("hybrid_decode", "hca_decode"))
    if proj is not None:
        n += proj["calls"]
    return n


def run_e2e(args, w, st, stream, units, world, dist):
    """Same metric through the public API (HybridStep.run), with every step's
    fresh inputs copied from pinned host memory and the outputs copied back.

    Steps are pipelined the way a serving loop runs them: two sets of step
    buffers (inputs and outputs each packed into one contiguous buffer, so one
    copy each way per step), host-to-device copies on one stream, device-to-host
    copies on another, so step i's copies overlap the compute of steps i-1 and
    i+1.  Every step still copies its whole input in and its output out inside
    the timed graph, and the compute of a step starts only after its input copy."""
    import torch

    from sparse_attention_gated_b300 import pipeline

    # a second step object over the same resident state (caches), with its own step buffers
    st2 = pipeline.HybridStep(st.w, dict(st.x))
    sts = [st, st2]
    io = [x.pack_step_io() for x in sts]
    host_in = [dev_in.cpu().pin_memory() for dev_in, _ in io]
    host_out = [torch.empty(dev_out.shape, dtype=torch.uint8, pin_memory=True) for _, dev_out in io]
    h2d = host_in[0].numel()
    d2h = host_out[0].numel()
    s_h2d, s_d2h = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)

    def steps(n):
        # fork the copy streams from the compute stream (joins them into a capture)
        fork = torch.cuda.Event()
        fork.record(stream)
        s_h2d.wait_event(fork)
        s_d2h.wait_event(fork)
        freed = [None, None]  # buffer b is free once the D2H of its last step is done
        for i in range(n):
            b = i % 2
            dev_in, dev_out = io[b]
            if freed[b] is not None:
                s_h2d.wait_event(freed[b])
                stream.wait_event(freed[b])
            with torch.cuda.stream(s_h2d):
                dev_in.copy_(host_in[b], non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_h2d)
            stream.wait_event(e_in)
            sts[b].run(stream)
            e_done = torch.cuda.Event()
            e_done.record(stream)
            s_d2h.wait_event(e_done)
            with torch.cuda.stream(s_d2h):
                host_out[b].copy_(dev_out, non_blocking=True)
            freed[b] = torch.cuda.Event()
            freed[b].record(s_d2h)
        for sx in (s_h2d, s_d2h):  # join
            j = torch.cuda.Event()
            j.record(sx)
            stream.wait_event(j)

    with torch.cuda.stream(stream):
        steps(max(args.warmup, 3))
    torch.cuda.synchronize()
    n = args.steps
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            steps(n)
        g.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s0.record(stream)
        g.replay()
        s1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(s0.elapsed_time(s1), dist, stream.device)
    return {"value": job_rate(units, world, ms / n), "unit": "queries/s" if w.decode else "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / n,
            "graph": "copies + step captured as one CUDA graph",
            "copies": "one H2D and one D2H per step (packed buffers), on their own streams, "
                      "double-buffered so copies overlap the neighbouring steps' compute"}


# ------------------------------------------------------------ CPU oracle


def oracle_query(w, x, b, proj=None):
    """The float64 oracle's chain for query b of a decode workload (the
    CPU-baseline unit of work), with the step's grouped output projection when
    proj (the step's matrices, CPU) is given.  x holds CPU tensors."""
    import numpy as np
    import torch

    import oracle

    t = w.n_ctx - 1
    sl = slice(b, b + 1)
    outs = []

    def in_branch(q, entry):
        # RMSNorm + partial RoPE of the queries and of the completed entry, at the query's position
        if not w.in_branch:
            return q
        oracle.rope_partial(oracle.rmsnorm(entry), t)
        return oracle.rope_partial(oracle.rmsnorm(q.float().numpy()), t).astype(np.float32)

    def sink(out_lse, key):
        return oracle.sink_merge(out_lse[0], out_lse[1], x[key])[0] if w.in_branch else out_lse[0]

    if w.kind == "swa_decode":
        q = x["q"][sl]
        o, _ = oracle.swa_merge(q, x["kv"][sl], x["kv"][sl], w.n_ctx - w.n_win, t, w.n_win, w.scale,
                                np.zeros(q.shape), np.full(q.shape[:3], -np.inf))
        outs.append(o)
    if w.kind in ("hybrid_decode", "csa_decode", "parallel_decode"):
        N = w.n_csa
        entry = oracle.compress(x["ca"][sl], x["za"][sl], x["bias"], w.m, cb=x["cb"][sl], zb=x["zb"][sl], overlap=True,
                                first_block=N - 2)
        kIn = oracle.compress(x["kIa"][sl], x["zIa"][sl], x["biasI"], w.m, cb=x["kIb"][sl], zb=x["zIb"][sl],
                              overlap=True, first_block=N - 2)
        if w.idx_fmt == "mxfp4":
            def dec(codes, scales):  # MXFP4 rows decoded by the oracle (element 2i in the low nibble)
                bts = codes.view(torch.uint8).numpy()
                un = np.empty(bts.shape[:-1] + (2 * bts.shape[-1],), dtype=np.uint8)
                un[..., 0::2], un[..., 1::2] = bts & 15, bts >> 4
                return oracle.mxfp4_decode(un, scales.view(torch.uint8).numpy()).astype(np.float32)

            oracle.quantise_mxfp4_rows(kIn.astype("float32"))
            s = oracle.index_scores(dec(x["qI"][sl], x["qI_scale"][sl]), x["w"][sl],
                                    dec(x["kI"][sl], x["kI_scale"][sl]), m=w.m, q_pos0=t)
        else:
            oracle.quantise_fp8_rows(kIn.astype("float32"))
            s = oracle.index_scores(x["qI"][sl], x["w"][sl], x["kI"][sl], m=w.m, q_pos0=t,
                                    qI_scale=x["qI_scale"][sl], kI_scale=x["kI_scale"][sl])
        idx = oracle.topk(s, [[N]], w.k)
        q = in_branch(x["q"][sl], entry)
        o, l = oracle.csa_attend(q, x["kc"][sl], x["kc"][sl], idx, w.scale)
        outs.append(sink(oracle.swa_merge(q, x["kv"][sl], x["kv"][sl], w.n_ctx - w.n_win, t, w.n_win, w.scale, o, l),
                         "sink"))
    if w.kind in ("hybrid_decode", "hca_decode", "parallel_decode"):
        sfx = "_h" if w.kind in ("hybrid_decode", "parallel_decode") else ""
        qsfx = "_h" if w.kind == "hybrid_decode" else ""
        kc = x["kc" + sfx][sl]
        entry = oracle.compress(x["ch"][sl], x["zh"][sl], x["bias_h"], w.m_hca, first_block=w.n_hca - 1)
        q = in_branch(x["q" + qsfx][sl], entry)
        o, l = oracle.hca_attend(q, kc, kc, m=w.m_hca, q_pos0=t, scale=w.scale)
        outs.append(sink(oracle.swa_merge(q, x["kv" + qsfx][sl], x["kv" + qsfx][sl], w.n_ctx - w.n_win, t, w.n_win,
                                          w.scale, o, l), "sink_h" if w.kind == "hybrid_decode" else "sink"))
    if proj is not None:
        if w.kind == "parallel_decode":  # one projection of the concatenated heads
            oracle.grouped_out_proj(np.concatenate(outs, axis=-2), proj["w"])
        else:
            for o_, key in zip(outs, ("w", "w_h")):
                oracle.grouped_out_proj(o_, proj[key])


def oracle_prefill_rows(w, x, rows):
    """Oracle chain of a prefill workload for the given query rows (plus the
    full compression of the chunk).  Returns the seconds spent on the rows."""
    import numpy as np

    import oracle

    ent = oracle.compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True)
    kIf = oracle.compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True)
    codes, scales = oracle.quantise_fp8_rows(kIf.astype(np.float32))
    e = oracle.round_bf16_bits(ent)
    t0 = time.perf_counter()
    for j in rows:
        js = slice(j, j + 1)
        s = oracle.index_scores(x["qI"][:, js], x["w"][:, js], codes, m=w.m, q_pos0=j, qI_scale=x["qI_scale"][:, js],
                                kI_scale=scales)
        idx = oracle.topk(s, [[oracle.visible(j, w.m)]], w.k)
        o, l = oracle.csa_attend(x["q"][:, js], e, e, idx, w.scale)
        oracle.swa_merge(x["q"][:, js], x["kv"], x["kv"], 0, j, w.n_win, w.scale, o, l)
    return time.perf_counter() - t0


def cpu_baseline(w, st=None, budget_s=25.0, prefill_rows=16):
    """The oracle, as it stands, on one host core, on a bounded sample."""
    import torch

    from sparse_attention_gated_b300 import workloads

    if st is not None:
        x = {k: v.detach().cpu() for k, v in st.x.items()}
    else:
        x = workloads.make_inputs(w, "cpu")
    proj = None
    if st is not None and st.proj is not None:
        proj = {k: v.float().cpu().numpy() for k, v in st.proj.items()}
    if w.decode:
        done, t0 = 0, time.perf_counter()
        while done < w.batch and (done == 0 or time.perf_counter() - t0 < budget_s):
            oracle_query(w, x, done, proj)
            done += 1
        dt = time.perf_counter() - t0
        return {"value": done / dt, "unit": "queries/s", "cores": 1, "kind": "oracle",
                "sample": f"{done} of the {w.batch} decode queries of one step, whole (float64, one thread)",
                "host_nproc": os.cpu_count()}
    rows = sorted(set([w.n_ctx - 1] + [int(r) for r in torch.linspace(0, w.n_ctx - 1, prefill_rows).tolist()]))
    dt = oracle_prefill_rows(w, x, rows)
    # extrapolate per-token time linearly in the attended work of each row
    def cost(j):
        return min(w.k, (j + 1) // w.m) + min(w.n_win, j + 1) + (j + 1) // w.m * 0.05
    sample_cost = sum(cost(j) for j in rows)
    total_cost = sum(cost(j) for j in range(w.n_ctx))
    est = dt * total_cost / sample_cost
    return {"value": w.n_ctx / est, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(rows)} evenly spaced query rows of the chunk (float64, one thread), extrapolated to "
                      f"all {w.n_ctx} rows by their attended work", "host_nproc": os.cpu_count()}


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from sparse_attention_gated_b300 import workloads

    x = {k: v for k, v in workloads.make_inputs(w, "cpu").items()}
    budget = 150.0
    if w.decode:
        for i in range(min(args.warmup, 1)):
            oracle_query(w, x, i % w.batch)
        t0 = time.perf_counter()
        done = 0
        while done < args.steps and (done == 0 or time.perf_counter() - t0 < budget):
            oracle_query(w, x, done % w.batch)
            done += 1
        dt = time.perf_counter() - t0
        value = done / dt
        sample = (f"{done} decode queries (one sequence per step: a CSA layer and an HCA layer, whole), "
                  f"float64 oracle on one core; {args.steps} steps were asked, capped at {budget:.0f} s")
        unit = "queries/s"
        ms = dt / done * 1e3
    else:
        rows = sorted(set([w.n_ctx - 1] + [int(r) for r in range(0, w.n_ctx, w.n_ctx // 8)]))
        dt = oracle_prefill_rows(w, x, rows)
        cb = cpu_baseline(w)
        value, unit, done, ms = cb["value"], "tokens/s", 1, w.n_ctx / cb["value"] * 1e3
        sample = cb["sample"]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1, "steps": done,
            "warmup": min(args.warmup, 1), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "context": w.n_ctx},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-session", action="store_true", help="skip the token-by-token session measurement")
    ap.add_argument("--no-configs", action="store_true", help="measure the headline workload only")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    from sparse_attention_gated_b300 import workloads

    w = workloads.WORKLOADS[args.workload]
    out = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
