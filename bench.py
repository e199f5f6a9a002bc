"""Benchmark of the MoE-layer hot path on GB300.

One step = route -> dispatch layout -> permute -> grouped SwiGLU FFN (+ the
shared expert where the workload has one) -> combine -> balancedness, over
one batch of seeded synthetic inputs already resident in HBM.

The headline line is the largest single-GPU layer: the group-limited layer
(4,096 tokens, hidden 7168, 256 routed experts in 8 groups, top-8 of the
top-4 groups, I=2048, plus a shared expert of width 2048, 32 simulated
ranks).  The same JSON line carries a record per further layer under
"workloads": the decode step (64 tokens), the 4,000-token prefill layer
(hidden 8192, 64 experts, top-2) and the replica layer (16,384 tokens,
hidden 4096, 32 experts, top-4, with its Zipf sweep of balancedness and
merged messages), each with its own stage table, roofline fraction and
clocks, timed over fewer steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--also decode,prefill,replica | --also none]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the path needs no exchange on one
GPU: ranks are simulated inside each replica), so scaling is weak.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s; grouped-GEMM % bf16 peak; permute/combine % HBM BW"
# the largest layer that fits one GPU (the most weights and flops per step)
HEADLINE = "group_limited"
DEFAULT_EXTRAS = ("decode", "prefill", "replica")
EXTRA_STEPS = 10


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


# ------------------------------------------------------------------ ncu traffic
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "grouped_ffn_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "grouped_ffn_gb300", "csrc", f)
                  for f in ("grouped_ffn.cu", "common.cuh", "tile_order.cuh", "umma.cuh")]


def kernel_source_hash() -> str:
    """sha256 of the kernel sources with comments and blank space removed, so
    that an edit to comments alone keeps a capture valid.  (The sources hold
    no comment markers inside string literals.)"""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()


def mode_name(args) -> str:
    """Non-default step variants; the committed traffic capture covers the
    default one only."""
    parts = [n for n, on in (("gather", args.gather), ("unpacked", args.unpacked),
                             ("masked", bool(args.masked_cap)), ("fp8", args.fp8_dispatch),
                             ("relax", bool(args.replica_relax)),
                             ("pair-ffn", getattr(args, "pair_ffn", False))) if on]
    return "+".join(parts)


def measured_traffic(workload: str, algorithmic_bytes: int):
    """DRAM bytes (read + write) of one grouped-FFN launch, scaled from the
    committed ncu capture of a smaller case of the same layer shape: the
    capture's traffic per algorithmic byte times this launch's algorithmic
    bytes (traffic grows with the weights streamed and the rows moved, as
    the algorithmic count does).  Returns (bytes, source) or (None, None) if
    there is no capture for this workload or the kernel source changed since
    it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, None
    if rec.get("kernel_sha256") != kernel_source_hash():
        return None, None
    w = rec.get("workloads", {}).get(workload)
    if w is None:
        return None, None
    ratio = (int(w["dram_bytes_read"]) + int(w["dram_bytes_write"])) / int(w["algorithmic_bytes"])
    src = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of %s (%s), %.3f per algorithmic "
           "byte, times this launch's algorithmic bytes; %s"
           % (w["case"], w["command"], ratio, os.path.relpath(TRAFFIC_FILE, ROOT)))
    return int(round(ratio * algorithmic_bytes)), src


# ------------------------------------------------------------------ dist
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 10 ms, each stamped with the host clock when
    read, so that the summary can keep only those taken during the timed
    region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0=None, t1=None, first=None):
        """Median SM clock and the throttle reasons seen in samples read in
        [t0, t1] (host monotonic seconds; None = unbounded), or in the first
        `first` samples read after t0."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        taken = 0
        for ts, ln in list(self.lines):
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            if first is not None and taken >= first:
                break
            taken += 1
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ algorithmic work
def algorithmic(w: wl.Workload, seg_counts: np.ndarray, slot_expert: np.ndarray,
                gather: bool = False, kept: int = None, fp8: bool = False,
                fused_shared: bool = False):
    """Bytes / flops per step by stage (the per-unit figures times the units).
    With the gather-fused FFN the rows come from x (2H bytes per token)
    instead of the permuted copy (2H per assignment).  kept: assignments
    that run (fewer than T*k when a fixed capacity drops some).  fp8: the
    dispatched rows carry H E4M3 bytes plus one fp32 scale per 128
    channels, restored to bf16 by a separate pass.  fused_shared: the shared
    expert runs in the routed FFN's launch, so its work counts there, and
    the permute writes its T extra rows."""
    A, T, H, I = w.A, w.T, w.H, w.I
    K = A if kept is None else kept
    active_slots = seg_counts > 0
    # weights are read once per active expert slot (replicas re-read: they
    # are separate copies in a real deployment)
    n_active = int(active_slots.sum())
    wbytes = n_active * 6 * H * I
    wire = H + 4 * (H // 128) if fp8 else 2 * H
    st = {
        "route": dict(bytes=T * w.E * 4 + T * w.k * 8),
        "layout": dict(bytes=A * 4 * 4 + A * 4),
        "permute": dict(bytes=T * H * 2 + K * wire),
        "grouped_ffn": dict(bytes=wbytes + (T if gather else K) * H * 2 + K * I * 2 * 2 + K * H * 2,
                            flops=6 * K * H * I, weight_bytes=wbytes),
        "combine": dict(bytes=K * H * 2 + T * H * 2 + (T * H * 2 if w.shared_I else 0) + A * 8),
    }
    if fp8:
        st["dequant"] = dict(bytes=K * wire + K * H * 2)
    if w.shared_I:
        sh = dict(bytes=6 * H * w.shared_I + T * H * 2 * 2 + T * w.shared_I * 4,
                  flops=6 * T * H * w.shared_I, weight_bytes=6 * H * w.shared_I)
        if fused_shared:
            g = st["grouped_ffn"]
            for key in ("bytes", "flops", "weight_bytes"):
                g[key] += sh[key]
            st["permute"]["bytes"] += T * H * 2
        else:
            st["shared_ffn"] = sh
    return st


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    from grouped_ffn_gb300 import MoELayer, moe

    dev = torch.device("cuda", torch.cuda.current_device())
    w = workload_from_args(args)
    pl = wl.make_placement(w)
    logits = wl.make_logits(w, dev)
    x = wl.make_x(w, dev)
    wgu = wl.make_w_gate_up(w, dev)
    wd = wl.make_w_down(w, dev)
    sgu, sd = wl.make_shared_weights(w, dev)
    layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=moe.DevicePlacement.from_tables(pl, dev),
                     w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                     n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                     shared_w_gate_up=sgu, shared_w_down=sd, device=dev,
                     packed=not args.unpacked, replica_relax=parse_relax(args.replica_relax),
                     gather=args.gather, masked_cap=args.masked_cap or None,
                     fp8_dispatch=args.fp8_dispatch, fuse_shared=not args.no_fuse_shared,
                     ffn_schedule=moe.FfnSchedule(cta_pairs=1) if args.pair_ffn else None)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    shared_stage = bool(w.shared_I) and not layer.fuse_shared   # a launch of its own
    names = ["route", "layout", "permute"] + (["dequant"] if args.fp8_dispatch else []) + \
        ["grouped_ffn"] + (["shared_ffn"] if shared_stage else []) + ["combine", "balance"]
    ffn_start = "dequant" if args.fp8_dispatch else "permute"
    ffn_stages = ["grouped_ffn"] + (["shared_ffn"] if shared_stage else [])
    K, W = args.steps, args.warmup
    ET = lambda: torch.cuda.Event(enable_timing=True)

    graph = None

    def step(marks=None):
        if graph is not None and marks is None:
            graph.replay()
        else:
            layer.forward(logits, x, y, stream, mark=marks)

    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
    stream.synchronize()
    layer.check(stream)
    if args.graph:
        # the whole step as one CUDA graph; replays run on `stream`
        with torch.cuda.stream(stream):
            graph = layer.capture(logits, x, y)
            for _ in range(W):
                graph.replay()
        stream.synchronize()

    # Timed region: K whole steps.  The only events inside it bracket the
    # grouped-FFN launches (their duration feeds the roofline); the other
    # stages run back to back with programmatic dependent launch.
    ffn_ev = [[ET() for _ in range(2 * len(ffn_stages))] for _ in range(K)]

    def timed_marks(i):
        evs = ffn_ev[i]
        slot = {ffn_start: 0, "grouped_ffn": 1}
        if shared_stage:
            slot.update({"grouped_ffn": 1, "shared_ffn": 3})
        def mark(name):
            if name in slot:
                evs[slot[name]].record(stream)
                if name == "grouped_ffn" and shared_stage:
                    evs[2].record(stream)
        return mark

    start, end = ET(), ET()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.2)   # let the sampler start
        barrier(world)
        torch.cuda.synchronize()
        t_start = time.monotonic()
        start.record(stream)
        with torch.cuda.stream(stream):
            for i in range(K):
                step(None if graph is not None else timed_marks(i))
        end.record(stream)
        stream.synchronize()
        t_end = time.monotonic()
        time.sleep(0.05)  # the last sample of the region reaches the reader
    torch.cuda.synchronize()
    barrier(world)
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    layer.check(stream)
    ffn_ms = {} if graph is not None else {
        n: float(np.mean([ffn_ev[i][2 * j].elapsed_time(ffn_ev[i][2 * j + 1]) for i in range(K)]))
        for j, n in enumerate(ffn_stages)}

    # Stage breakdown (not the headline): a separate pass with an event
    # after every stage; events between kernels also break their overlap.
    n_bd = min(K, 10)
    bd_ev = [[ET() for _ in range(len(names) + 1)] for _ in range(n_bd)]
    with torch.cuda.stream(stream):
        for i in range(n_bd):
            it = iter(bd_ev[i][1:])
            bd_ev[i][0].record(stream)
            step(lambda n, it=it: next(it).record(stream))
    stream.synchronize()
    stage_ms = {n: float(np.mean([bd_ev[i][j].elapsed_time(bd_ev[i][j + 1]) for i in range(n_bd)]))
                for j, n in enumerate(names)}
    stage_ms.update(ffn_ms)   # the FFN figures come from the timed region
    iso_ms = isolated_movers(args, w, layer, x, y, stream, K)

    # Merge (simulated): inter-node dispatch messages before / after merge
    # and the pre-reducing combine timed like the plain one (not in the step;
    # contiguous layout only)
    merge = None if args.masked_cap else run_merge(layer, w, y, stream, K)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(layer, logits, x, y, stream, world, K, W)
        e2e["value"] = world * w.T / (e2e["ms_per_step"] * 1e-3)
        e2e["h2d_bytes_per_step"] = logits.numel() * 4 + x.numel() * 2
        e2e["d2h_bytes_per_step"] = y.numel() * 2

    peaks = load_peaks()
    seg_counts = layer.seg_counts.cpu().numpy()
    dropped = int(layer.n_dropped.item()) if args.masked_cap else 0
    alg = algorithmic(w, seg_counts, pl.slot_expert, args.gather, kept=w.A - dropped,
                      fp8=args.fp8_dispatch, fused_shared=layer.fuse_shared)
    # samples read while the timed steps ran (one sampling interval of slack);
    # a region shorter than the interval may hold none, then the first three
    # read after it started stand in
    clock_rec = clocks.summary(t_start, t_end + 0.01)
    clock_rec["samples_in_region"] = clock_rec["samples"]
    if clock_rec["samples"] == 0:
        clock_rec = clocks.summary(t_start, None, first=3)
        clock_rec["samples_in_region"] = 0
    clock_rec["region_s"] = round(t_end - t_start, 4)
    return finish(args, w, pl, layer, logits, x, wgu, wd, sgu, sd, names, stage_ms, ms_step,
                  world, rank, K, W, alg, peaks, merge, e2e, dropped, clock_rec, dev, iso_ms)


def isolated_movers(args, w, layer, x, y, stream, K):
    """Per-launch duration of the permute and combine kernels, each launch
    timed alone between two events on its stream, with L2 flushed before
    it by writing a buffer twice the L2 size (default step only).  The
    in-step breakdown above also counts each kernel's launch and its wait
    for the previous one."""
    from grouped_ffn_gb300 import moe
    if args.gather or args.masked_cap or args.fp8_dispatch:
        return {}
    A, T = w.A, w.T
    shared = layer.shared_output(T)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=y.device)
    if layer.fuse_shared:   # the step's permute also writes the shared expert's rows
        perm = lambda: moe.moe_permute_shared(x, w.k, layer.dest_row[:A], layer.x_perm[:A + T],
                                              layer.ws, stream)
    else:
        perm = lambda: moe.moe_permute(x, w.k, layer.dest_row[:A], layer.x_perm[:A],
                                       layer.ws, stream)
    calls = {
        "permute": perm,
        "combine": lambda: moe.moe_combine(layer.y_perm[:A], layer.dest_row[:A],
                                           layer.topk_w[:T], y, layer.ws, shared, stream),
    }
    out = {}
    reps = max(3, min(K, 20))
    for name, fn in calls.items():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        with torch.cuda.stream(stream):
            for e0, e1 in ev:
                flush.fill_(1)
                e0.record(stream)
                fn()
                e1.record(stream)
        stream.synchronize()
        out[name] = float(np.mean([e0.elapsed_time(e1) for e0, e1 in ev]))
    layer.check(stream)
    return out


def run_merge(layer, w, y, stream, K):
    from grouped_ffn_gb300 import moe
    ET = lambda: torch.cuda.Event(enable_timing=True)
    dev = y.device
    msgs = torch.zeros(2, dtype=torch.int32, device=dev)
    y_m = torch.empty_like(y)
    shared_arg = layer.shared_output(w.T)
    mev = [ET() for _ in range(2)]
    with torch.cuda.stream(stream):
        for i in range(3 + K):
            if i == 3:
                mev[0].record(stream)
            moe.moe_combine_merged(layer.y_perm[:w.A], layer.dest_row[:w.A], layer.topk_w[:w.T],
                                   layer.slot[:w.A], layer.placement, y_m, msgs, layer.ws,
                                   shared_arg, stream)
        mev[1].record(stream)
    stream.synchronize()
    layer.check(stream)
    return {"inter_node_assignments": int(msgs[0].item()),
            "inter_node_messages_after_merge": int(msgs[1].item()),
            "bytes_saved_per_step": (int(msgs[0].item()) - int(msgs[1].item())) * w.H * 2 * 2,
            "combine_merged_us": mev[0].elapsed_time(mev[1]) / K * 1e3}


def tensor_peak(peaks, clocks):
    """bf16 peak (TFLOP/s) for the grouped GEMM timed inside the step, and its
    label.  The burst figure was measured at the maximum SM clock, the
    sustained one under the power cap after seconds of load; the timed
    region's own clock samples decide which conditions it ran under.  With
    no samples, or at the maximum clock without a power cap, it is the burst
    figure (the larger denominator)."""
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    if capped or (sm and mx and sm < 0.97 * mx):
        return peaks["bf16_tflops_sustained"], "sustained (SM clock %s of %s MHz%s in the timed region)" % (
            sm, mx, ", power cap" if capped else "")
    return peaks["bf16_tflops"], "burst (SM clock %s of %s MHz, no power cap in the timed region)" % (sm, mx)


def finish(args, w, pl, layer, logits, x, wgu, wd, sgu, sd, names, stage_ms, ms_step, world,
           rank, K, W, alg, peaks, merge, e2e, dropped, clocks, dev, iso_ms):
    """Stage table, roofline and the JSON record of our arm."""
    t_peak, t_peak_label = tensor_peak(peaks, clocks)
    stages = {}
    for n in names:
        if n == "balance":
            stages[n] = {"us": stage_ms[n] * 1e3}
            continue
        if n == "permute" and args.gather:
            stages[n] = {"us": stage_ms[n] * 1e3, "fused_into": "grouped_ffn"}
            continue
        a = alg[n]
        s = {"us": stage_ms[n] * 1e3, "gbs": a["bytes"] / (stage_ms[n] * 1e-3) / 1e9}
        s["hbm_frac"] = s["gbs"] / peaks["hbm_gbs"]
        if "flops" in a:
            s["tflops"] = a["flops"] / (stage_ms[n] * 1e-3) / 1e12
            s["tensor_frac"] = s["tflops"] / t_peak
            s["weight_gbs"] = a["weight_bytes"] / (stage_ms[n] * 1e-3) / 1e9
            bound_ms = max(a["flops"] / (t_peak * 1e12),
                           a["bytes"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
            s["roofline_frac"] = bound_ms / stage_ms[n]
        if n in iso_ms:   # the kernel alone, cold L2 (see isolated_movers)
            s["us_alone"] = iso_ms[n] * 1e3
            s["hbm_frac_alone"] = a["bytes"] / (iso_ms[n] * 1e-3) / 1e9 / peaks["hbm_gbs"]
        stages[n] = s
    g = alg["grouped_ffn"]
    g_ms = stage_ms["grouped_ffn"]
    intensity = g["flops"] / g["bytes"]
    ridge = t_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if intensity < ridge:
        roof = {"bound": "hbm", "achieved": g["bytes"] / (g_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": g["flops"] / (g_ms * 1e-3) / 1e12,
                "peak": t_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = (
        measured_traffic(w.name, g["bytes"]) if mode_name(args) == "" else (None, None))
    roof["kernel"] = "grouped_ffn_kernel (gate/up + down launches)"
    roof["peak_source"] = peaks["source"] + (" " + t_peak_label if roof["bound"] == "tensor" else
                                             " copy bandwidth")
    roof["algorithmic_bytes_per_step"] = g["bytes"]
    roof["algorithmic_flops_per_step"] = g["flops"]

    value = world * w.T / (ms_step * 1e-3)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.T, "hidden": w.H, "experts": w.E, "top_k": w.k,
                   "ffn_intermediate": w.I, "shared_intermediate": w.shared_I,
                   "simulated_ranks": w.R, "zipf_s": w.zipf_s, "assignments": w.A,
                   "parallelism": f"replicas{world}",
                   "weight_layout": "plain" if args.unpacked else "packed",
                   "dispatch": "gather-fused" if args.gather else
                               ("fp8-e4m3 permute + dequant (128-channel power-of-two scales)"
                                if args.fp8_dispatch else "permute"),
                   "layout": ("fixed capacity %d rows per slot" % args.masked_cap)
                             if args.masked_cap else "contiguous",
                   "shared_expert": None if not w.shared_I else
                                    ("in the routed FFN launch" if layer.fuse_shared
                                     else "second FFN launch"),
                   "launch": "cuda-graph replay" if args.graph else "stream (PDL)",
                   "l2": "inputs larger than L2: %.2f GB of expert weights stream per step"
                         % (g["weight_bytes"] / 1e9)},
        "e2e": e2e,
        "gpu_launches": layer.launches_per_step * K,
        "roofline": roof,
        "stages": stages,
        "gemm_pct_bf16_peak": 100.0 * stages["grouped_ffn"]["tflops"] / peaks["bf16_tflops"],
        "permute_pct_hbm": None if args.gather else 100.0 * stages["permute"].get(
            "hbm_frac_alone", stages["permute"]["hbm_frac"]),
        "combine_pct_hbm": 100.0 * stages["combine"].get("hbm_frac_alone",
                                                         stages["combine"]["hbm_frac"]),
        "balancedness": float(layer.balancedness.item()),
        "dropped_assignments": dropped,
        "merge": merge,
        "clocks": clocks,
    }
    if w.hot_experts > 0:
        out["replica_zipf_sweep"] = replica_sweep(w, dev, parse_relax(args.replica_relax) or (1, 10))
        out["config"]["replica_routing"] = ("waterfill C=" + args.replica_relax) \
            if args.replica_relax else "fixed rule (own node, else t mod copies)"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, pl, logits, x, wgu, wd, sgu, sd, args.cpu_seconds)
    return out


def run_e2e(layer, logits, x, y, stream, world, K, W):
    """The same step end to end through the public API: every step copies its
    inputs from pinned host memory and its output back, inside the timer.
    HostPipeline overlaps step i's copies with the neighbouring steps'
    compute on separate streams."""
    from grouped_ffn_gb300.layer import HostPipeline
    T, E = logits.shape
    logits_h = logits.cpu().pin_memory()
    x_h = x.cpu().pin_memory()
    y_h = torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()
    pipe = HostPipeline(layer, T, E, depth=2, device=y.device)
    for _ in range(W):
        pipe.submit(logits_h, x_h, y_h)
    pipe.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(pipe.h2d)
    for _ in range(K):
        pipe.submit(logits_h, x_h, y_h)
    e1.record(pipe.d2h)
    pipe.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / K
    layer.check(pipe.comp)
    assert torch.equal(y_h, y.cpu()), "end-to-end output differs from the device-resident run"
    return {"unit": "tokens/s", "ms_per_step": e2e_ms, "copies": "overlapped (3 streams, 2 buffers)"}


def parse_relax(text):
    """'1/10' -> (1, 10); '' -> None (fixed replica rule)."""
    if not text:
        return None
    num, _, den = text.partition("/")
    return int(num), int(den or 1)


def replica_sweep(w, dev, relax):
    """Balancedness, inter-node assignments and merged dispatch messages
    (distinct (token, remote node) pairs) at each Zipf exponent of the
    sweep, for the fixed replica rule, for water-filling routing and for
    water-filling followed by the consolidation refinement (route + layout
    only; the FFN result does not depend on the copy chosen)."""
    from grouped_ffn_gb300 import moe
    pl = wl.make_placement(w)
    pl_dev = moe.DevicePlacement.from_tables(pl, dev)
    out = []
    A, S, R = w.A, pl.n_slots, w.R
    i32 = lambda n: torch.empty(n, dtype=torch.int32, device=dev)
    ws = moe.new_workspace(w.T, w.k, S, device=dev, n_experts=w.E, n_ranks=R)
    bal = torch.empty(1, dtype=torch.float64, device=dev)
    mx, tot = i32(1), torch.empty(1, dtype=torch.int64, device=dev)
    for z in wl.REPLICA_ZIPF_SWEEP:
        wz = w.with_zipf(z)
        logits = wl.make_logits(wz, dev)
        ids, wts = i32(A).view(w.T, w.k), torch.empty(w.T, w.k, dtype=torch.float32, device=dev)
        moe.moe_route(logits, moe.RouteCfg(w.score_fn, w.k, w.n_groups, w.topk_groups,
                                           w.group_topn), ids, wts)
        rec = {"zipf_s": z}
        slot, counts, offs, dest, src, rc = i32(A), i32(S), i32(S + 1), i32(A), i32(A), i32(R)
        moe.moe_dispatch_layout(ids, pl_dev, slot, counts, offs, dest, src, rc, ws)
        moe.moe_balance_stats(rc, bal, mx, tot)
        node = pl_dev.slot_rank[slot.long()] // w.ranks_per_node
        tok_node = (torch.arange(A, device=dev) // w.k % R) // w.ranks_per_node
        remote = node != tok_node
        tok = torch.arange(A, device=dev) // w.k
        n_nodes = (R + w.ranks_per_node - 1) // w.ranks_per_node
        fixed_msgs = int(torch.unique(tok[remote] * n_nodes + node[remote]).numel())
        rec["fixed_rule"] = {"balancedness": float(bal.item()), "max_rank_load": int(mx.item()),
                             "inter_node": int(remote.sum().item()),
                             "messages_after_merge": fixed_msgs}
        inter = i32(1)
        moe.moe_route_replicas(ids, pl_dev, relax[0], relax[1], slot, inter, ws)
        moe.moe_dispatch_layout_routed(ids, slot, pl_dev, counts, offs, dest, src, rc, ws)
        moe.moe_balance_stats(rc, bal, mx, tot)
        moe.moe_check_device_status(ws)
        rec["waterfill"] = {"relax_C": relax[0] / relax[1], "balancedness": float(bal.item()),
                            "max_rank_load": int(mx.item()), "inter_node": int(inter.item())}
        # the greedy consolidation of each token's remote requests, timed
        msgs = i32(2)
        stream = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        moe.moe_route_refine(ids, pl_dev, slot, msgs, ws, stream)
        e1.record(stream)
        moe.moe_dispatch_layout_routed(ids, slot, pl_dev, counts, offs, dest, src, rc, ws)
        moe.moe_balance_stats(rc, bal, mx, tot)
        moe.moe_check_device_status(ws)
        before, after = (int(v) for v in msgs.cpu())
        rec["waterfill"]["messages_after_merge"] = before
        rec["waterfill_refined"] = {"balancedness": float(bal.item()),
                                    "max_rank_load": int(mx.item()),
                                    "inter_node": int(inter.item()),
                                    "messages_after_merge": after,
                                    "refine_us": round(e0.elapsed_time(e1) * 1e3, 1)}
        out.append(rec)
    return out


def workload_from_args(args) -> wl.Workload:
    w = wl.WORKLOADS[args.workload]
    if args.zipf is not None:
        w = w.with_zipf(args.zipf)
    over = {}
    if args.tokens:
        over["T"] = args.tokens
    if args.experts:
        # a smaller case of the same layer shape (profiling captures)
        over["E"] = args.experts
        over["R"] = min(w.R, args.experts)
        over["ranks_per_node"] = min(w.ranks_per_node, over["R"])
    if over:
        w = w.scaled(name=w.name + "_scaled", **over)
    return w


# ------------------------------------------------------------------ CPU oracle
def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_cpu_model() -> str:
    """The host CPU's model as /proc/cpuinfo names it (x86 'model name'; Arm
    cores report implementer and part codes instead)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip()
                if key in ("model name", "CPU implementer", "CPU part") and key not in fields:
                    fields[key] = val.strip()
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return "%s, implementer %s part %s" % (platform.machine(), fields.get("CPU implementer", "?"),
                                               fields["CPU part"])
    return platform.machine()


def oracle_sample_step(w, pl, logits_np, x_bits, experts_gu, experts_d, shared, tokens,
                       stage_s=None):
    """The oracle's stage-wise path on a sample of tokens: route, layout,
    permute, grouped FFN (+ shared expert), combine, balancedness.  If
    stage_s (a dict) is given, each stage's seconds are added to it."""
    import oracle
    clock = [time.perf_counter()]

    def lap(name):
        now = time.perf_counter()
        if stage_s is not None:
            stage_s[name] = stage_s.get(name, 0.0) + now - clock[0]
        clock[0] = now

    lg = logits_np[tokens]
    if w.score_fn == wl.SCORE_SOFTMAX and w.n_groups == 1:
        ids, wts = oracle.route_softmax_topk(lg, w.k)
    else:
        ids, wts, _ = oracle.route_group_limited(lg, w.k, w.n_groups, w.topk_groups, w.group_topn)
    lap("route")
    lay = oracle.dispatch_layout(ids, pl if pl.token_src_rank is None else pl)
    lap("layout")
    xs = oracle.bf16_bits_to_f64(x_bits[tokens])
    xp = oracle.permute(xs, lay["dest_row"], w.k)
    lap("permute")
    _, yp = oracle.grouped_ffn(xp, lay["seg_offsets"], pl.slot_expert, experts_gu, experts_d, w.I)
    sh = None
    if shared is not None:
        _, sh = oracle.swiglu_expert(xs, shared[0], shared[1], w.shared_I)
    lap("grouped_ffn")
    y = oracle.combine_f64(yp, lay["dest_row"], wts.astype(np.float32).astype(np.float64), sh)
    lap("combine")
    oracle.balance_stats(lay["rank_counts"])
    lap("balance")
    return y


class _HostExperts:
    """Expert weights for the oracle: bf16 bits copied to the host once
    (outside any timer), converted to fp64 on each use (inside it)."""

    def __init__(self, t):
        self.t, self.cache = t, {}

    def fetch(self, e):
        if e not in self.cache:
            self.cache[e] = _bits(self.t[e])

    def __getitem__(self, e):
        import oracle
        self.fetch(e)
        return oracle.bf16_bits_to_f64(self.cache[e])


def cpu_baseline(w, pl, logits, x, wgu, wd, sgu, sd, seconds):
    """Time the oracle, as it stands, on a bounded sample of the workload."""
    rng = np.random.default_rng(12345)
    logits_np = logits.cpu().numpy()
    x_bits = _bits(x)
    gu, d = _HostExperts(wgu), _HostExperts(wd)
    shared = None if sgu is None else (
        __import__("oracle").bf16_bits_to_f64(_bits(sgu[0])),
        __import__("oracle").bf16_bits_to_f64(_bits(sd[0])))
    n = 4
    done_tokens, t_used = 0, 0.0
    stage_s = {}
    while t_used < seconds and done_tokens < w.T and n <= 256:
        toks = np.sort(rng.choice(w.T, size=min(n, w.T), replace=False))
        # host copies of the experts this sample needs are made outside the timer
        import oracle
        ids = (oracle.route_softmax_topk(logits_np[toks], w.k)[0]
               if (w.score_fn == wl.SCORE_SOFTMAX and w.n_groups == 1)
               else oracle.route_group_limited(logits_np[toks], w.k, w.n_groups,
                                               w.topk_groups, w.group_topn)[0])
        for e in np.unique(ids):
            gu.fetch(int(e))
            d.fetch(int(e))
        t0 = time.perf_counter()
        oracle_sample_step(w, pl, logits_np, x_bits, gu, d, shared, toks, stage_s)
        t_used += time.perf_counter() - t0
        done_tokens += len(toks)
        n *= 2
    return {"value": done_tokens / t_used, "unit": "tokens/s", "cores": os.cpu_count(),
            "cpu_model": host_cpu_model(),
            "kind": "oracle",
            "sample": f"{done_tokens} of {w.T} tokens of the {w.name} layer through the oracle's "
                      f"stage-wise path (route, layout, permute, grouped FFN, combine, balance) "
                      f"in {t_used:.1f} s; numpy fp64, BLAS threads = host cores",
            # route, layout and balance run single-threaded (plain Python /
            # numpy loops); the FFN's matmuls use the BLAS threads
            "stage_us_per_token": {k: v / done_tokens * 1e6 for k, v in stage_s.items()}}


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle, timed per step on a bounded sample."""
    if rank != 0:
        return None
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    w = workload_from_args(args)
    pl = wl.make_placement(w)
    logits = wl.make_logits(w, dev)
    x = wl.make_x(w, dev)
    wgu = wl.make_w_gate_up(w, dev)
    wd = wl.make_w_down(w, dev)
    sgu, sd = wl.make_shared_weights(w, dev)
    import oracle
    logits_np = logits.cpu().numpy()
    x_bits = _bits(x)
    gu, d = _HostExperts(wgu), _HostExperts(wd)
    shared = None if sgu is None else (oracle.bf16_bits_to_f64(_bits(sgu[0])),
                                       oracle.bf16_bits_to_f64(_bits(sd[0])))
    rng = np.random.default_rng(777)
    # a step's sample: about 32 routed assignments (its expert weights
    # dominate the oracle's time)
    n_tok = max(1, min(w.T, args.ref_tokens or max(1, 32 // w.k)))
    samples = [np.sort(rng.choice(w.T, size=n_tok, replace=False))
               for _ in range(args.warmup + args.steps)]
    for toks in samples:      # host copies of the needed experts, outside the timer
        ids = (oracle.route_softmax_topk(logits_np[toks], w.k)[0]
               if (w.score_fn == wl.SCORE_SOFTMAX and w.n_groups == 1)
               else oracle.route_group_limited(logits_np[toks], w.k, w.n_groups,
                                               w.topk_groups, w.group_topn)[0])
        for e in np.unique(ids):
            gu.fetch(int(e))
            d.fetch(int(e))
    for toks in samples[: args.warmup]:
        oracle_sample_step(w, pl, logits_np, x_bits, gu, d, shared, toks)
    t0 = time.perf_counter()
    for toks in samples[args.warmup:]:
        oracle_sample_step(w, pl, logits_np, x_bits, gu, d, shared, toks)
    dt = (time.perf_counter() - t0) / args.steps
    value = n_tok / dt
    sample = (f"{n_tok} of {w.T} tokens per step of the {w.name} layer through the oracle's "
              f"stage-wise path; numpy fp64")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.T, "hidden": w.H, "experts": w.E,
                       "top_k": w.k, "ffn_intermediate": w.I, "zipf_s": w.zipf_s,
                       "parallelism": "replicas1", "sampled_tokens_per_step": n_tok},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                             "cpu_model": host_cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def extra_workloads(args):
    """Workloads recorded after the headline: the default set behind the
    default headline with the default step, else what --also names."""
    if args.also == "none" or not args.also:
        return []
    if args.also == "auto":
        plain = (args.workload == HEADLINE and mode_name(args) == "" and not args.graph
                 and args.zipf is None and not args.tokens and not args.experts)
        return list(DEFAULT_EXTRAS) if plain else []
    names = [n.strip() for n in args.also.split(",") if n.strip()]
    for n in names:
        if n not in wl.WORKLOADS:
            raise SystemExit(f"unknown workload in --also: {n}")
    return [n for n in names if n != args.workload]


def compact_record(rec):
    """A further workload's record: its throughput, stage table, roofline,
    target fractions, balancedness and clocks (no end-to-end or CPU legs)."""
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "gpu_launches",
            "roofline", "stages", "gemm_pct_bf16_peak", "permute_pct_hbm", "combine_pct_hbm",
            "balancedness", "merge", "clocks", "replica_zipf_sweep")
    return {k: rec[k] for k in keep if k in rec}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--also", default="auto",
                    help="further workloads recorded in the same line (comma list, 'none'; "
                         "auto: decode,prefill,replica after the default headline)")
    ap.add_argument("--zipf", type=float, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens per reference step (0: 32 routed assignments' worth)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as CUDA-graph replays (FFN roofline from the breakdown pass)")
    ap.add_argument("--gather", action="store_true",
                    help="FFN reads rows from x through the inverse permutation (no permute)")
    ap.add_argument("--replica-relax", default="",
                    help="choose replicas by water-filling with load bounds C, e.g. 1/10")
    ap.add_argument("--unpacked", action="store_true",
                    help="stream the expert weights in their plain [E,2I,H]/[E,H,I] layout")
    ap.add_argument("--masked-cap", type=int, default=0,
                    help="fixed-capacity layout with this many rows per slot (0: contiguous)")
    ap.add_argument("--fp8-dispatch", action="store_true",
                    help="dispatch E4M3 codes + block scales, restore bf16 before the FFN")
    ap.add_argument("--pair-ffn", action="store_true",
                    help="run the grouped FFN's tiles on pairs of SMs (tcgen05 cta_group::2)")
    ap.add_argument("--no-fuse-shared", action="store_true",
                    help="run the shared expert as a second FFN launch")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's expert count")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
        out = run_ours(args, world, rank, local)
        extras = extra_workloads(args)
        if extras:
            out["workloads"] = {}
            for name in extras:
                torch.cuda.empty_cache()
                sub = argparse.Namespace(**vars(args))
                sub.workload, sub.zipf, sub.tokens, sub.experts = name, None, 0, 0
                sub.steps = max(3, min(args.steps, EXTRA_STEPS))
                sub.warmup = max(3, min(args.warmup, 3))
                sub.no_e2e = sub.no_cpu_baseline = True
                out["workloads"][name] = compact_record(run_ours(sub, world, rank, local))
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
