#!/usr/bin/env python3
"""Benchmark of the MXFP8 MoE decode step (FFN half) on GB300: one JSON line.

Metric: microseconds per MoE decode step, with the achieved HBM GB/s of the
dominant kernel against the measured copy bandwidth. A step is one pass of the
whole path (seam, router, top-k with the operand panels, the experts, combine) over one
batch of M synthetic token rows, replayed from a CUDA graph with every input
resident in HBM; L2 is flushed before every timed step: a 512 MB buffer is
written and then read back, so that L2 holds none of the step's data and no
dirty lines (a write-only flush leaves ~126 MB of dirty lines that the step
would write back to HBM while it streams its weights; that time is reported
beside the headline as us_per_step_after_write_only_flush).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl mine|reference] [--no-sweep]

--impl reference times the CPU oracle (the reference arm of this build):
complete steps of the same workload, as many of the requested ones as fit a
fixed budget (it prints the counts it ran). Under torchrun
(N > 1) each rank runs an independent replica of the step (the layer does not
shard on one box); rank 0 prints.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per MoE decode step and achieved HBM GB/s (% of 8 TB/s) at M=1..48"
DEFAULT_WORKLOAD = "full_m48_uniform"
SWEEP = ["full_m48_zipf", "full_m1", "full_m16", "small_m4"]
# beyond the step at M = 1..48 of the 256-expert layer: the 384-expert layer
# and the attention seam's MXFP8 (reported under "next_rows")
NEXT_ROWS = ["full_e384_m1", "full_e384_m48", "full_e384_fp4_m1", "full_e384_fp4_m48"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-experts", type=int, default=4,
                    help="experts of the CPU baseline's sampled estimate (0: none)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


NOMINAL_GBS = 8000.0  # GB300 HBM3e nominal bandwidth: the metric's "% of 8 TB/s"


def kernel_hash() -> str:
    """Hash of the expert kernel's sources without comments and whitespace
    (an edit of a comment leaves the kernel, and its counters, as they were)."""
    h = hashlib.sha256()
    for f in ("expert.cu", "ptx.cuh", "mx.cuh", "internal.cuh"):
        with open(os.path.join(ROOT, "mxfp8_moe_decode_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, alg_bytes: int):
    """DRAM bytes per launch of `kernel` (dram__bytes_read.sum + write.sum)
    from the committed ncu summary, if it was taken on the current kernel
    source (else None). Captured on this workload: the measured bytes;
    captured on a smaller layer (multi-metric captures stay a few GB on the
    device): the measured bytes per algorithmic byte there, times this
    launch's algorithmic bytes. Returns (bytes, how)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_hash():
        return None, None
    if e.get("workload") == workload:
        return e.get("bytes_per_launch"), f"measured on {workload}"
    ratio = e["bytes_per_launch"] / e["alg_bytes_per_launch"]
    return round(ratio * alg_bytes), (f"scaled: {ratio:.4f} x the algorithmic bytes, the ratio "
                                      f"measured on {e['workload']}")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def base_config(wl, unique: int) -> dict:
    """The workload's keys, the same in both arms' lines."""
    from mxfp8_moe_decode_gb300 import workloads as W

    d = wl.dims
    return {"workload": wl.name, "desc": wl.note, "M": wl.tokens, "hidden": d.hidden,
            "experts": d.experts, "topk": d.topk, "inter": d.inter, "routed_format": d.routed,
            "shared_experts": 1, "unique_routed_experts": unique,
            "alg_bytes_per_step": W.algorithmic_bytes(d, unique)}


# ---------------------------------------------------------------- GPU arm
def make_layer(wl, dev, ew=None):
    import torch

    from mxfp8_moe_decode_gb300 import MoeDecode
    from mxfp8_moe_decode_gb300 import workloads as W

    d = wl.dims
    ri = W.router_inputs(wl)
    if ew is None:
        ew = W.expert_weights(wl, device=dev)
    weights = {"norm_w": ri["norm_w"].to(dev), "gate_w": ri["gate_w"].to(dev),
               "bias": ri["bias"].to(dev), **ew}
    layer = MoeDecode(d.hidden, d.experts, d.topk, d.inter, weights, max_tokens=d.max_tokens,
                      eps=d.eps, routed=d.routed)
    x = W.token_rows(wl).to(dev)
    torch.cuda.synchronize(dev)
    return layer, x, ew


def capture(layer, x, dev, events=None):
    """A CUDA graph of one step (per-kernel timing events recorded as graph
    nodes when `events` is given; the events must outlive the graph)."""
    import torch

    out = torch.empty_like(x)
    layer.set_timing_events(events)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        layer.step(x, out=out, stream=s)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer.step(x, out=out, stream=s)
    torch.cuda.synchronize(dev)
    layer.set_timing_events(None)
    return g, out


def time_attn_seam(wl, dev, flush, steps: int) -> dict:
    """moe_attn_seam_x8 on the workload's M rows: CUDA events around each
    launch, L2 flushed before each; bytes = x, weight, E4M3 bytes and codes."""
    import torch

    from mxfp8_moe_decode_gb300 import attn_seam_x8
    from mxfp8_moe_decode_gb300 import workloads as W
    x = W.token_rows(wl).to(dev)
    w = W.attn_norm_weight(wl).to(dev)
    M, H = x.shape
    x8 = torch.empty((M, H), dtype=torch.uint8, device=dev)
    codes = torch.empty((M, H // 32), dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream(dev)
    for _ in range(3):
        attn_seam_x8(x, w, wl.dims.eps, x8=x8, codes=codes)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for e0, e1 in ev:
        flush()
        e0.record(cur)
        attn_seam_x8(x, w, wl.dims.eps, x8=x8, codes=codes)
        e1.record(cur)
    torch.cuda.synchronize(dev)
    us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
    nbytes = M * H * 2 + H * 2 + M * H + M * H // 32
    return {"M": M, "hidden": H, "us_per_call": round(us, 3), "bytes": nbytes,
            "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "note": "one CTA per token row, latency-bound (bytes << what HBM moves in "
                    "a launch's latency); L2 flushed before each timed launch"}


def time_layer(layer, x, dev, steps: int, warmup: int, flush):
    """Graph-replay timing, L2 flushed (untimed) before every replay. The step
    time is taken by two event nodes inside the step's graph, just before its
    first kernel and after its last (the kernels still overlap through
    programmatic dependent launch; the graph's own launch latency is outside);
    the same graph replayed between stream events gives the replay time,
    launch latency included. The per-kernel breakdown comes from a third
    graph with an event node between kernels.
    Returns (per-step ms, per-kernel mean ms, unique routed, graph, out,
    per-replay ms)."""
    import torch

    from mxfp8_moe_decode_gb300 import kernel_names

    for _ in range(max(warmup, 3)):
        layer.step(x)
    torch.cuda.synchronize(dev)
    g, out = capture(layer, x, dev)
    if layer.status() != 0:
        raise RuntimeError(f"device status {layer.status()}")
    unique = layer.unique_experts()
    cur = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        flush()
        g.replay()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    replay_ms = []
    for _ in range(steps):
        flush()
        t0.record(cur)
        g.replay()
        t1.record(cur)
        t1.synchronize()
        replay_ms.append(t0.elapsed_time(t1))

    eb = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    gb, _ = capture(layer, x, dev, events=eb)
    step_ms = []
    for i in range(warmup + steps):
        flush()
        gb.replay()
        eb[1].synchronize()
        if i >= warmup:
            step_ms.append(eb[0].elapsed_time(eb[1]))
    torch.cuda.synchronize(dev)
    del gb  # the graph holds record nodes of `eb`: drop it before the events

    nk = len(kernel_names())
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    gk, _ = capture(layer, x, dev, events=evs)
    kern = [[] for _ in range(nk)]
    for i in range(warmup + steps):
        flush()
        gk.replay()
        evs[-1].synchronize()
        if i >= warmup:
            for k in range(nk):
                kern[k].append(evs[k].elapsed_time(evs[k + 1]))
    torch.cuda.synchronize(dev)
    del gk  # the graph holds record nodes of `evs`: drop it before the events
    torch.cuda.synchronize(dev)
    if layer.status() != 0:
        raise RuntimeError(f"device status {layer.status()}")
    kmean = [statistics.mean(k) for k in kern]
    return step_ms, kmean, unique, g, out, replay_ms


def kernel_table(names, ms, launches: int) -> dict:
    """Per-kernel µs; a step that launches one kernel fewer runs the seam in
    the router (its seam events bracket nothing: reported as null)."""
    out = {n: round(k * 1e3, 2) for n, k in zip(names, ms)}
    if launches == len(names) - 1 and "seam" in out:
        out["seam"] = None
    return out


def per_step_us(total_ms: float, steps: int, world: int, device=None) -> float:
    """Whole-job microseconds per step: the slowest rank's timed total (a MAX
    all-reduce over the process group when world > 1) over the steps all
    ranks ran (each rank runs an independent replica of the step)."""
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms * 1e3 / (steps * world)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from mxfp8_moe_decode_gb300 import build, kernel_names
    from mxfp8_moe_decode_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    build.build()
    wl = W.WORKLOADS[args.workload]
    d = wl.dims
    peaks = measured_peaks()
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty(1, dtype=torch.int64, device=dev)

    def flush_write_only():
        flush_buf.fill_(1)

    def flush():
        # write the buffer (evicts the step's data), then read it back: L2 is
        # left holding clean lines of this buffer only
        flush_buf.fill_(1)
        flush_sink.copy_(flush_buf.view(torch.int64).sum().view(1))

    layer, x, ew = make_layer(wl, dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        step_ms, kmean, unique, graph, out, replay_ms = time_layer(layer, x, dev, args.steps,
                                                                   args.warmup, flush)
    clocks = clk.summary()
    # the same step after a write-only flush (L2 full of the flush's dirty lines)
    wo_ms, _, _, _, _, _ = time_layer(layer, x, dev, max(10, args.steps // 4), args.warmup,
                                      flush_write_only)
    launches_per_step = layer.step_launches(wl.tokens)
    us_step = per_step_us(sum(step_ms), args.steps, world, dev)
    names = kernel_names()
    alg = W.algorithmic_bytes(d, unique)
    ix = names.index("experts")
    # the expert kernel streams every touched expert (w13 + w2 + their scales) once
    exp_bytes = unique * d.expert_bytes() + d.shared_bytes()
    ach = exp_bytes / (kmean[ix] * 1e-3) / 1e9
    traffic, traffic_how = ncu_traffic("experts", wl.name, exp_bytes)
    roofline = {"bound": "hbm", "kernel": "experts", "achieved": round(ach, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "traffic": traffic,
                "traffic_source": traffic_how,
                "alg_bytes_per_launch": exp_bytes,
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)"
                if peaks["source"] == "measured" else "fallback 6.8 TB/s"}
    step_gbs = alg / (us_step * 1e-6) / 1e9 if world == 1 else None

    # end to end: host (pinned) x -> device, the step, device out -> host,
    # on one stream between two events, L2 flushed before each step. Two legs:
    # the public call (MoeDecode.step -> moe_decode_step, launches enqueued
    # by the host every step) and the step's CUDA graph replayed between the
    # same copies.
    xh = x.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    cur = torch.cuda.current_stream(dev)
    xd = x  # the graph reads x's storage
    out_call = torch.empty_like(x)

    def e2e_leg(one_step) -> float:
        for _ in range(args.warmup):
            xd.copy_(xh, non_blocking=True)
            one_step()
            oh.copy_(out_call, non_blocking=True)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t = []
        for _ in range(args.steps):
            flush()
            e0.record(cur)
            xd.copy_(xh, non_blocking=True)
            one_step()
            oh.copy_(out_call, non_blocking=True)
            e1.record(cur)
            e1.synchronize()
            t.append(e0.elapsed_time(e1))
        return statistics.mean(t) * 1e3

    e2e_us = e2e_leg(lambda: layer.step(xd, out=out_call))
    if layer.status() != 0:
        raise RuntimeError(f"device status {layer.status()}")
    got_call = out_call.clone()

    def graph_step():
        graph.replay()
        out_call.copy_(out, non_blocking=True)

    e2e_graph_us = e2e_leg(graph_step)
    if not torch.equal(out_call, got_call):
        raise RuntimeError("graph replay and the direct call disagree")
    cpu_ref = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu_ref = cpu_baseline(wl, ew, unique, args.cpu_experts)

    sweep, next_rows = {}, {}
    if not args.no_sweep and world == 1:
        layer.close()
        del layer, graph
        torch.cuda.empty_cache()
        prev_seed, prev_ew = wl.seed, ew
        for name in SWEEP + NEXT_ROWS:
            swl = W.WORKLOADS[name]
            reuse = prev_ew if (swl.seed == prev_seed and swl.dims == d) else None
            if reuse is None:
                prev_ew = None
                torch.cuda.empty_cache()
            L2, x2, ew2 = make_layer(swl, dev, ew=reuse)
            ms, km, u2, g2, _, rms = time_layer(L2, x2, dev, max(5, args.steps // 2), 3, flush)
            del g2
            us2 = statistics.mean(ms) * 1e3
            a2 = W.algorithmic_bytes(swl.dims, u2)
            e2 = u2 * swl.dims.expert_bytes() + swl.dims.shared_bytes()
            (sweep if name in SWEEP else next_rows)[name] = {
                           "M": swl.tokens, "experts": swl.dims.experts, "us_per_step": round(us2, 2),
                           "replay_us_per_step": round(statistics.mean(rms) * 1e3, 2),
                           "unique_routed": u2, "alg_bytes": a2,
                           "step_gbs": round(a2 / (us2 * 1e-6) / 1e9, 1),
                           "step_frac": round(a2 / (us2 * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                           "step_frac_of_8tbs": round(a2 / (us2 * 1e-6) / 1e9 / NOMINAL_GBS, 4),
                           "experts_gbs": round(e2 / (km[ix] * 1e-3) / 1e9, 1),
                           "kernel_us": kernel_table(names, km, L2.step_launches(swl.tokens))}
            L2.close()
            del L2
            prev_seed, prev_ew = swl.seed, ew2
        del prev_ew
        torch.cuda.empty_cache()
        next_rows["attn_seam_x8"] = time_attn_seam(W.WORKLOADS[DEFAULT_WORKLOAD], dev, flush,
                                                   max(10, args.steps // 2))

    line = {
        "metric": METRIC,
        "value": round(us_step, 3),
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_step / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (mxfp8 block-scaled MMA, fp32 accumulate)",
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {**base_config(wl, unique),
                   "step_gbs": round(step_gbs, 1) if step_gbs else None,
                   "step_frac_of_peak": round(step_gbs / peaks["hbm_gbs"], 4) if step_gbs else None,
                   "step_frac_of_8tbs": round(step_gbs / NOMINAL_GBS, 4) if step_gbs else None,
                   "median_us_per_step": round(statistics.median(step_ms) * 1e3, 3),
                   "l2": "flushed before every timed step: a 512 MB buffer written, then read "
                         "back (none of the step's data in L2, no dirty lines); weights > L2",
                   "us_per_step_after_write_only_flush": round(statistics.mean(wo_ms) * 1e3, 3),
                   "timing": "CUDA-graph replay; the step is timed by event nodes inside its graph "
                             "just before its first kernel and after its last (replay_us_per_step: the "
                             "same graph between stream events, graph launch latency included); "
                             "kernel_us from a graph with event nodes between kernels",
                   "replay_us_per_step": round(statistics.mean(replay_ms) * 1e3, 3),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "kernel_us": kernel_table(names, kmean, launches_per_step),
        "e2e": {"value": round(e2e_us, 3), "unit": "us",
                "h2d_bytes_per_step": xh.numel() * 2, "d2h_bytes_per_step": oh.numel() * 2,
                "method": "per step: pinned host x -> device copy, the public call "
                          "(MoeDecode.step -> moe_decode_step, its launches enqueued by the "
                          "host), device out -> pinned host copy; one stream, CUDA events "
                          "around the three, L2 flushed before each step",
                "graph_replay_value": round(e2e_graph_us, 3),
                "graph_replay_method": "the same copies around a replay of the step's "
                                       "CUDA graph (captured from the same call)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if sweep:
        line["sweep"] = sweep
    if next_rows:
        line["next_rows"] = next_rows
    if cpu_ref is not None:
        line["cpu_baseline"] = cpu_ref
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- CPU oracle
_CPU_WEIGHTS: dict = {}


def blas_threads() -> str:
    """The numpy BLAS thread count the oracle runs with (threadpoolctl where
    installed, else the usual environment variables, else the library default)."""
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return str(n[0])
    except Exception:  # noqa: BLE001 - optional package
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v):
            return os.environ[v]
    return "library default"


def _host_expert_getters(wl, ew_host):
    """Oracle accessors over host copies of the layer's weight tensors."""
    from oracle import moe as O

    make = O.ExpertWeights.from_fp4 if wl.dims.routed == "e2m1" else O.ExpertWeights.from_quantised

    def get_expert(e):
        return make(ew_host["w13"][e].numpy(), ew_host["w13_s"][e].numpy(),
                    ew_host["w2"][e].numpy(), ew_host["w2_s"][e].numpy())

    def get_shared():
        return O.ExpertWeights.from_quantised(ew_host["sw13"].numpy(), ew_host["sw13_s"].numpy(),
                                              ew_host["sw2"].numpy(), ew_host["sw2_s"].numpy())

    return get_expert, get_shared


def oracle_step(wl, ew_host):
    """One complete oracle step of the workload on the host: the seam and the
    router on all M rows, every touched routed expert and the shared expert
    over their rows, the combine. Returns (seconds, unique routed experts)."""
    from mxfp8_moe_decode_gb300 import workloads as W
    from oracle import moe as O

    d = wl.dims
    ri = W.router_inputs(wl)
    f64 = lambda t: t.float().double().numpy()  # noqa: E731
    x, nw, gw, b = f64(W.token_rows(wl)), f64(ri["norm_w"]), f64(ri["gate_w"]), f64(ri["bias"])
    get_expert, get_shared = _host_expert_getters(wl, ew_host)
    t0 = time.perf_counter()
    res = O.decode_step(x, nw, gw, b, d.topk, get_expert, get_shared, d.eps)
    dt = time.perf_counter() - t0
    return dt, len(set(res.routing.ids.reshape(-1).tolist()))


def cpu_baseline(wl, ew, unique: int, n_sample: int = 4) -> dict:
    """The oracle, as it stands, on the host cores: one complete step of the
    workload (value), on host copies of the weights the GPU step ran on (the
    copies are not timed); beside it, the older sampled estimate (the expert
    path of n_sample touched experts scaled to all of them), labelled."""
    ew_host = {k: v.cpu() for k, v in ew.items()}
    dt, u = oracle_step(wl, ew_host)
    line = {"value": round(dt * 1e6, 1), "unit": "us", "cores": len(os.sched_getaffinity(0)),
            "blas_threads": blas_threads(), "kind": "oracle",
            "sample": f"one complete oracle step of {wl.name}: {wl.tokens} rows, {u} touched "
                      f"routed experts + the shared one, fp64 (timed once; no scaling)"}
    if u != unique:
        line["note"] = f"oracle touched {u} routed experts, the GPU step {unique}"
    if n_sample > 0:
        # the older estimate: the expert path (dequantise + contraction) of the
        # first n_sample touched experts over their own rows, scaled to all
        import numpy as np

        from mxfp8_moe_decode_gb300 import workloads as W
        from oracle import moe as O
        from oracle.mx import dequant_rows

        d = wl.dims
        ri = W.router_inputs(wl)
        f64 = lambda t: t.float().double().numpy()  # noqa: E731
        x = f64(W.token_rows(wl))
        normed = O.rmsnorm(x, f64(ri["norm_w"]), d.eps)
        x_hat = dequant_rows(*O.seam_quant(normed))
        rt = O.router(normed, f64(ri["gate_w"]), f64(ri["bias"]), d.topk)
        get_expert, _ = _host_expert_getters(wl, ew_host)
        sample = [int(e) for e in np.unique(rt.ids)[:n_sample]]
        t = 0.0
        for e in sample:
            rows = [r for r in range(x.shape[0]) if e in rt.ids[r]]
            t1 = time.perf_counter()
            O.expert(x_hat[rows], get_expert(e))
            t += time.perf_counter() - t1
        line["sampled_estimate_us"] = round(t / max(1, len(sample)) * (unique + 1) * 1e6, 1)
        line["sampled_estimate"] = (f"expert path of {len(sample)} touched experts over their "
                                    f"rows, scaled to {unique} + 1 experts (an estimate)")
    del ew_host
    return line


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, complete steps of
    the same workload. Each step takes seconds to tens of seconds, so the arm
    runs as many of the requested steps as fit a fixed budget (at least one,
    after one warm-up step) and prints the counts it ran."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    from mxfp8_moe_decode_gb300 import workloads as W

    wl = W.WORKLOADS[args.workload]
    # inputs: the weights drawn exactly as the GPU arm draws them (on the GPU
    # when there is one), then held in host memory; not timed
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    ew = W.expert_weights(wl, device=dev)
    ew_host = {k: v.cpu() for k, v in ew.items()}
    del ew
    if dev != "cpu":
        torch.cuda.empty_cache()
    budget_s = float(os.environ.get("MOE_REFERENCE_BUDGET_S", "150"))
    warm = 0
    t_warm = None
    if args.warmup > 0:
        t_warm, _ = oracle_step(wl, ew_host)
        warm = 1
    n = args.steps
    if t_warm is not None:
        n = max(1, min(args.steps, int(budget_s // max(t_warm, 1e-9))))
    vals, unique = [], 0
    for _ in range(n):
        dt, unique = oracle_step(wl, ew_host)
        vals.append(dt)
    v = statistics.mean(vals) * 1e6
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 1),
        "unit": "us",
        "n_gpus": world,
        "steps": n,
        "warmup": warm,
        "requested": {"steps": args.steps, "warmup": args.warmup},
        "ms_per_step": round(v / 1e3, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; the same draws as the GPU arm)",
        "config": base_config(wl, unique),
        "cpu_baseline": {"value": round(v, 1), "unit": "us", "cores": len(os.sched_getaffinity(0)),
                         "blas_threads": blas_threads(), "kind": "oracle",
                         "sample": f"complete oracle steps of {wl.name} ({wl.tokens} rows, "
                                   f"{unique} routed + 1 shared experts, fp64); {warm} warm-up "
                                   f"and {n} timed of the {args.steps} requested, as many as "
                                   f"fit {budget_s:.0f} s"},
        "e2e": {"value": round(v, 1), "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
