"""Benchmark: 16-layer q8 verification attention over a paged E4M3 KV cache on one GB300.

A step is one pass of the whole path (16 layers x [partial attention + combine]) over the
workload's resident inputs, replayed from one CUDA graph; each kernel is launched as a programmatic
dependent of the kernel before it (it starts while that one drains and waits for it before reading
Q or writing anything; `--pdl off`: plain stream order, which the line also reports). Default
workload: 16 layers, batch 1,
q_len 8, Hq 6, Hkv 1, D 256, context 261888 (the capacity boundary window), page 16, shuffled
block tables, 2.15 GB of distinct E4M3 K/V per step (far larger than L2, so no flush is needed;
smaller workloads get a 512 MB L2 flush between timed steps).

Prints one JSON line (rank 0). `--impl reference` times the FP64 CPU oracle instead, on a bounded
sample of the same workload, scaled to the same unit.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "16-layer q8 verify-attention ms at 32K-262K ctx; achieved HBM GB/s vs peak"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, about 8 TB/s
TARGET_FRAC = 0.70  # the 16-layer step at 261888 tokens is to run at >= 70 % of the HBM roofline
PROFILES = os.path.join(ROOT, "profiles")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c3",
                    help="c0|c1|c2|c3|c4:<q_len>:<context>|c5|c6:<batch>:<context>")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tcgen05")
    ap.add_argument("--splits", type=int, default=0, help="force the split count (0: planner)")
    ap.add_argument("--layers", type=int, default=0,
                    help="time only the first L layers (profiling captures; 0: all)")
    ap.add_argument("--fused-combine", action="store_true",
                    help="merge the splits inside the partial launch (one kernel per layer)")
    ap.add_argument("--pdl", choices=["on", "off"], default="on",
                    help="launch the kernels as programmatic dependents of the preceding kernel "
                         "(on: the step line also reports the same step in plain stream order)")
    ap.add_argument("--l2", choices=["auto", "warm"], default="auto",
                    help="auto: flush L2 (512 MB write) between timed steps when the workload's "
                         "KV is under 4x L2; warm: never flush (cache-resident small workloads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--time-oracle-layer", type=int, default=-1, help=argparse.SUPPRESS)
    return ap.parse_args()


def workload(name):
    from speculative_verify_paged_e4m3_gb300 import workload as W
    if name.startswith("c4"):
        _, q, n = name.split(":")
        return W.config4(int(q), int(n))
    if name.startswith("c6"):
        _, bsz, n = name.split(":")
        return W.config6(int(bsz), int(n))
    return {"c0": W.config0, "c1": W.config1, "c2": W.config2, "c3": W.config3,
            "c5": W.config5}[name]()


def measured_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_verify_paged_e4m3_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_tag, workload_name, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    path = os.path.join(PROFILES, f"{kernel_tag}_{workload_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hm = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not hm or hm.group(1) != src_hash:
        return None
    return float(m.group(1))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        try:
            lines = open(self.path).read().strip().splitlines()
        except OSError:
            lines = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_ms_per_step(w, layers_sample, rows_note, steps=1):
    """Time the FP64 oracle on whole sample layers; scale to ms per len(w.layers) layers."""
    import numpy as np

    import oracle
    from speculative_verify_paged_e4m3_gb300 import workload as W
    orc = oracle.load()
    data = [W.make_layer(w, l, device="cpu") for l in layers_sample]
    args = [(d["q"].numpy(), d["k_pool"].numpy(), d["v_pool"].numpy(), d["block_table"].numpy(),
             d["context_lens"].numpy(), float(d["k_scale"].item()), float(d["v_scale"].item()))
            for d in data]
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        for a in args:
            orc.verify_attn(*a)
        times.append(time.perf_counter() - t0)
    per_layer = statistics.median(times) / len(layers_sample)
    return per_layer * w.layers * 1e3, orc.num_threads(), times


def max_over_ranks(value, world, device):
    """Largest value over the ranks of the process group (the job is as slow as its slowest
    rank); works for NCCL (CUDA tensors) and gloo (CPU tensors)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one whole layer of the workload (all query
    rows, every key) through the FP64 oracle, layers 0 and 1 taken in turn. ms_per_step is that
    measured time; value is the 16-layer figure of the metric, ms_per_step x layers (declared in
    layers_per_step and value_is)."""
    w = workload(args.config)
    if rank != 0:
        return
    total_steps = args.warmup + args.steps
    import oracle
    from speculative_verify_paged_e4m3_gb300 import workload as W
    orc = oracle.load()
    sample_layers = list(range(min(2, w.layers)))
    args_by_layer = []
    for lay in sample_layers:
        d = W.make_layer(w, lay, device="cpu")
        args_by_layer.append((d["q"].numpy(), d["k_pool"].numpy(), d["v_pool"].numpy(),
                              d["block_table"].numpy(), d["context_lens"].numpy(),
                              float(d["k_scale"].item()), float(d["v_scale"].item())))
    times = []
    for s in range(total_steps):
        a = args_by_layer[s % len(args_by_layer)]
        t0 = time.perf_counter()
        orc.verify_attn(*a)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt * 1e3)
    step_ms = statistics.mean(times)
    ms = step_ms * w.layers
    sample = (f"each step: one layer of {w.name} (layers {sample_layers} in turn; all "
              f"{w.q_len * w.num_q_heads} query rows, {w.context[0]} keys) through the oracle; "
              f"value = ms_per_step x {w.layers} layers")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(ms, 3), "unit": "ms",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 3), "layers_per_step": 1,
        "value_is": f"ms_per_step x {w.layers} (one of the {w.layers} layers per step)",
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "layers": w.layers},
        "cpu_baseline": {"value": round(ms, 3), "unit": "ms", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(ms, 3), "unit": "ms", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_oracle_layer(config, layer):
    """ms of one whole layer through the oracle in this process (run in a child process with
    OMP_NUM_THREADS=1 for the one-thread figure)."""
    import oracle
    from speculative_verify_paged_e4m3_gb300 import workload as W
    w = workload(config)
    d = W.make_layer(w, layer, device="cpu")
    a = (d["q"].numpy(), d["k_pool"].numpy(), d["v_pool"].numpy(), d["block_table"].numpy(),
         d["context_lens"].numpy(), float(d["k_scale"].item()), float(d["v_scale"].item()))
    orc = oracle.load()
    t0 = time.perf_counter()
    orc.verify_attn(*a)
    return (time.perf_counter() - t0) * 1e3, orc.num_threads()


def oracle_one_thread_ms(config, layer):
    """The oracle on one host thread: one layer timed in a child process."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--config", config,
                        "--time-oracle-layer", str(layer)], env=env, capture_output=True,
                       text=True, timeout=600)
    if r.returncode != 0:
        return None
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return out["ms"], out["threads"]


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from speculative_verify_paged_e4m3_gb300 import binding as B
    from speculative_verify_paged_e4m3_gb300 import build as build_mod
    from speculative_verify_paged_e4m3_gb300.runner import LayerStack, algorithmic_bytes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build_mod.build()
    w = workload(args.config)
    stack = LayerStack(w, device=dev, num_splits=args.splits, kernel=args.kernel,
                       layers=args.layers or None,
                       flags=(B.DFLASH_PROBLEM_FUSED_COMBINE if args.fused_combine else 0) |
                       (B.DFLASH_PROBLEM_PDL if args.pdl == "on" else 0))
    plan = stack.plan
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if args.l2 == "auto" and w.kv_bytes_per_layer() * w.layers < 4 * l2_bytes:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stack.capture()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        stack.replay()
    barrier()

    # timed region: K graph replays, CUDA events on the replay stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    with clocks:
        barrier()
        for s in range(args.steps):
            if flush is not None:
                flush.fill_(s & 0xFF)
            starts[s].record()
            stack.replay()
            ends[s].record()
        barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)

    # kernel attribution: with the merge fused into the partial kernel, a step is one launch per
    # layer and the kernel time is the step time per layer; otherwise the same 16 partial
    # launches (and, separately, the 16 combine launches) are replayed from their own graphs,
    # CUDA events around each replay on the replay stream
    fused = bool(plan.combine_fused)
    nl = len(stack.layers)

    def timed_replays(graph):
        for _ in range(max(1, args.warmup)):
            graph.replay()
        barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for s in range(args.steps):
            if flush is not None:
                flush.fill_(s & 0xFF)
            ev[s][0].record()
            graph.replay()
            ev[s][1].record()
        barrier()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) / nl

    if fused:
        partial_ms = statistics.mean(step_ms) / nl
        combine_ms = 0.0
    else:
        g_partial, g_combine = stack.capture_kernel_graphs()
        partial_ms = timed_replays(g_partial)
        combine_ms = timed_replays(g_combine)

    # with programmatic launch, the same step in plain stream order (same layers, workspace and
    # split plan; only the launch flag differs), for comparison
    stream_order = None
    if args.pdl == "on" and not fused:
        plain = B.Plan.from_buffer_copy(plan)
        plain.problem.flags = plan.problem.flags & ~B.DFLASH_PROBLEM_PDL
        g_plain = stack._capture(lambda: stack.launch(plan=plain))
        so_ms = max_over_ranks(timed_replays(g_plain) * nl, world, dev)
        stream_order = {"ms_per_step": round(so_ms, 4),
                        "frac_of_measured": None}  # filled in below, once the peak is known

    # end to end through the public API: per step, H2D of the step's inputs from pinned host
    # memory (Q, block tables, context lengths, scales of all layers), the 16 layers, and D2H of
    # the outputs and LSEs; the KV cache stays resident (it is the model's state, not an input)
    e2e = None
    if not args.no_e2e:
        # one pinned buffer per direction: every layer's inputs (Q, block table, context length,
        # scales) go up in one copy, every layer's out and lse come back in one copy; the layer
        # tensors become views of the device-side buffers, so the forward reads and writes them
        # in place
        keys = ("q", "block_table", "context_lens", "k_scale", "v_scale")

        def layout(tensors):
            offs, total = [], 0
            for t in tensors:
                total = (total + 255) // 256 * 256
                offs.append(total)
                total += t.numel() * t.element_size()
            return offs, total

        def view(buf, off, t):
            return buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

        ins = [(lay, k) for lay in stack.layers for k in keys]
        in_offs, in_total = layout([lay[k] for lay, k in ins])
        dev_in = torch.empty(in_total, dtype=torch.uint8, device=dev)
        host_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
        for (lay, k), off in zip(ins, in_offs):
            view(host_in, off, lay[k]).copy_(lay[k].cpu())
            v = view(dev_in, off, lay[k])
            v.copy_(lay[k])
            lay[k] = v
        outs = [t for pair in zip(stack.outs, stack.lses) for t in pair]
        out_offs, out_total = layout(outs)
        dev_out = torch.empty(out_total, dtype=torch.uint8, device=dev)
        host_out = torch.empty(out_total, dtype=torch.uint8).pin_memory()
        views = [view(dev_out, off, t) for t, off in zip(outs, out_offs)]
        stack.outs, stack.lses = views[0::2], views[1::2]
        h2d, d2h = in_total, out_total

        def e2e_calls():
            dev_in.copy_(host_in, non_blocking=True)
            stack.launch()
            host_out.copy_(dev_out, non_blocking=True)

        # the step as a serving loop runs it: the copies and the 16 forward calls captured once
        # (every call is capture-safe: lengths and scales are read on the device), replayed
        e2e_graph = stack._capture(e2e_calls)

        def e2e_step():
            e2e_graph.replay()

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for s in range(args.steps):
            if flush is not None:
                flush.fill_(s & 0xFF)
            ev[s][0].record()
            e2e_step()
            ev[s][1].record()
        barrier()
        e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, dev)
        e2e = {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "how": "per step: one pinned H2D copy of every layer's inputs, the 16 forward "
                      "calls, one D2H copy of every out and lse, captured in a CUDA graph"}

    # the step before verification: the drafted tokens' K/V rows written into every layer's
    # pools (16 launches in one graph, CUDA events around replays; done last, since it rewrites
    # the drafted tokens' slots)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    kv_shape = (w.batch, w.q_len, w.num_kv_heads, w.head_dim)
    new_rows = [(torch.randn(kv_shape, generator=gen, device=dev).half(),
                 torch.randn(kv_shape, generator=gen, device=dev).half()) for _ in stack.layers]

    def launch_kv_write():
        for lay, (kn, vn) in zip(stack.layers, new_rows):
            B.dflash_verify_attn_kv_write(plan, kn, vn, lay["block_table"], lay["context_lens"],
                                          lay["k_scale"], lay["v_scale"], lay["k_pool"],
                                          lay["v_pool"], stack.att.workspace)

    kvw_ms = timed_replays(stack._capture(launch_kv_write))
    kvw_bytes = 2 * w.batch * w.q_len * w.num_kv_heads * w.head_dim * 3 + w.batch * 8
    kv_write = {"us_per_layer": round(kvw_ms * 1e3, 3), "bytes_per_layer": kvw_bytes,
                "gb_s": round(kvw_bytes / (kvw_ms * 1e-3) / 1e9, 2),
                "what": "E4M3 quantise + scatter of the q drafted tokens' K and V rows "
                        "(FP16 in, codes out), one launch per layer"}

    nbytes = algorithmic_bytes(w, plan)
    peak, peak_kind = measured_peak()
    launch_bytes = nbytes["partial"] + (nbytes["combine"] if fused else 0)
    achieved = launch_bytes / (partial_ms * 1e-3) / 1e9
    src_hash = kernel_source_hash()
    ktag = {1: "simt_partial", 2: "tc_fused" if fused else "tc_partial"}.get(plan.kernel,
                                                                           "partial")
    traffic = ncu_traffic(ktag, w.name, src_hash)
    # the 16-layer step against the roofline: every byte the step's kernels must move (K, V,
    # block tables, Q, the split state written and read back, out and lse), and the same without
    # the split state (so that more splits cannot raise the fraction)
    step_bytes = (nbytes["partial"] + nbytes["combine"]) * nl
    step_bytes_ws_free = (nbytes["kv"] + nbytes["bt"] + nbytes["q"] + nbytes["out"]) * nl
    step_gbs = step_bytes / (ms * 1e-3) / 1e9
    step_roofline = {
        "what": f"{nl}-layer step (partial + combine per layer), algorithmic bytes / step time",
        "bytes": step_bytes, "bytes_without_split_state": step_bytes_ws_free,
        "achieved_gbs": round(step_gbs, 1),
        "frac_of_measured": round(step_gbs / peak, 4),
        "frac_of_nominal_8000": round(step_gbs / NOMINAL_HBM_GBS, 4),
        "frac_without_split_state": round(step_bytes_ws_free / (ms * 1e-3) / 1e9 / peak, 4),
        "target_frac": TARGET_FRAC,
        "target_ms_at_measured_peak": round(step_bytes / (TARGET_FRAC * peak * 1e9) * 1e3, 4),
    }
    if stream_order is not None:
        stream_order["frac_of_measured"] = round(
            step_bytes / (stream_order["ms_per_step"] * 1e-3) / 1e9 / peak, 4)
    kernel_bytes_ws_free = nbytes["kv"] + nbytes["bt"] + nbytes["q"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample_layers = [0, 1]
        cms, cores, _ = oracle_ms_per_step(w, sample_layers, "all rows")
        cpu = {"value": round(cms, 1), "unit": "ms", "cores": cores, "kind": "oracle",
               "sample": f"layers {sample_layers} of {w.name}, all "
                         f"{w.q_len * w.num_q_heads} query rows, FP64 oracle; time per layer "
                         f"x {w.layers}"}
        one = oracle_one_thread_ms(args.config, 0)
        if one is not None:
            cpu["one_thread"] = {"value": round(one[0] * w.layers, 1), "unit": "ms",
                                 "cores": one[1],
                                 "sample": f"layer 0 of {w.name} on one thread (a child process "
                                           f"with OMP_NUM_THREADS=1); time x {w.layers}"}
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(ms, 4),
        "unit": "ms",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "step_ms_median": round(statistics.median(step_ms), 4),
        "step_ms_min": round(min(step_ms), 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if plan.kernel == B.DFLASH_KERNEL_SIMT else "e4m3->f32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "layers": nl, "batch": w.batch, "q_len": w.q_len,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "context": list(w.context), "page_size": w.page_size,
            "kv_gb_per_step": round(w.kv_bytes_per_layer() * w.layers / 1e9, 4),
            "l2": ("512 MB flush between timed steps" if flush is not None else
                   "warm: no flush between timed steps" if args.l2 == "warm" else
                   "inputs larger than L2 (distinct KV per layer)"),
            "kernel": ktag, "num_splits": plan.num_splits,
            "active_splits": nbytes["active_splits"],
            "timing": f"CUDA graph replay of {nl} layers",
            "launch": ("programmatic dependent launch (each kernel starts while the previous one "
                       "drains)" if args.pdl == "on" and not plan.combine_fused else
                       "stream order"),
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_kind": peak_kind, "kernel": ktag,
            "kernel_ms": round(partial_ms, 5), "bytes_per_launch": launch_bytes,
            "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
            "frac_without_split_state": (None if fused else round(
                kernel_bytes_ws_free / (partial_ms * 1e-3) / 1e9 / peak, 4)),
        },
        "step_roofline": step_roofline,
        "step_in_stream_order": stream_order,
        "step_hbm_gbs": round(step_gbs, 1),
        "step_frac_of_peak": round(step_gbs / peak, 4),
        "combine_kernel_ms": round(combine_ms, 5),
        "kv_write": kv_write,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (1 if fused else 2) * nl * args.steps,
        "kernel_timing": ("one fused launch per layer: kernel time = timed step / layers"
                          if fused else
                          "per-kernel times from graph replays of the 16 partial (or combine) "
                          "launches alone, CUDA events on the replay stream"),
        "clocks": clocks.summary(),
        "kernel_source_hash": src_hash,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.time_oracle_layer >= 0:
        ms, threads = time_oracle_layer(args.config, args.time_oracle_layer)
        print(json.dumps({"ms": ms, "threads": threads}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
