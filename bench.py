#!/usr/bin/env python
"""Throughput of exact tensor-network contraction on one GB300.

One step = one full tn_execute of the workload (every slice, every tree
step, the leaf permutations) on inputs already resident in HBM.  The metric
is the effective rate C_t / time, C_t = sum over nodes of 8 m n k (times the
slice count).  Prints one JSON line.

  python bench.py [--workload circuit_7x7_d10] [--steps K] [--warmup W] [--gpus N]
  python bench.py --impl reference ...   # the fp64 CPU oracle on this host

With torchrun (N > 1): a sliced workload is split over the ranks by slices
(round robin; each step ends with one sum of the small output over the
ranks) and the value is C_t over the slowest rank's time (strong scaling);
an unsliced one runs one replica per rank (no collective on the data path)
and the value is the total over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective contraction TFLOP/s (C_t/time) on 1 GB300; % of 3xTF32 tensor peak"
L2_BYTES = 129 * 1024 * 1024

# Kernel whose peak bounds a precision's tensor-core nodes.
PRECISION_KERNEL = {"tf32x3": "dense_tf32x3", "bf16": "dense_bf16", "bf16x3": "dense_bf16x3",
                    "fp32": "simt"}

# Nominal ratios and unit counts used where a peak is derived rather than
# measured: tf32 dense is half the bf16 dense rate on this part; fp32 FMA
# on CUDA cores = 152 SMs x 128 lanes x 2 flops x clock.
TF32_PER_BF16 = 1.1 / 2.25
SMS, FP32_LANES = 152, 128


def peaks():
    """HBM copy bandwidth and bf16 tensor rates: the measured figures of
    MEASURED_PEAKS.json (burst = a GEMM timed alone, sustained = back to
    back for seconds under the power cap), else one earlier GB300
    measurement (fallback)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


# A timed region at least this long runs the tensor cores under the power
# cap: its kernels are compared with the sustained bf16 figure.
SUSTAINED_AFTER_S = 2.0


def kernel_peak(kernel: str, pk, sustained: bool = False):
    """(bound, peak, unit, note) for a kernel name of the launch records."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    kind = "sustained" if sustained else "burst"
    bf16 = pk[key]
    if kernel in ("dense_tf32x3", "dense_tf32x3_3p"):
        tf32 = bf16 * TF32_PER_BF16
        return "tensor", tf32 / 3.0, "TFLOP/s", (f"3xTF32-effective = bf16 {kind} {pk['source']} x "
                                                 f"{TF32_PER_BF16:.3f} / 3")
    if kernel == "dense_bf16":
        return "tensor", bf16, "TFLOP/s", f"bf16 dense, {kind} {pk['source']}"
    if kernel == "dense_bf16x3":
        return "tensor", bf16 / 3.0, "TFLOP/s", f"split-bf16-effective = bf16 {kind} {pk['source']} / 3"
    if kernel in ("simt", "tiny"):
        alu = SMS * FP32_LANES * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
        return "alu", alu, "TFLOP/s", "fp32 FMA: 152 SMs x 128 lanes x 2 x max SM clock"
    return "hbm", pk["hbm_gbs"], "GB/s", f"copy bandwidth, {pk['source']}"


# Sources whose digest identifies a kernel's build in the traffic table.
KERNEL_SOURCES = {
    "dense_tf32x3": ["k_dense.cu", "common.cuh", "kernels.h", "plan.h"],
    "dense_bf16": ["k_dense.cu", "common.cuh", "kernels.h", "plan.h"],
    "dense_bf16x3": ["k_dense.cu", "common.cuh", "kernels.h", "plan.h"],
    "permute": ["k_permute.cu", "common.cuh", "kernels.h", "plan.h"],
    "stream": ["k_stream.cu", "common.cuh", "kernels.h", "plan.h"],
}
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def kernel_digest(kernel: str):
    import hashlib
    srcs = KERNEL_SOURCES.get(kernel)
    if not srcs:
        return None
    h = hashlib.sha1()
    for f in srcs:
        with open(os.path.join(ROOT, "exact_tensor_network_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per
    launch of `kernel` on `workload`, from the traffic table, when the
    kernel's sources still have the digest the counters were taken with;
    else None.  Returns (bytes, how the figure was obtained)."""
    sha = kernel_digest(kernel)
    if sha is None or not os.path.exists(TRAFFIC_TABLE):
        return None, None
    with open(TRAFFIC_TABLE) as fh:
        table = json.load(fh)
    for e in table.get("entries", []):
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("sources") == sha:
            return float(e["bytes_per_launch"]), e.get("method")
    return None, None


def network_roofline(plan, records, flops_peak_tflops: float, hbm_gbs: float):
    """The pages' per-step time model, max(flops / F, bytes / B), summed over
    the launches of one execute (every slice; hoisted launches are counted
    once, as they run).  Node launches take the node's complex64 algorithmic
    bytes 8 (mk + nk + mn); batched tiny launches and leaf permutations the
    bytes of their records (the same rule, and 16 per leaf entry); split-K
    reductions are part of their node and add nothing.  Returns seconds."""
    F = flops_peak_tflops * 1e12
    B = hbm_gbs * 1e9
    mnk = {}
    t = 0.0
    for r in records:
        if r["kernel"] == "reduce":
            continue
        if r["step"] >= 0:
            if r["step"] not in mnk:
                mnk[r["step"]] = plan.node_mnk(r["step"])
            m, n, k = mnk[r["step"]]
            flops, nbytes = 8 * m * n * k, 8 * (m * k + n * k + m * n)
        else:
            flops, nbytes = r["flops"], r["bytes"]
        t += max(flops / F, nbytes / B)
    return t


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
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
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def load_workload(name: str, with_data: bool = True):
    from workloads import configs
    return configs.by_name(name, with_data=with_data)


def oracle_rate(net, tree, slices, min_seconds: float, max_runs: int):
    """Run the oracle on the full workload until min_seconds have passed
    (at least once); return (flops per second, runs, seconds, threads)."""
    import oracle
    from oracle import planner
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, slices)
    runs, t0 = 0, time.perf_counter()
    while True:
        if slices:
            oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree, slices)
        else:
            oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
        runs += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or runs >= max_runs:
            break
    return p.C_t_total * runs / el, runs, el, oracle.num_threads(), p.C_t_total


ORACLE_FULL_LIMIT = 1.5e12   # flops the oracle runs in full (tens of seconds at most)


def oracle_subtree_sample(net, tree, slices, budget: float, max_seconds: float = float("inf")):
    """The oracle on whole subtrees of the workload's own tree (slice 0),
    largest first, until `budget` flops are covered or `max_seconds` have
    passed.  Returns (flops, seconds, number of subtrees, threads)."""
    import oracle
    from oracle import planner
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, slices)
    n = net.n_tensors
    cost = {t: 0 for t in range(n)}
    kids = {}
    for nd in p.nodes:
        cost[nd.out] = nd.flops + cost[nd.a] + cost[nd.b]
        kids[nd.out] = (nd.a, nd.b)
    root = n + len(tree) - 1
    chosen, left, frontier = [], budget, [root]
    while frontier and left > 0:
        frontier.sort(key=lambda x: cost[x])
        x = frontier.pop()
        if x < n or cost[x] == 0:
            continue
        if cost[x] <= left:
            chosen.append(x)
            left -= cost[x]
        else:
            frontier.extend(kids[x])
    modes = planner.tensor_modes(net.tensors, tree, slices)
    leaves_t, leaves_d = oracle.slice_leaves(net.tensors, net.data, slices, [0] * len(slices))
    flops, secs = 0, 0.0
    if not chosen:
        # not even one subtree fits: contract one block of the output
        # instead, fixing leading open modes at index 0
        from workloads.trees import step_volume
        fixed = []
        for x in net.open_modes:
            if 8 * step_volume(net, tree, exclude=list(slices) + fixed) <= budget:
                break
            fixed.append(x)
        cost_b = 8 * step_volume(net, tree, exclude=list(slices) + fixed)
        t2, d2 = oracle.slice_leaves(leaves_t, leaves_d, fixed, [0] * len(fixed))
        t0 = time.perf_counter()
        oracle.contract(t2, net.extents, [x for x in net.open_modes if x not in fixed], d2, tree)
        return cost_b, time.perf_counter() - t0, 1, oracle.num_threads()
    done = 0
    for x in chosen:
        if secs >= max_seconds:
            break
        done += 1
        sub_leaves, steps = [], []

        def walk(y):
            if y < n:
                sub_leaves.append(y)
                return
            walk(kids[y][0])
            walk(kids[y][1])
            steps.append(y)
        walk(x)
        ids = {y: i for i, y in enumerate(sub_leaves)}
        pairs = []
        for y in sorted(steps):
            a, b = kids[y]
            pairs.append((ids[a], ids[b]))
            ids[y] = len(sub_leaves) + len(pairs) - 1
        t0 = time.perf_counter()
        oracle.contract([leaves_t[y] for y in sub_leaves], net.extents, modes[x],
                        [leaves_d[y] for y in sub_leaves], pairs)
        secs += time.perf_counter() - t0
        flops += cost[x]
    return flops, secs, done, oracle.num_threads()


def subtree_budget(net, tree, slices, seconds: float):
    """Flops of whole subtrees the oracle covers in about `seconds`: its
    rate on this tree's subtrees measured on a first sample of ~1e10 flops."""
    f, s, _, _ = oracle_subtree_sample(net, tree, slices, 1e10)
    rate = f / max(s, 1e-3)
    return min(5e11, max(1e9, rate * seconds))


def cpu_baseline_leg(net, tree, slices, seconds: float):
    """fp64 oracle rate on this workload: full contractions when they fit
    in a few tens of seconds, else whole subtrees of its tree."""
    from oracle import planner
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, slices)
    if p.C_t_total <= ORACLE_FULL_LIMIT:
        rate, runs, el, threads, _ = oracle_rate(net, tree, slices, seconds, 50)
        return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": f"{runs} full fp64 oracle contraction(s) of {net.name} ({el:.1f} s)"}
    budget = subtree_budget(net, tree, slices, seconds)
    flops, secs, nsub, threads = oracle_subtree_sample(net, tree, slices, budget, seconds)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": (f"fp64 oracle on {nsub} whole subtrees of {net.name}'s tree "
                       f"({flops:.3e} flop = {100 * flops / p.C_t_total:.2g}% of C_t, {secs:.1f} s)")}


def run_reference(args, rank: int):
    if rank != 0:
        return
    net, tree, slices = load_workload(args.workload)
    import oracle
    from oracle import planner
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, slices)

    full = p.C_t_total <= ORACLE_FULL_LIMIT
    # a step is the full contraction when the oracle can do it in seconds,
    # else whole subtrees of the workload's tree, sized from the oracle's
    # measured rate so that all warm-up and timed steps take about 150 s
    per_step = 150.0 / max(1, args.steps + args.warmup)
    budget = 0.0 if full else subtree_budget(net, tree, slices, per_step)

    def one():
        if full:
            t0 = time.perf_counter()
            if slices:
                oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree,
                                       slices)
            else:
                oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
            return p.C_t_total, time.perf_counter() - t0
        f, s, _, _ = oracle_subtree_sample(net, tree, slices, budget, per_step)
        return f, s

    for _ in range(args.warmup):
        one()
    flops, el = 0, 0.0
    for _ in range(args.steps):
        f, s = one()
        flops += f
        el += s
    value = flops / el / 1e12
    cores = oracle.num_threads()
    sample = (f"full fp64 oracle contraction of {net.name} per step" if full else
              f"fp64 oracle on whole subtrees of {net.name}'s tree, {flops / args.steps:.3e} "
              f"flop per step ({100 * flops / args.steps / p.C_t_total:.2g}% of C_t)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "c128", "data": "synthetic",
            "config": {"workload": net.name, "C_t": p.C_t_total, "C_s": p.C_s,
                       "slices": p.n_slices},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch
    import exact_tensor_network_gb300 as tn
    from exact_tensor_network_gb300 import build as tnbuild

    tnbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    device_leaves = args.leaves == "device"
    net, tree, slices = load_workload(args.workload, with_data=not device_leaves)
    plan = tn.Plan.from_network(net, tree, slices, args.precision)
    if args.cta_pairs:
        plan.set_cta_pairs(True)
    if args.promotion_chunk:
        plan.set_promotion_chunk(args.promotion_chunk)
    plan.bind_workspace(dev)
    if device_leaves:
        # seeded N(0, 1) complex entries drawn on the device (no host copy:
        # single nodes of tens of GiB)
        gen = torch.Generator(device=dev)
        gen.manual_seed(1234)
        leaves = [torch.randn([net.extents[x] for x in t], dtype=torch.complex64, device=dev,
                              generator=gen).mul_(2 ** 0.5) for t in net.tensors]
    else:
        leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev)
    ct = plan.flops
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    dist = world > 1

    def barrier():
        if dist:
            torch.distributed.barrier()

    # Sliced networks are split over ranks by slices (independent
    # sub-contractions; one sum of the small output per step); other
    # networks run one replica per rank.
    sharded = dist and plan.num_slices > 1
    first, step_, _ = tn.shard_slices(plan.num_slices, rank, world)

    def one_step(lv, o):
        if sharded:
            plan.execute_slices(lv, o, first, step_, stream)
            torch.distributed.all_reduce(torch.view_as_real(o), op=torch.distributed.ReduceOp.SUM)
        else:
            plan.execute(lv, o, stream)

    units = ct if sharded else ct * world   # flops all ranks together complete per step
    # slicing's FLOP overhead: C_t over all slices against the unsliced
    # network's C_t (the same tree; planned on the host only)
    ct_unsliced = ct
    if slices:
        h = tn.tn_plan(net.tensors, net.extents, net.open_modes, tree, (), tn.PRECISIONS[args.precision])
        try:
            ct_unsliced = tn.tn_plan_flops(h)
        finally:
            tn.tn_plan_destroy(h)

    for _ in range(args.warmup):
        one_step(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)          # evict L2 between steps (untimed)
            starts[i].record(stream)
            one_step(leaves, out)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    plan.check()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    if dist:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    value = units * args.steps / (ms / 1e3) / 1e12

    # Per-launch device times (a second pass of a few of the same steps with
    # CUDA events around every launch, on the launching stream).
    plan.set_profiling(True)
    agg = {}
    records = []
    prof_steps = min(args.steps, 3)
    # a spin kernel ahead of each profiled step keeps the GPU busy while the
    # host enqueues every launch, so the events time launches back to back
    # (device time) rather than host submission gaps
    sleep_cycles = int(2.0e9 * (0.002 + 50e-6 * plan.launches))
    for i in range(prof_steps):
        flush.fill_(i & 0xFF)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(sleep_cycles)
        plan.execute(leaves, out, stream)
        torch.cuda.synchronize(dev)
        records = plan.profile()
        for r in records:
            a = agg.setdefault(r["kernel"], {"ms": 0.0, "flops": 0, "bytes": 0, "launches": 0})
            a["ms"] += r["ms"]
            a["flops"] += r["flops"]
            a["bytes"] += r["bytes"]
            a["launches"] += 1
    plan.set_profiling(False)
    plan.check()
    pk = peaks()
    # a seconds-long timed region runs under the power cap: sustained peak
    sustained = ms / 1e3 >= SUSTAINED_AFTER_S
    dom = max(agg, key=lambda k: agg[k]["ms"])
    bound, peak, unit, note = kernel_peak(dom, pk, sustained)
    d = agg[dom]
    if unit == "TFLOP/s":
        achieved = d["flops"] / (d["ms"] / 1e3) / 1e12
    else:
        achieved = d["bytes"] / (d["ms"] / 1e3) / 1e9
    per_launch = d["flops" if unit == "TFLOP/s" else "bytes"] / d["launches"]
    traffic, traffic_method = measured_traffic(dom, net.name)
    # the whole step against the pages' cost model at the precision's
    # tensor peak and the HBM bandwidth
    _, net_peak, net_unit, net_note = kernel_peak(PRECISION_KERNEL[args.precision], pk, sustained)
    t_roof = network_roofline(plan, records, net_peak, pk["hbm_gbs"])
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic,
                "traffic_unit": "bytes per launch (ncu dram read + write)",
                "traffic_method": traffic_method,
                "peak_note": note + " (of " + pk["source"] + ")",
                "peak_kind": "sustained" if sustained else "burst",
                "algorithmic_per_launch": per_launch,
                "avg_launch_ms": d["ms"] / d["launches"],
                "network_frac": t_roof / (ms / args.steps / 1e3),
                "network_roof_ms": t_roof * 1e3,
                "network_note": ("sum over one execute's launches of max(flops / F, bytes / B), "
                                 f"F = {net_peak:.1f} {net_unit} ({net_note}), "
                                 f"B = {pk['hbm_gbs']:.0f} GB/s; divided by ms_per_step")}
    kernels = {k: {"ms_per_step": v["ms"] / prof_steps, "launches_per_step": v["launches"] / prof_steps,
                   "share": v["ms"] / sum(x["ms"] for x in agg.values())}
               for k, v in agg.items()}
    executed = sum(r["flops"] for r in records)
    cfg_extra = {"C_t_unsliced": ct_unsliced, "flop_overhead": ct / ct_unsliced,
                 "flops_executed": executed,
                 "hoisting": ("on: later slices rerun only launches below a sliced leaf"
                              if plan.num_slices > 1 else "no slices")}

    # End to end through the public API with host buffers: pinned host
    # leaves copied in, contraction, result copied out, every step.
    if device_leaves:
        e2e_none = {"value": None, "unit": "TFLOP/s", "note": "leaves drawn on the device"}
        return finish(args, rank, world, net, plan, ct, units, value, ms, sharded, roofline, kernels,
                      e2e_none, None, clk, cfg_extra)
    host_leaves = [torch.from_numpy(np.ascontiguousarray(d)).pin_memory() for d in net.data]
    host_out = torch.empty(plan.out_shape, dtype=torch.complex64).pin_memory()
    dev_leaves = [torch.empty_like(h, device=dev) for h in host_leaves]
    h2d = sum(h.numel() * 8 for h in host_leaves)
    d2h = host_out.numel() * 8

    # the public call with host buffers, prepared once for these buffers
    host_call = None if sharded else plan.prepare_host(host_leaves, host_out, dev_leaves, out, stream)

    def e2e_step():
        if not sharded:
            host_call()
            return
        with torch.cuda.stream(stream):
            for d, h in zip(dev_leaves, host_leaves):
                d.copy_(h, non_blocking=True)
            one_step(dev_leaves, out)
            host_out.copy_(out, non_blocking=True)
        stream.synchronize()
    for _ in range(2):   # the first call records the whole call as a graph
        e2e_step()
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    if dist:
        t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e = {"value": units * args.steps / e2e_s / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(net, tree, slices, args.cpu_seconds)
    finish(args, rank, world, net, plan, ct, units, value, ms, sharded, roofline, kernels, e2e, cpu,
           clk, cfg_extra)


def finish(args, rank, world, net, plan, ct, units, value, ms, sharded, roofline, kernels, e2e, cpu,
           clk, cfg_extra):
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "strong" if sharded else "weak",
                "vs_baseline": None, "dtype": "c64",
                "data": "synthetic" + (" (leaves drawn on the device)" if args.leaves == "device" else ""),
                "config": {"workload": net.name, "tensors": net.n_tensors, "C_t": ct,
                           "C_s": plan.peak, "slices": plan.num_slices, "precision": args.precision,
                           "cta_pairs": bool(args.cta_pairs),
                           "promotion_chunk": args.promotion_chunk or "per plan",
                           "l2": "flushed between timed steps (untimed 258 MiB fill)",
                           "parallelism": (f"slices round-robin over {world} ranks" if sharded
                                           else f"replicas x{world}"), **cfg_extra},
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": plan.launches * args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="circuit_7x7_d10",
                    help="circuit_7x7_d10 (default: the largest, sliced), circuit_6x6_d12, "
                         "random_60, circuit_3x3_d4, gemm_mX_nY_kZ")
    ap.add_argument("--precision", default="tf32x3", choices=["tf32x3", "bf16", "bf16x3", "fp32"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cta-pairs", action="store_true",
                    help="tensor-core nodes on CTA pairs (tn_plan_set_cta_pairs)")
    ap.add_argument("--promotion-chunk", type=int, default=0,
                    help="complex k per TMEM promotion (tn_plan_set_promotion_chunk; 0: per plan)")
    ap.add_argument("--leaves", choices=["host", "device"], default="host",
                    help="device: draw the leaves on the GPU (no end-to-end or CPU leg)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
