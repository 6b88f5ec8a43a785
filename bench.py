#!/usr/bin/env python
"""Throughput of exact tensor-network contraction on one GB300.

One step = one full tn_execute of the workload (every slice, every tree
step, the leaf permutations) on inputs already resident in HBM.  The metric
is the effective rate C_t / time, C_t = sum over nodes of 8 m n k (times the
slice count).  Prints one JSON line.

  python bench.py [--workload random_60] [--steps K] [--warmup W] [--gpus N]
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

# Nominal ratios and unit counts used where a peak is derived rather than
# measured: tf32 dense is half the bf16 dense rate on this part; fp32 FMA
# on CUDA cores = 152 SMs x 128 lanes x 2 flops x clock.
TF32_PER_BF16 = 1.1 / 2.25
SMS, FP32_LANES = 152, 128


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def kernel_peak(kernel: str, pk):
    """(bound, peak, unit, note) for a kernel name of the launch records."""
    if kernel == "dense_tf32x3":
        tf32 = pk["bf16_tflops"] * TF32_PER_BF16
        return "tensor", tf32 / 3.0, "TFLOP/s", f"3xTF32-effective = bf16 {pk['source']} x {TF32_PER_BF16:.3f} / 3"
    if kernel == "dense_bf16":
        return "tensor", pk["bf16_tflops"], "TFLOP/s", f"bf16 dense, {pk['source']}"
    if kernel == "dense_bf16x3":
        return "tensor", pk["bf16_tflops"] / 3.0, "TFLOP/s", f"split-bf16-effective = bf16 {pk['source']} / 3"
    if kernel in ("simt", "tiny"):
        alu = SMS * FP32_LANES * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
        return "alu", alu, "TFLOP/s", "fp32 FMA: 152 SMs x 128 lanes x 2 x max SM clock"
    return "hbm", pk["hbm_gbs"], "GB/s", f"copy bandwidth, {pk['source']}"


KERNEL_SOURCES = {
    "dense_tf32x3": ["k_dense.cu", "common.cuh"],
    "dense_bf16": ["k_dense.cu", "common.cuh"],
    "dense_bf16x3": ["k_dense.cu", "common.cuh"],
}


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture in
    profiles/dram_traffic.md, if the kernel's source still matches."""
    import hashlib
    srcs = KERNEL_SOURCES.get(kernel)
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not srcs or not os.path.exists(path):
        return None
    h = hashlib.sha1()
    for f in srcs:
        with open(os.path.join(ROOT, "exact_tensor_network_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()[:16]
    with open(path) as fh:
        for line in fh:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) == 5 and cells[0] == kernel and cells[1] == workload and cells[2] == sha:
                return float(cells[4])
    return None


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


def oracle_subtree_sample(net, tree, slices, budget: float):
    """The oracle on whole subtrees of the workload's own tree (slice 0),
    largest first, until `budget` flops are covered.  Returns (flops,
    seconds, number of subtrees, threads)."""
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
    for x in chosen:
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
    return flops, secs, len(chosen), oracle.num_threads()


def cpu_baseline_leg(net, tree, slices, seconds: float):
    """fp64 oracle rate on this workload: full contractions when they fit
    in a few tens of seconds, else whole subtrees of its tree."""
    from oracle import planner
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, slices)
    if p.C_t_total <= ORACLE_FULL_LIMIT:
        rate, runs, el, threads, _ = oracle_rate(net, tree, slices, seconds, 50)
        return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": f"{runs} full fp64 oracle contraction(s) of {net.name} ({el:.1f} s)"}
    flops, secs, nsub, threads = oracle_subtree_sample(net, tree, slices, 5e10 * seconds)
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
    # else whole subtrees of the workload's tree (bounded so that all
    # warm-up and timed steps fit in about three minutes)
    budget = min(5e11, 5e10 * 150.0 / max(1, args.steps + args.warmup))

    def one():
        if full:
            t0 = time.perf_counter()
            if slices:
                oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree,
                                       slices)
            else:
                oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
            return p.C_t_total, time.perf_counter() - t0
        f, s, _, _ = oracle_subtree_sample(net, tree, slices, budget)
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
              f"flop per step")
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

    # Per-launch device times (a second pass of the same steps with CUDA
    # events around every launch, on the launching stream).
    plan.set_profiling(True)
    agg = {}
    # a spin kernel ahead of each profiled step keeps the GPU busy while the
    # host enqueues every launch, so the events time launches back to back
    # (device time) rather than host submission gaps
    sleep_cycles = int(2.0e9 * (0.002 + 50e-6 * plan.launches))
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(sleep_cycles)
        plan.execute(leaves, out, stream)
        torch.cuda.synchronize(dev)
        for r in plan.profile():
            a = agg.setdefault(r["kernel"], {"ms": 0.0, "flops": 0, "bytes": 0, "launches": 0})
            a["ms"] += r["ms"]
            a["flops"] += r["flops"]
            a["bytes"] += r["bytes"]
            a["launches"] += 1
    plan.set_profiling(False)
    pk = peaks()
    dom = max(agg, key=lambda k: agg[k]["ms"])
    bound, peak, unit, note = kernel_peak(dom, pk)
    d = agg[dom]
    if unit == "TFLOP/s":
        achieved = d["flops"] / (d["ms"] / 1e3) / 1e12
    else:
        achieved = d["bytes"] / (d["ms"] / 1e3) / 1e9
    per_launch = d["flops" if unit == "TFLOP/s" else "bytes"] / d["launches"]
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": measured_traffic(dom, net.name),
                "traffic_unit": "bytes per launch (ncu dram read + write)",
                "peak_note": note + " (of " + pk["source"] + ")",
                "algorithmic_per_launch": per_launch,
                "avg_launch_ms": d["ms"] / d["launches"]}
    kernels = {k: {"ms_per_step": v["ms"] / args.steps, "launches_per_step": v["launches"] / args.steps,
                   "share": v["ms"] / sum(x["ms"] for x in agg.values())}
               for k, v in agg.items()}

    # End to end through the public API with host buffers: pinned host
    # leaves copied in, contraction, result copied out, every step.
    if device_leaves:
        e2e_none = {"value": None, "unit": "TFLOP/s", "note": "leaves drawn on the device"}
        return finish(args, rank, world, net, plan, ct, units, value, ms, sharded, roofline, kernels,
                      e2e_none, None, clk)
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
    for _ in range(max(1, args.warmup)):
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
           clk)


def finish(args, rank, world, net, plan, ct, units, value, ms, sharded, roofline, kernels, e2e, cpu,
           clk):
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "strong" if sharded else "weak",
                "vs_baseline": None, "dtype": "c64",
                "data": "synthetic" + (" (leaves drawn on the device)" if args.leaves == "device" else ""),
                "config": {"workload": net.name, "tensors": net.n_tensors, "C_t": ct,
                           "C_s": plan.peak, "slices": plan.num_slices, "precision": args.precision,
                           "l2": "flushed between timed steps (untimed 258 MiB fill)",
                           "parallelism": (f"slices round-robin over {world} ranks" if sharded
                                           else f"replicas x{world}")},
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": plan.launches * args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="random_60")
    ap.add_argument("--precision", default="tf32x3", choices=["tf32x3", "bf16", "bf16x3", "fp32"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
