"""Benchmark of the full-model Muon step on GB300.

A "step" is one muon_step_grouped call over every 2-D weight of the workload:
prologue (momentum, Nesterov blend, bf16 cast, norm partials), five quintic
Newton-Schulz rounds (Gram, polynomial, update on the tensor cores; fp32 for
matrices with min(rows, cols) < 64) and the parameter write.

Default workload: the GPT-2 124M d=768 model (10 QKVO weights viewed as 40
768x768 blocks, 11 + 11 MLP matrices, 10 attention gates, 1 smear gate).
Value: counted NS5 FLOPs per step, 5 * (4 m^2 n + 2 m^3) per matrix (m <= n),
divided by the device time of the whole step: TFLOP/s, higher is better.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (the step has no cross-GPU exchange on one node: replicas only); the
timed region is bracketed by barriers and the max over ranks is reported.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NS5 TFLOP/s (frac of GB300 BF16 peak); us per full-model Muon step"
DEFAULT_WORKLOAD = "gpt2-124M-d768"


# ---------------------------------------------------------------- counting
def counted_ns_flops(groups, steps):
    """5 rounds x (4 m^2 n + 2 m^3) per matrix, m = min(rows, cols), n = max."""
    tot = 0.0
    for g in groups:
        m, n = min(g.rows, g.cols), max(g.rows, g.cols)
        tot += g.batch * steps * (4.0 * m * m * n + 2.0 * m ** 3)
    return tot


def elementwise_bytes(wl):
    """Algorithmic HBM bytes of the elementwise work of one step: read g, read and
    write the fp32 momentum buffer, write bf16 u (prologue), read and write the fp32
    parameter (last update epilogue)."""
    gbytes = 2 if str(wl.grad_dtype).endswith("bfloat16") else 4
    return wl.n_elements * (gbytes + 8 + 2 + 8)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------- ranks
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def aggregate_over_ranks(local_ms: float, local_units: float, world: int):
    """Max time and summed work over ranks (identity when world == 1)."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for k, name in enumerate(names):
                    if r[5 + k].strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing
# A workload whose counted NS flops per step stay under this is timed whole on the
# host (the GPT-2 124M step is ~1.4 TFLOP, a few seconds on 16 cores); a larger
# one is timed on one stored matrix per group and the time multiplied by the
# group's stored count ("extrapolated").
ORACLE_FULL_MAX_FLOPS = 2.0e12
ORACLE_REPEATS = 3
# steps at least this long run their tensor-core kernels against the sustained
# (power-capped) bf16 peak rather than the burst one
LONG_STEP_MS = 10.0
# end-to-end leg: untimed pipelined steps, then timed runs of at most E2E_STEPS
E2E_STEPS = 20
E2E_WARMUP = 3
E2E_TRIALS = 5


def _oracle_group_inputs(wl, gi, stored, device="cpu"):
    """(params, grads, bufs) as float64 numpy [k, rows, cols] for the first `stored`
    stored matrices of group gi (k = stored x the blocks each one is viewed as)."""
    import workloads
    grp = wl.groups[gi]
    per_stored = grp.batch // grp.stored_shape[0]
    ps, gs, bs = [], [], []
    for j in range(stored):
        p, g, b = workloads.draw_stored_matrix(wl, gi, j, device)
        shape = (per_stored, grp.rows, grp.cols)
        ps.append(p.reshape(shape).double().numpy())
        gs.append(g.float().reshape(shape).double().numpy())
        bs.append(b.reshape(shape).double().numpy())
    import numpy as np
    return np.concatenate(ps), np.concatenate(gs), np.concatenate(bs)


def oracle_plan(wl):
    """'full' or 'extrapolated' for this workload's CPU oracle timing."""
    return "full" if counted_ns_flops(wl.groups, wl.steps) <= ORACLE_FULL_MAX_FLOPS \
        else "extrapolated"


def time_oracle_step(wl, repeats=ORACLE_REPEATS):
    """Seconds per Muon step of the CPU float64 oracle on the workload.

    'full': every matrix of the step, the median of `repeats` timed steps on the
    same inputs.  'extrapolated': one stored matrix per group, timed once, times the
    group's stored count.  Returns (seconds, description)."""
    import oracle
    kw = dict(momentum=wl.momentum, nesterov=wl.nesterov, lr=wl.lr,
              weight_decay=wl.weight_decay, steps=wl.steps)
    if oracle_plan(wl) == "full":
        inputs = [_oracle_group_inputs(wl, gi, grp.stored_shape[0])
                  for gi, grp in enumerate(wl.groups)]
        times = []
        for _ in range(repeats):
            t0 = time.perf_counter()
            for p, g, b in inputs:
                oracle.muon_step_batched(p, g, b, **kw)
            times.append(time.perf_counter() - t0)
        return statistics.median(times), (f"whole step ({wl.n_matrices} matrices), median of "
                                          f"{repeats} timed steps")
    total = 0.0
    for gi, grp in enumerate(wl.groups):
        p, g, b = _oracle_group_inputs(wl, gi, 1)
        t0 = time.perf_counter()
        oracle.muon_step_batched(p, g, b, **kw)
        total += (time.perf_counter() - t0) * grp.stored_shape[0]
    return total, ("extrapolated: one stored matrix per group ("
                   + ", ".join(f"{g.rows}x{g.cols} x{g.stored_shape[0]}" for g in wl.groups)
                   + ") timed once, times the group's count")


def cpu_cores():
    n = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ---------------------------------------------------------------- reference arm
def run_reference(args, wl):
    """The CPU float64 oracle timed on the host cores, on the same workload and metric:
    each step is one whole oracle step ('full' workloads) or the extrapolated
    one-matrix-per-group sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    flops = counted_ns_flops(wl.groups, wl.steps)
    for _ in range(args.warmup):
        time_oracle_step(wl, repeats=1)
    times, how = [], ""
    for _ in range(args.steps):
        t, how = time_oracle_step(wl, repeats=1)
        times.append(t)
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = f"{how}; {args.steps} steps"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "oracle": oracle_plan(wl), "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "cpu": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
NS_KINDS = ("gram", "poly", "update", "small_ns", "fused_ns", "rounds")
# timed steps of the other workloads in the `configs` object (the headline
# workload takes --steps): the d=4096 step is ~0.33 s
CONFIG_STEPS = {"single-128x256": 50, "gpt-9L-d512": 50, "gpt2-124M-d768": 20,
                "gpt-24L-d2048": 5, "gpt-32L-d4096": 3}


def time_workload(muon, wl, dev, steps, warmup, use_graph, peaks, local, world):
    """One workload on this GPU: the step timed with CUDA events (replayed as a CUDA
    graph), then a traced pass of the same steps for per-kernel times.  Returns
    (result dict, (tensors, step)) -- the tensors stay alive for the caller."""
    import torch

    import workloads
    groups = workloads.make_workload(wl, dev)
    tensors = [(P, G, B) for _, P, G, B in groups]
    step = muon.GroupedStep(tensors, momentum=wl.momentum, lr=wl.lr,
                            weight_decay=wl.weight_decay, nesterov=wl.nesterov, steps=wl.steps)
    flops = counted_ns_flops(wl.groups, wl.steps)
    stream = torch.cuda.current_stream()

    run = step
    graph = None
    if use_graph:
        # capture the whole step (all launches) once; replay it every step
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        run = graph.replay

    lps = launches_per_step(step)
    for _ in range(max(warmup, 0)):
        run()
    torch.cuda.synchronize()

    # inputs that fit in L2 (the 128x256 workload): L2 is flushed before every
    # timed step by writing a buffer twice its size, outside that step's events
    in_bytes = wl.n_elements * (2 + 4 + 4)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
             if in_bytes <= l2_bytes else None)

    clocks = ClockSampler(local)
    clocks.start()
    n0 = muon.kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if flush is None:
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        local_ms = e0.elapsed_time(e1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        local_ms = sum(a.elapsed_time(b) for a, b in evs)
    barrier(world)
    # graph replays launch the captured kernels without passing through the host counter
    launches = lps * steps if graph is not None else muon.kernel_launch_count() - n0
    clock = clocks.stop()
    ms, units = aggregate_over_ranks(local_ms, flops * steps, world)
    value = units / (ms / 1e3) / 1e12
    flushed = flush is not None
    del flush

    # per-kernel times from a traced pass over the same steps (eager launches)
    muon.trace_begin(100000)
    for _ in range(steps):
        step()
    recs = muon.trace_end(100000)
    torch.cuda.synchronize()
    kinds = {}
    for r in recs:
        k = kinds.setdefault(r["kind"], {"ms": 0.0, "n": 0, "flops": 0.0, "bytes": 0.0})
        k["ms"] += r["ms"]
        k["n"] += 1
        k["flops"] += r["flops"]
        k["bytes"] += r["bytes"]
    ns_ms = sum(kinds[k]["ms"] for k in NS_KINDS if k in kinds) / steps
    ns_flops_exec = sum(kinds[k]["flops"] for k in NS_KINDS if k in kinds) / steps
    traced_ms = sum(k["ms"] for k in kinds.values()) / steps
    dom_name, dom = max(kinds.items(), key=lambda kv: kv[1]["ms"])
    per_launch_ms = dom["ms"] / dom["n"]
    if dom["flops"] > 0:
        achieved = dom["flops"] / dom["n"] / (per_launch_ms / 1e3) / 1e12
        peak, which = tensor_peak(ms / steps, clock.get("reasons", []), peaks)
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_for(dom_name, wl.name),
                "peak_source": f"{peaks['source']} {which} bf16",
                "frac_of_burst": achieved / peaks["bf16_tflops"], "ms_per_launch": per_launch_ms,
                "flops_per_launch": dom["flops"] / dom["n"]}
    else:
        achieved = dom["bytes"] / dom["n"] / (per_launch_ms / 1e3) / 1e9
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic_for(dom_name, wl.name), "peak_source": peaks["source"],
                "ms_per_launch": per_launch_ms, "bytes_per_launch": dom["bytes"] / dom["n"]}
    # elementwise kernels (HBM-bound): prologue and apply, bytes they must move
    ew = [kinds[k] for k in ("prologue", "apply") if k in kinds]
    elementwise = None
    if ew:
        ew_bytes = sum(k["bytes"] for k in ew)
        ew_ms = sum(k["ms"] for k in ew)
        gbs = ew_bytes / (ew_ms / 1e3) / 1e9
        elementwise = {"gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
                       "ms_per_step": ew_ms / steps,
                       "per_kernel": {name: {"gbs": kinds[name]["bytes"] / (kinds[name]["ms"] / 1e3) / 1e9,
                                             "ms_per_step": kinds[name]["ms"] / steps}
                                      for name in ("prologue", "apply") if name in kinds}}
    per_step_ms = ms / steps
    res = {
        "workload": wl.name, "steps": steps, "warmup": warmup, "ms_per_step": per_step_ms,
        "us_per_step": 1e3 * per_step_ms, "tflops": value,
        "frac_of_peak": value / peaks["bf16_tflops"],
        "frac_of_sustained_peak": value / peaks["bf16_tflops_sustained"],
        # the flops the kernels execute (Gram and Poly on the upper tiles only)
        "method_tflops": ns_flops_exec / (per_step_ms / 1e3) / 1e12,
        "counted_gflop_per_step": flops / 1e9,
        "executed_gflop_per_step": ns_flops_exec / 1e9,
        "matrices": wl.n_matrices,
        "groups": [f"{g.batch}x{g.rows}x{g.cols}" for g in wl.groups],
        "graph": bool(use_graph),
        "l2": ("inputs larger than L2: %.0f MB of grads, params and momentum moved per step"
               % (wl.n_elements * (2 + 8 + 8) / 1e6)) if not flushed else
              ("L2 flushed before every timed step (%.0f MB written outside the step's "
               "events); inputs %.1f MB" % (2 * l2_bytes / 1e6, in_bytes / 1e6)),
        "ns_chain": {"ms_per_step": ns_ms, "tflops": flops / (ns_ms / 1e3) / 1e12,
                     "frac": flops / (ns_ms / 1e3) / 1e12 / peaks["bf16_tflops"]},
        "traced_ms_per_step": traced_ms,
        "kernels": {k: {"ms_per_step": v["ms"] / steps, "launches_per_step": v["n"] / steps}
                    for k, v in kinds.items()},
        "elementwise": elementwise, "roofline": roof, "gpu_launches": launches, "clocks": clock,
    }
    return res, (tensors, step)


def tensor_peak(step_ms, reasons, peaks):
    """The bf16 peak a tensor-core kernel is measured against: the burst figure in a
    short step, the sustained one (the long loop under the power cap) in a step of
    LONG_STEP_MS or more or once the power cap showed in the timed region."""
    if step_ms >= LONG_STEP_MS or "sw_power_cap" in reasons:
        return peaks["bf16_tflops_sustained"], "sustained"
    return peaks["bf16_tflops"], "burst"


def median_trial(trials, steps):
    """(every trial's ms per step, sorted; the (device ms, wall ms) of the median trial),
    a trial's time per step being the longer of its device and wall clocks."""
    per_step = sorted(max(t) / steps for t in trials)
    med = per_step[len(per_step) // 2]
    return per_step, next(t for t in trials if max(t) / steps == med)


def time_e2e(muon, wl, tensors, step, world, max_steps=E2E_STEPS):
    """The same grouped step end to end through the public binding with host buffers:
    every step's gradients uploaded from pinned host memory and its parameters read
    back, inside the timed region."""
    import torch
    dev = tensors[0][0].device
    stream = torch.cuda.current_stream()
    flops = counted_ns_flops(wl.groups, wl.steps)
    host_g = [G.cpu().pin_memory() for _, G, _ in tensors]
    host_p = [torch.empty(P.shape, dtype=P.dtype, pin_memory=True) for P, _, _ in tensors]
    h2d = sum(t.numel() * t.element_size() for t in host_g)
    d2h = sum(t.numel() * t.element_size() for t in host_p)
    e2e_steps = max(3, min(E2E_STEPS, max_steps))
    # Three streams, two device gradient buffers and two device parameter
    # snapshots.  Step k's gradient upload (copy stream in) goes into buffer
    # k % 2 once step k-2 is done with it, so it runs beside step k-1; step k
    # runs on the main stream once its upload is in; its parameters are then
    # copied on the device into snapshot k % 2 (once the read-back of step k-2
    # from that snapshot is done) and read back to the host from it (copy stream
    # out) while step k+1 computes, so the read-back stream never waits for a
    # snapshot.  Every copy of every step is inside the timed region.
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    grads2 = [G.clone() for _, G, _ in tensors]
    step2 = muon.GroupedStep([(P, G2, B) for (P, _, B), G2 in zip(tensors, grads2)],
                             momentum=wl.momentum, lr=wl.lr, weight_decay=wl.weight_decay,
                             nesterov=wl.nesterov, steps=wl.steps)
    dev_g = [[G for _, G, _ in tensors], grads2]
    steps_ab = [step, step2]
    snap = [[torch.empty_like(P) for P, _, _ in tensors] for _ in range(2)]
    def run(n):
        """n pipelined steps; returns (device ms, wall ms) for all of them."""
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        e0.record(stream)
        for k in range(n):
            up.wait_event(ev_done[k - 2] if k > 1 else e0)
            with torch.cuda.stream(up):
                for G, hg in zip(dev_g[k % 2], host_g):
                    G.copy_(hg, non_blocking=True)
                ev_in[k].record(up)
            stream.wait_event(ev_in[k])
            steps_ab[k % 2]()
            if k > 1:
                stream.wait_event(ev_out[k - 2])
            for (P, _, _), sp in zip(tensors, snap[k % 2]):
                sp.copy_(P, non_blocking=True)
            ev_done[k].record(stream)
            down.wait_event(ev_done[k])
            with torch.cuda.stream(down):
                for sp, hp in zip(snap[k % 2], host_p):
                    hp.copy_(sp, non_blocking=True)
                ev_out[k].record(down)
        stream.wait_event(ev_out[n - 1])
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1), 1e3 * (time.perf_counter() - t0)

    run(E2E_WARMUP)  # untimed: the second step object's first calls, first touch of host pages
    # The host link is shared with the machine's other jobs: E2E_TRIALS timed runs, the
    # median reported, all of them listed.
    trials = [run(e2e_steps) for _ in range(E2E_TRIALS)]
    per_step, (dev_ms, wall_ms) = median_trial(trials, e2e_steps)
    med = max(dev_ms, wall_ms) / e2e_steps
    e2e_ms, e2e_units = aggregate_over_ranks(med * e2e_steps, flops * e2e_steps, world)
    return {"value": e2e_units / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
            "warmup": E2E_WARMUP, "trials_ms_per_step": per_step,
            "device_ms_per_step": dev_ms / e2e_steps, "wall_ms_per_step": wall_ms / e2e_steps,
            "schedule": "gradient upload (copy stream, two device gradient buffers) and "
                        "parameter read-back from device snapshots (second copy stream, two "
                        "snapshots) of neighbouring steps overlap the compute; every copy of "
                        "every step inside the timed region; median of five timed runs"}


def run_gpu(args, wl):
    import torch

    import newton_schulz_step_gb300 as muon
    import workloads

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    head, (tensors, step) = time_workload(muon, wl, dev, args.steps, args.warmup,
                                          bool(args.graph), peaks, local, world)
    adam = time_adam(args, wl, dev, peaks) if wl.adam else None
    e2e = time_e2e(muon, wl, tensors, step, world, args.steps)
    del tensors, step
    torch.cuda.empty_cache()

    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    cpu = None
    if do_cpu:
        secs, how = time_oracle_step(wl)
        flops = counted_ns_flops(wl.groups, wl.steps)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
               "cpu": cpu_model(), "kind": "oracle", "sample": how,
               "ms_per_step": 1e3 * secs, "oracle": oracle_plan(wl)}

    # every workload of the build, on the same GPU, one after the other
    configs = {}
    if not args.headline_only:
        for name in workloads.WORKLOADS:
            if name == wl.name:
                res = dict(head)
            else:
                w = workloads.get(name)
                res, keep = time_workload(muon, w, dev, min(args.steps, CONFIG_STEPS[name]),
                                          args.warmup, bool(args.graph), peaks, local, world)
                del keep
                torch.cuda.empty_cache()
            if do_cpu:
                w = workloads.get(name)
                if name == wl.name:
                    secs, how = cpu["ms_per_step"] / 1e3, cpu["sample"]
                else:
                    secs, how = time_oracle_step(w)
                res["oracle"] = {"ms_per_step": 1e3 * secs, "plan": oracle_plan(w),
                                 "sample": how, "cores": cpu_cores(),
                                 "speedup": 1e3 * secs / res["ms_per_step"]}
            configs[name] = res

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["tflops"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "us_per_step": head["us_per_step"], "frac_of_peak": head["frac_of_peak"],
            "frac_of_sustained_peak": head["frac_of_sustained_peak"],
            "method_tflops": head["method_tflops"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "matrices": wl.n_matrices, "groups": head["groups"],
                       "counted_gflop_per_step": head["counted_gflop_per_step"],
                       "graph": head["graph"], "l2": head["l2"]},
            "ns_chain": head["ns_chain"], "traced_ms_per_step": head["traced_ms_per_step"],
            "kernels": head["kernels"], "elementwise": head["elementwise"], "adam": adam,
            "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
            "peaks": {k: peaks[k] for k in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs",
                                            "source")},
            "configs": configs or None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_adam(args, wl, dev, peaks):
    """The Adam half of the optimizer on the workload's non-matrix parameters
    (embedding, head, scalars): one fused launch per step, timed on its own.
    Not part of the Muon-step metric above; reported beside it."""
    import torch

    import newton_schulz_step_gb300 as muon
    import workloads

    sets = workloads.make_adam_set(wl, dev)
    run = muon.AdamStep([(p, g, m, v, t.lr_scale, t.wd_scale) for t, p, g, m, v in sets],
                        lr=muon.ADAM_LR, betas=muon.ADAM_BETAS, eps=muon.ADAM_EPS,
                        weight_decay=0.0)
    nbytes = sum(p.numel() * (12 + g.element_size() + 12) for _, p, g, m, v in sets)
    stream = torch.cuda.current_stream()
    t = wl.adam_step
    for _ in range(max(args.warmup, 3)):
        run(t)
        t += 1
    torch.cuda.synchronize()
    n0 = muon.kernel_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run(t)
        t += 1
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"kernel": "adam", "bound": "hbm", "us_per_step": 1e3 * ms, "gbs": gbs,
            "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"], "bytes_per_step": nbytes,
            "launches_per_step": (muon.kernel_launch_count() - n0) / args.steps,
            "tensors": [f"{t.name}:{t.numel}" for t, *_ in sets],
            "l2": "inputs larger than L2: %.0f MB moved per step" % (nbytes / 1e6)}


def launches_per_step(step):
    import newton_schulz_step_gb300 as muon
    n0 = muon.kernel_launch_count()
    step()
    return muon.kernel_launch_count() - n0


# The sources each traced kernel is built from: a committed DRAM-traffic figure is
# used only while these files are unchanged since it was captured.
KERNEL_SOURCES = {
    "gram": ("ns_gemm.cu", "ptx.cuh"), "poly": ("ns_gemm.cu", "ptx.cuh"),
    "update": ("ns_gemm.cu", "ptx.cuh"), "prologue": ("prologue.cu",), "apply": ("prologue.cu",),
    "small_ns": ("ns_small.cu",), "fused_ns": ("ns_fused.cu", "ptx.cuh"), "adam": ("adam.cu",),
    "rounds": ("ns_gemm.cu", "ptx.cuh"),
}


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this build."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{workload}/{kernel}")
        if not e or e.get("source_hash") != source_hash(kernel):
            return None
        return e["dram_bytes_per_launch"]
    except (OSError, ValueError):
        return None


def source_hash(kernel: str):
    """Hash of a kernel's sources with comments and blank space removed, so that a
    recorded ncu capture stays valid across comment edits but not code changes."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "newton_schulz_step_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, tuple(sorted(os.listdir(csrc)))):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(f.encode() + text.encode())
    return h.hexdigest()[:16]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--graph", type=int, default=1, help="replay the step as a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only --workload (no `configs` object)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    import workloads
    wl = workloads.get(args.workload)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
