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
def oracle_sample(wl, per_group=1):
    """A bounded sample of the workload for the CPU oracle: the first `per_group`
    matrices of every group, drawn with the workload's CPU seeds."""
    import workloads
    sample = []
    for gi, grp in enumerate(wl.groups):
        n_stored = grp.stored_shape[0]
        per_stored = grp.batch // n_stored
        for j in range(min(per_group, n_stored)):
            p, g, b = workloads.draw_stored_matrix(wl, gi, j, "cpu")
            shape = (per_stored, grp.rows, grp.cols)
            sample.append((grp, p.reshape(shape), g.reshape(shape), b.reshape(shape)))
    return sample


def time_oracle(wl, per_group=1, repeats=1):
    """Times the CPU float64 oracle on oracle_sample(); returns (seconds, counted flops)."""
    import numpy as np
    import oracle
    import workloads  # noqa: F401
    sample = oracle_sample(wl, per_group)
    mats = [(grp, p.double().numpy(), g.float().double().numpy(), b.double().numpy())
            for grp, p, g, b in sample]
    flops = 0.0
    for grp, p, _, _ in mats:
        m, n = min(grp.rows, grp.cols), max(grp.rows, grp.cols)
        flops += p.shape[0] * wl.steps * (4.0 * m * m * n + 2.0 * m ** 3)
    best = float("inf")
    for _ in range(repeats):
        t0 = time.perf_counter()
        for grp, p, g, b in mats:
            oracle.muon_step_batched(p, g, b, momentum=wl.momentum, nesterov=wl.nesterov,
                                     lr=wl.lr, weight_decay=wl.weight_decay, steps=wl.steps)
        best = min(best, time.perf_counter() - t0)
    del np
    return best, flops


CPU_BASELINE_SECONDS = 10.0


def cpu_cores():
    n = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def sample_text(wl, per_group):
    return (f"first {per_group} stored matrix of each of the {len(wl.groups)} groups "
            f"({', '.join(f'{g.rows}x{g.cols}' for g in wl.groups)}), full NS5 in float64")


# ---------------------------------------------------------------- reference arm
def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    per_group = 1
    for _ in range(args.warmup):
        time_oracle(wl, per_group)
    times, flops = [], 0.0
    for _ in range(args.steps):
        t, flops = time_oracle(wl, per_group)
        times.append(t)
    total = sum(times)
    value = flops * len(times) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample": sample_text(wl, per_group)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample_text(wl, per_group)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
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

    groups = workloads.make_workload(wl, dev)
    tensors = [(P, G, B) for _, P, G, B in groups]
    step = muon.GroupedStep(tensors, momentum=wl.momentum, lr=wl.lr,
                            weight_decay=wl.weight_decay, nesterov=wl.nesterov, steps=wl.steps)
    flops = counted_ns_flops(wl.groups, wl.steps)
    stream = torch.cuda.current_stream()

    run = step
    graph = None
    if args.graph:
        # capture the whole step (all launches) once; replay it every step
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        run = graph.replay

    lps = launches_per_step(step)
    for _ in range(max(args.warmup, 0)):
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
        for _ in range(args.steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        local_ms = e0.elapsed_time(e1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        local_ms = sum(a.elapsed_time(b) for a, b in evs)
    barrier(world)
    # graph replays launch the captured kernels without passing through the host counter
    launches = lps * args.steps if graph is not None else muon.kernel_launch_count() - n0
    clock = clocks.stop()
    ms, units = aggregate_over_ranks(local_ms, flops * args.steps, world)
    value = units / (ms / 1e3) / 1e12

    # per-kernel times from a traced pass over the same steps (eager launches)
    muon.trace_begin(100000)
    for _ in range(args.steps):
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
    ns_kinds = ("gram", "poly", "update", "small_ns", "fused_ns", "rounds")
    ns_ms = sum(kinds[k]["ms"] for k in ns_kinds if k in kinds) / args.steps
    traced_ms = sum(k["ms"] for k in kinds.values()) / args.steps
    dom_name, dom = max(kinds.items(), key=lambda kv: kv[1]["ms"])
    per_launch_ms = dom["ms"] / dom["n"]
    if dom["flops"] > 0:
        achieved = dom["flops"] / dom["n"] / (per_launch_ms / 1e3) / 1e12
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic_for(dom_name, wl.name),
                "peak_source": f"{peaks['source']} burst bf16", "ms_per_launch": per_launch_ms,
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
                       "ms_per_step": ew_ms / args.steps,
                       "per_kernel": {name: {"gbs": kinds[name]["bytes"] / (kinds[name]["ms"] / 1e3) / 1e9,
                                             "ms_per_step": kinds[name]["ms"] / args.steps}
                                      for name in ("prologue", "apply") if name in kinds}}

    adam = time_adam(args, wl, dev, peaks) if wl.adam else None

    # end to end through the public API with host buffers: grads in, params out
    host_g = [G.cpu().pin_memory() for _, G, _ in tensors]
    host_p = [torch.empty(P.shape, dtype=P.dtype, pin_memory=True) for P, _, _ in tensors]
    h2d = sum(t.numel() * t.element_size() for t in host_g)
    d2h = sum(t.numel() * t.element_size() for t in host_p)
    e2e_steps = max(1, min(args.steps, 20))
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
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e0.record(stream)
    for k in range(e2e_steps):
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
    stream.wait_event(ev_out[e2e_steps - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max(e0.elapsed_time(e1), 1e3 * (time.perf_counter() - t0))
    e2e_ms, e2e_units = aggregate_over_ranks(e2e_ms, flops * e2e_steps, world)
    e2e = {"value": e2e_units / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_ms / e2e_steps,
           "schedule": "gradient upload (copy stream, two device gradient buffers) and "
                       "parameter read-back from device snapshots (second copy stream, two "
                       "snapshots) of neighbouring steps overlap the compute; every copy of "
                       "every step inside the timed region"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the sample, repeated until about 10 s of CPU work have been timed
        secs, cflops, reps = 0.0, 0.0, 0
        while reps == 0 or secs < CPU_BASELINE_SECONDS:
            t, f = time_oracle(wl, 1)
            secs, cflops, reps = secs + t, cflops + f, reps + 1
        cpu = {"value": cflops / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
               "kind": "oracle", "sample": f"{sample_text(wl, 1)}, {reps} times",
               "seconds": secs}

    if rank == 0:
        per_step_ms = ms / args.steps
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms,
            "us_per_step": 1e3 * per_step_ms, "frac_of_peak": value / peaks["bf16_tflops"],
            "frac_of_sustained_peak": value / peaks["bf16_tflops_sustained"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "matrices": wl.n_matrices,
                       "groups": [f"{g.batch}x{g.rows}x{g.cols}" for g in wl.groups],
                       "counted_gflop_per_step": flops / 1e9, "graph": bool(args.graph),
                       "l2": ("inputs larger than L2: %.0f MB of grads, params and momentum "
                              "moved per step" % (wl.n_elements * (2 + 8 + 8) / 1e6))
                       if flush is None else
                       ("L2 flushed before every timed step (%.0f MB written outside the "
                        "step's events); inputs %.1f MB" % (flush.numel() / 1e6, in_bytes / 1e6))},
            "ns_chain": {"ms_per_step": ns_ms, "tflops": flops / (ns_ms / 1e3) / 1e12,
                         "frac": flops / (ns_ms / 1e3) / 1e12 / peaks["bf16_tflops"]},
            "traced_ms_per_step": traced_ms,
            "kernels": {k: {"ms_per_step": v["ms"] / args.steps, "launches_per_step":
                            v["n"] / args.steps} for k, v in kinds.items()},
            "elementwise": elementwise,
            "adam": adam,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clock,
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
