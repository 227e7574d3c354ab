"""Benchmark of the fused row-parallel GEMV + one-shot all-reduce on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mlp_down_decode]

One step is one ``gemv_all_reduce`` call over the workload (default: the MLP
down-projection decode, R=8 ranks as symmetric slots, N=8192, K=28672,
K/R=3584, B=1).  Inputs are synthetic (seeded generator), resident in HBM when
the timed region starts; W rotates over several copies so the bytes touched
between two reads of the same W exceed the 129 MB L2 (no flush is needed).

``value`` is the algorithmic HBM throughput of the call in GB/s (bytes that
the method must move: W_r and x_r of every rank, the fp32 partials written and
read back, and the R bf16 output replicas) divided by the measured time;
``ms_per_step`` gives the call latency.  The ``roofline`` object divides the
same bytes by the kernel's average launch time (CUDA events around every
launch on the launching stream) and by the measured copy bandwidth.

``--impl reference`` times the CPU oracle (fp64, plain C, all host cores) on
the same workload, each step a bounded sample of the rows; it is a deliberately
slow baseline, not the target.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the R ranks of the method are slots of one GPU; nothing
crosses GPUs), timing is max over ranks, and ``value`` sums the ranks' bytes.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gemv_all_reduce µs/call and achieved HBM GB/s (% of GB300 peak), R=8 decode"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def algorithmic_bytes(R, N, K, B):
    """Bytes the fused call must move: W (N x K bf16 over all ranks), x
    (B x K bf16), the fp32 partials of every rank written and read back
    (2 * R * B * N * 4) and the bf16 result in R slots (R * B * N * 2)."""
    return N * K * 2 + B * K * 2 + 2 * R * B * N * 4 + R * B * N * 2


def workload(name):
    import synth

    w = dict(synth.WORKLOADS[name])
    if w["kind"] != "gemv":
        raise SystemExit(f"bench workloads are GEMV + all-reduce cases, not {name}")
    return w


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s, p in zip(sm, power) if p >= 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------- GPU arm


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel: str, workload_name: str, source_sha: str):
    """DRAM bytes per launch from a committed ncu summary, only if it was taken
    on the kernel source as it is now."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[kernel][workload_name]
        if e.get("source_sha") == source_sha:
            return e["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


def kernel_name(plan):
    if plan["path"] == 1:
        return "gemv_ar_ffma_kernel"
    if plan["path"] == 2:
        return "gemv_ar_tc_kernel"
    engine = "tcgen05" if plan["engine"] == 0 else "ffma"
    name = "gemv_ar_sk_kernel" if plan["path"] == 3 else "gemv_ar_dyn_kernel"
    return f"{name}<{engine},slabs={plan['slabs']},ctas_per_sm={plan['ctas_per_sm']}>"


def kernel_source_sha():
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "collective_split_gemv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import __graft_entry__
    import collective_split_gemv_gb300 as csg
    import synth
    from collective_split_gemv_gb300.workspace import GemvWorkspace

    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()   # the other ranks load what rank 0 built
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args.workload)
    R, N, K, B = w["R"], w["N"], w["K"], w["B"]
    nbytes = algorithmic_bytes(R, N, K, B)
    W, x = synth.gemv_inputs(R, N, K, B, w["seed"], w["w_std"], w["x"])
    w_total = W.nbytes
    copies = max(1, min(8, math.ceil(3 * L2_BYTES / max(w_total, 1))))
    ws = GemvWorkspace(R, N, K, B, copies=copies, device=local_rank)
    paths = {"auto": csg.GEMV_PATH_AUTO, "ffma": csg.GEMV_PATH_FFMA, "tc": csg.GEMV_PATH_TC,
             "sk": csg.GEMV_PATH_SK, "dyn": csg.GEMV_PATH_DYN}
    csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, paths[args.gemv_path])
    csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_SLABS, args.sk_slabs)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_ENGINE, args.sk_engine)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_CTAS_PER_SM, args.sk_cps)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_GRID, args.sk_grid)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, args.dyn_splits)
    plan = csg.symm_gemv_plan(ws.h, N, K, B)
    for c in range(copies):
        ws.load_W(W, copy=c)
    ws.load_x(x)
    stream = torch.cuda.Stream(device=dev)
    working_set = copies * w_total
    flush = working_set < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def step(i):
        ws.run(stream, copy=i % copies)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if flush:
                flush_buf.fill_(i & 0xFF)
            step(i)
    stream.synchronize()
    code, _, _ = csg.symm_status(ws.h, stream)
    if code != csg.SYMM_OK:
        raise SystemExit(f"protocol error during warm-up: {csg.symm_last_error()}")

    # ---- timed region: K calls, CUDA events around each launch ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(str(local_rank) if not visible else visible.split(",")[local_rank].strip())
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            if flush:
                flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step(i)
            ends[i].record(stream)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region_ms = t0.elapsed_time(t1)
    code, _, _ = csg.symm_status(ws.h, stream)
    if code != csg.SYMM_OK:
        raise SystemExit(f"protocol error in the timed region: {csg.symm_last_error()}")
    # with L2 flushes inside the region, the per-step time is the kernels' own
    step_ms = sum(launch_ms) / len(launch_ms) if flush else region_ms / args.steps

    # ---- e2e: same call through the ABI with host buffers every step ----
    x_host = [torch.from_numpy(np.ascontiguousarray(x[r])).view(torch.uint8).reshape(-1).pin_memory()
              for r in range(R)]
    y_host = torch.empty(ws.y_bytes, dtype=torch.uint8).pin_memory()
    x_dev = [ws.x_view(r) for r in range(R)]
    w_dev = [ws.w_view(r, 0) for r in range(R)]
    y_dev = ws.y_view(0)
    e2e_steps = max(3, min(args.steps, 200))
    torch.cuda.synchronize(dev)
    tt = time.perf_counter()
    for i in range(e2e_steps):
        with torch.cuda.stream(stream):
            for r in range(R):
                x_dev[r].copy_(x_host[r], non_blocking=True)
            step(i)
            y_host.copy_(y_dev, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - tt) * 1e3 / e2e_steps
    # weights streamed from the host as well (every step copies all W_r)
    W_host = [torch.from_numpy(np.ascontiguousarray(W[r])).view(torch.uint8).reshape(-1).pin_memory()
              for r in range(R)]
    ew_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize(dev)
    tt = time.perf_counter()
    for i in range(ew_steps):
        with torch.cuda.stream(stream):
            for r in range(R):
                w_dev[r].copy_(W_host[r], non_blocking=True)
                x_dev[r].copy_(x_host[r], non_blocking=True)
            ws.run(stream, copy=0)
            y_host.copy_(y_dev, non_blocking=True)
        stream.synchronize()
    ew_ms = (time.perf_counter() - tt) * 1e3 / ew_steps
    code, _, _ = csg.symm_status(ws.h, stream)
    assert code == csg.SYMM_OK

    # ---- max over ranks ----
    vals = torch.tensor([step_ms, e2e_ms, ew_ms, statistics.mean(launch_ms)], dtype=torch.float64)
    if world > 1:
        t = vals.to(dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        vals = t.cpu()
    step_ms, e2e_ms, ew_ms, mean_launch_ms = [float(v) for v in vals]
    ws.close()
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes / (mean_launch_ms * 1e-3) / 1e9
    kernel = kernel_name(plan)
    line = {
        "metric": METRIC,
        "value": round(world * nbytes / (step_ms * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 6),
        "us_per_call": round(step_ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "f32",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, bf16 RNE)",
        "config": {
            "workload": args.workload, "R": R, "N": N, "K": K, "K_per_rank": K // R, "B": B,
            "algorithmic_bytes_per_call": nbytes,
            "l2": (f"L2 flushed (2x{L2_BYTES // 10**6} MB write) between launches; step time = kernel time"
                   if flush else
                   f"inputs larger than L2: {copies} rotating copies of W ({working_set / 1e9:.2f} GB)"),
            "parallelism": "R ranks as symmetric slots on one GPU" + (f"; {world} independent replicas"
                                                                     if world > 1 else ""),
            "plan": plan,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": kernel,
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(kernel, args.workload, kernel_source_sha()),
            "mean_launch_us": round(mean_launch_ms * 1e3, 3),
            "median_launch_us": round(statistics.median(launch_ms) * 1e3, 3),
        },
        "clocks": clocks,
        "e2e": {
            "value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "us_per_call": round(e2e_ms * 1e3, 2),
            "h2d_bytes_per_step": R * B * (K // R) * 2, "d2h_bytes_per_step": B * N * 2,
            "what": "x_r of every rank H2D from pinned memory, gemv_all_reduce, y (slot 0) D2H, "
                    "stream synchronised every step; W_r resident (model weights)",
        },
        "e2e_weights_from_host": {
            "value": round(nbytes / (ew_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "us_per_call": round(ew_ms * 1e3, 2),
            "h2d_bytes_per_step": N * K * 2 + R * B * (K // R) * 2, "d2h_bytes_per_step": B * N * 2,
        },
        "gpu_launches": args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
    return line


# ------------------------------------------------------------ CPU oracle


def _oracle_sample(name, rows):
    """Inputs restricted to the first `rows` output rows of the workload."""
    import synth

    w = workload(name)
    W, x = synth.gemv_inputs(w["R"], w["N"], w["K"], w["B"], w["seed"], w["w_std"], w["x"])
    return w, W, x


def cpu_baseline(name, budget_s=10.0, steps=None, warmup=0):
    """Time the oracle (as it is) on this host's cores on row samples of the
    workload; returns the cpu_baseline object (value in GB/s of algorithmic
    bytes, scaled to the rows processed)."""
    import numpy as np

    import oracle

    w, W, x = _oracle_sample(name, None)
    R, N, K, B = w["R"], w["N"], w["K"], w["B"]
    threads = host_cores()
    t = time.perf_counter()
    oracle.gemv_all_reduce(W[:, :64], x, threads=threads)
    per_row = max((time.perf_counter() - t) / 64, 1e-9)
    if steps is None:
        rows = N
        reps = max(1, int(budget_s / (per_row * N)))
    else:
        per_step = budget_s / max(1, steps + warmup)
        rows = int(max(1, min(N, per_step / per_row)))
        reps = steps
    Ws = np.ascontiguousarray(W[:, :rows])
    for _ in range(warmup):
        oracle.gemv_all_reduce(Ws, x, threads=threads)
    t = time.perf_counter()
    for _ in range(reps):
        oracle.gemv_all_reduce(Ws, x, threads=threads)
    el = time.perf_counter() - t
    frac = rows / N
    sec_per_call = el / reps / frac
    return {
        "value": round(algorithmic_bytes(R, N, K, B) / sec_per_call / 1e9, 4),
        "unit": "GB/s",
        "us_per_call_equiv": round(sec_per_call * 1e6, 1),
        "cores": threads,
        "kind": "oracle",
        "sample": f"{rows} of {N} rows of {name} (all R={R} ranks, full K={K}), {reps} repetitions, "
                  f"{el:.1f} s; time scaled to the full call",
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = workload(args.workload)
    R, N, K, B = w["R"], w["N"], w["K"], w["B"]
    cb = cpu_baseline(args.workload, budget_s=min(120.0, 2.0 * (args.steps + args.warmup)),
                      steps=args.steps, warmup=args.warmup)
    sec = cb["us_per_call_equiv"] * 1e-6
    return {
        "metric": METRIC, "impl": "reference", "value": cb["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, bf16 RNE)",
        "config": {"workload": args.workload, "R": R, "N": N, "K": K, "B": B,
                   "algorithmic_bytes_per_call": algorithmic_bytes(R, N, K, B)},
        "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=100)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="mlp_down_decode")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--gemv-path", choices=("auto", "ffma", "tc", "sk", "dyn"), default="auto",
                   help="force one kernel (measurement only)")
    p.add_argument("--sk-slabs", type=int, default=0, choices=(0, 1, 2, 4),
                   help="stream-K slabs per pipeline stage (0 = library default)")
    p.add_argument("--sk-cps", type=int, default=0, choices=(0, 1, 2, 3),
                   help="stream-K resident CTAs per SM (0 = library default)")
    p.add_argument("--sk-grid", type=int, default=0,
                   help="stream-K grid: 0 library default, -1 one CTA per (tile, rank), or a count")
    p.add_argument("--dyn-splits", type=int, default=0,
                   help="persistent kernel: K splits per (tile, rank) (0 = library default)")
    p.add_argument("--sk-engine", type=int, default=-1, choices=(-1, 0, 1),
                   help="stream-K engine: -1 auto, 0 tcgen05, 1 FFMA")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch

            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
