"""Benchmark of the fused row-parallel GEMV + one-shot all-reduce on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mlp_down_decode]

One step is one library call over the workload: ``gemv_all_reduce`` for the
GEMV workloads (default: the MLP down-projection decode, R=8 ranks as
symmetric slots, N=8192, K=28672, K/R=3584, B=1) and ``one_shot_all_reduce``
for ``--workload allreduce`` (R=8 slots of 4,194,304 bf16).  Inputs are
synthetic (seeded generator) and resident in HBM when the timed region
starts; inputs rotate over enough copies that the bytes touched between two
reads of the same data exceed the 129 MB L2, otherwise L2 is flushed between
launches outside the per-launch events.  Where the call runs on the
persistent kernel its weights are packed once before timing (``symm_pack_w``,
as at model load; the same bytes per call), and the same calls on the
row-major weights are timed after the main leg (``row_major_w``).

``value`` is the algorithmic HBM throughput of the call in GB/s -- the bytes
the method must move (GEMV: W_r and x_r of every rank, the fp32 partials
written and read back, the R bf16 output replicas; all-reduce: R inputs read,
R outputs written) over the measured time per step; ``ms_per_step`` is the
call latency.  ``roofline`` divides the same bytes by the kernel's mean launch
time (CUDA events on the launching stream: around every launch, or around the
whole region when calls are chained) and by the measured copy bandwidth.  ``e2e`` is the same call with its per-step inputs
copied from pinned host memory and its result read back every step;
``e2e_graph`` is that step captured once into a CUDA graph and replayed.

``--impl reference`` times the CPU oracle (fp64, plain C, all host cores) on
the same workload, each step a bounded sample of it; a deliberately slow
baseline, not the target.

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (the R ranks of the method are slots of one GPU;
nothing crosses GPUs), timing is max over ranks and ``value`` sums the ranks'
bytes.
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
DATA = "synthetic (seeded SplitMix64 + Box-Muller, bf16 RNE)"


def algorithmic_bytes(R, N, K, B):
    """Bytes the fused call must move: W (N x K bf16 over all ranks), x
    (B x K bf16), the fp32 partials of every rank written and read back
    (2 * R * B * N * 4) and the bf16 result in R slots (R * B * N * 2)."""
    return N * K * 2 + B * K * 2 + 2 * R * B * N * 4 + R * B * N * 2


def allreduce_bytes(R, n, op="one_shot"):
    """All-reduce (one- or two-shot): R inputs of n bf16 read, R outputs
    written.  Reduce-scatter: R inputs read, one block of n / R written per
    rank (n elements in all)."""
    if op == "reduce_scatter":
        return R * n * 2 + n * 2
    return 2 * R * n * 2


def gemv_rs_bytes(R, N, K, B):
    """Fused layer ending in a reduce-scatter: as algorithmic_bytes, but each
    output row is stored once (in its owner's slot): B * N * 2."""
    return N * K * 2 + B * K * 2 + 2 * R * B * N * 4 + B * N * 2


def gemv_rmsnorm_bytes(R, N, K, B):
    """Fused layer + bias + RMSNorm: algorithmic_bytes plus bias and gamma
    (N bf16 each)."""
    return algorithmic_bytes(R, N, K, B) + 2 * N * 2


def ar_rmsnorm_bytes(R, rows, H):
    """All-reduce + bias + RMSNorm: R inputs read, R outputs written, bias and
    gamma read (H bf16 each)."""
    return 2 * R * rows * H * 2 + 2 * H * 2


def tile_bytes(R, rows, cols, ntiles):
    """Tile reduce: per tile R input tiles read, one output tile written."""
    return ntiles * (R + 1) * rows * cols * 2


def workload(name):
    """A named workload (synth.WORKLOADS), or "gemv:R,N,K,B": the fused GEMV +
    all-reduce of that shape on seeded inputs (W ~ N(0, 0.01), x ~ N(0, 1))."""
    import synth

    if name.startswith("gemv:"):
        try:
            R, N, K, B = (int(v) for v in name[len("gemv:"):].split(","))
        except ValueError:
            raise SystemExit(f"workload {name!r}: expected gemv:R,N,K,B") from None
        if not (1 <= R <= 64 and N >= 1 and K >= R and K % R == 0 and (K // R) % 8 == 0 and 1 <= B <= 16):
            raise SystemExit(f"workload {name!r}: needs 1 <= R <= 64, K a multiple of R with K/R a multiple "
                             "of 8, N >= 1 and 1 <= B <= 16")
        return dict(kind="gemv", R=R, N=N, K=K, B=B, seed=5, w_std=0.01, x="normal")
    if name not in synth.WORKLOADS:
        raise SystemExit(f"unknown workload {name!r}: one of {sorted(synth.WORKLOADS)} or gemv:R,N,K,B")
    return dict(synth.WORKLOADS[name])


def workload_bytes(w, ar_op="one_shot"):
    k = w["kind"]
    if k == "allreduce":
        return allreduce_bytes(w["R"], w["n"], ar_op)
    if k == "gemv_rs":
        return gemv_rs_bytes(w["R"], w["N"], w["K"], w["B"])
    if k == "gemv_rmsnorm":
        return gemv_rmsnorm_bytes(w["R"], w["N"], w["K"], w["B"])
    if k == "ar_rmsnorm":
        return ar_rmsnorm_bytes(w["R"], w["rows"], w["H"])
    if k == "tile":
        return tile_bytes(w["R"], w["rows"] // 2, w["cols"] // 2, 4)
    return algorithmic_bytes(w["R"], w["N"], w["K"], w["B"])


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def max_over_ranks(values, world, device=None):
    """Element-wise max of a list of floats over all ranks (identity at N=1)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    if device is not None:
        t = t.to(device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def _p10_p90(values):
    v = sorted(values)
    return v[int(0.1 * (len(v) - 1))], v[int(0.9 * (len(v) - 1))]


def throughput_gbs(nbytes, ms, world=1):
    """Whole-job GB/s: every rank moved `nbytes` in `ms` (the max over ranks)."""
    return world * nbytes / (ms * 1e-3) / 1e9


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
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


# --------------------------------------------------------- GPU arm pieces


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
    on the kernel sources as they are now."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[kernel][workload_name]
        if e.get("source_sha") == source_sha:
            return e["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


# Device-code files each kernel is built from (the host runtime, which only
# plans and launches, is left out).
KERNEL_SOURCES = {
    "gemv_ar_ffma_kernel": ("gemv_ffma.cu",),
    "gemv_ar_dyn_kernel": ("gemv_dyn.cu", "sm100.cuh"),
    "gemv_ar_cluster_kernel": ("gemv_cluster.cu", "sm100.cuh"),
    "one_shot_ar_kernel": ("allreduce.cu",),
    "one_shot_ar_staged_kernel": ("allreduce.cu", "sm100.cuh"),
    "reduce_scatter_kernel": ("allreduce.cu",),
    "all_gather_blocks_kernel": ("allreduce.cu",),
    "rmsnorm_rows_kernel": ("rmsnorm.cu",),
    "tile_reduce_kernel": ("tile_reduce.cu",),
}


def kernel_source_sha(kernel=None):
    """Hash of the device code a kernel is built from: its own file plus the
    shared headers (protocol.cuh, internal.h).  `kernel` is a kernel name as
    the bench reports it (template arguments and '+second kernel' ignored);
    None hashes every device-code file."""
    import hashlib

    csrc = os.path.join(ROOT, "collective_split_gemv_gb300", "csrc")
    if kernel is None:
        files = sorted(f for f in os.listdir(csrc) if f != "symm_runtime.cu")
    else:
        files = {"protocol.cuh", "internal.h"}
        for part in kernel.split("+"):           # a step of two kernels hashes both
            files |= set(KERNEL_SOURCES.get(part.split("<")[0], ()))
        files = sorted(files)
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def kernel_name(plan):
    if plan["path"] == 1:
        return "gemv_ar_ffma_kernel"
    if plan["path"] == 5:
        return "gemv_ar_cluster_kernel"
    engine = "tcgen05"
    cl = f",cluster={plan['cluster']}" if plan.get("cluster") else ""
    return f"gemv_ar_dyn_kernel<{engine},slabs={plan['slabs']},ctas_per_sm={plan['ctas_per_sm']}{cl}>"


def timed_loop(step, n_steps, n_warmup, stream, dev, world, flush_buf, gpu_id, per_launch=True):
    """Warm up, then time exactly n_steps calls of step(i) on `stream`, each
    bracketed by CUDA events (per_launch; otherwise only the region is timed,
    so that nothing separates consecutive launches on the stream); clocks
    sampled during the region.  Returns (step_ms, launch_ms list, clocks)."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(n_warmup):
            if flush_buf is not None:
                flush_buf.fill_(i & 0xFF)
            step(i)
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(n_steps):
            if flush_buf is not None:
                flush_buf.fill_(i & 0xFF)
            if per_launch:
                starts[i].record(stream)
            step(i)
            if per_launch:
                ends[i].record(stream)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if not per_launch:
        region = t0.elapsed_time(t1) / n_steps
        return region, [region] * n_steps, clocks
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # with L2 flushes inside the region, a step's time is its launch's own
    step_ms = (sum(launch_ms) / len(launch_ms)) if flush_buf is not None else t0.elapsed_time(t1) / n_steps
    return step_ms, launch_ms, clocks


def empty_launch_floor(stream, dev, flush_buf, n=50):
    """CUDA-event time of an empty kernel (torch.cuda._sleep(0)) launched in
    the per-launch pattern of timed_loop (events around each launch, the L2
    flush between launches where there is one): the launch and completion
    cost that every per-launch figure carries whatever the kernel does."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(n):
            if flush_buf is not None:
                flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            torch.cuda._sleep(0)
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return statistics.median(s.elapsed_time(e) for s, e in zip(starts, ends))


def gpu_bound_region(fn, n_steps, stream, dev, world, sleep_ms=20.0):
    """Per-step time of fn(0..n-1) as the GPU runs them back to back: the
    steps are enqueued behind a sleep kernel, so the host's launch rate does
    not set the pace, and timed from an event after the sleep.  Returns
    (ms per step, whether the host fell behind the sleep)."""
    import torch

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(sleep_ms * 1e-3 * 2.2e9))    # at most this many SM cycles
        t = time.perf_counter()
        a.record(stream)
        for i in range(n_steps):
            fn(i)
        b.record(stream)
        host_ms = (time.perf_counter() - t) * 1e3
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / n_steps, host_ms > 0.5 * sleep_ms


def chunked_spread(step, n_steps, stream, dev, world, chunk=None):
    """The same n_steps chained calls once more, with an event after every
    `chunk` calls (each event ends one chain: the call after it starts in
    plain stream order).  Returns the per-call time of every chunk (ms), from
    which the bench reports median and p10 / p90 of chained calls."""
    import torch

    chunk = chunk or max(5, n_steps // 10)
    bounds = list(range(0, n_steps, chunk)) + [n_steps]
    evs = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for j in range(1, len(bounds)):
            for i in range(bounds[j - 1], bounds[j]):
                step(i)
            evs[j].record(stream)
    torch.cuda.synchronize(dev)
    return [evs[j - 1].elapsed_time(evs[j]) / (bounds[j] - bounds[j - 1]) for j in range(1, len(bounds))], chunk


def _pinned(a):
    import numpy as np
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.uint8).reshape(-1).pin_memory()


def _copies_for(per_copy):
    """Rotating input copies so that the bytes touched between two uses of a
    copy exceed the L2 three times over (at most 8)."""
    return max(1, min(8, math.ceil(3 * L2_BYTES / max(per_copy, 1))))


def make_case(args, w, local_rank, stream):
    """Workspace, inputs and the per-step call of one workload.  Returns a dict:
    ws, step(i) (copy i % copies), run0() (copy 0, for the end-to-end leg),
    in_host / in_dst / in_bytes (per-step inputs for the end-to-end leg: one
    pinned buffer of R blocks, their symmetric destination and the bytes per
    rank), out_src / out_bytes (the result in slot 0, read back), kernel, config, per_copy, copies,
    launches_per_step, W (GEMV weights, for the weights-from-host leg), read_out() (every slot's
    result), producer() (GEMV: one kernel rewriting every rank's x in place, for the in-step leg)."""
    import collective_split_gemv_gb300 as csg
    import synth
    from collective_split_gemv_gb300.workspace import (AllReduceWorkspace, GemvWorkspace, RmsNormWorkspace,
                                                       TileWorkspace)

    kind, R = w["kind"], w["R"]
    if kind in ("gemv", "gemv_rs", "gemv_rmsnorm"):
        N, K, B = w["N"], w["K"], w["B"]
        W, x = synth.gemv_inputs(R, N, K, B, w["seed"], w["w_std"], w["x"])
        copies = _copies_for(W.nbytes)
        paths = {"auto": csg.GEMV_PATH_AUTO, "ffma": csg.GEMV_PATH_FFMA, "dyn": csg.GEMV_PATH_DYN,
                 "cluster": csg.GEMV_PATH_CLUSTER}

        def gemv_ws(packed):
            ws_ = GemvWorkspace(R, N, K, B, copies=copies, device=local_rank, packed=packed)
            for opt, val in ((csg.SYMM_OPT_GEMV_PATH, paths[args.gemv_path]), (csg.SYMM_OPT_SK_SLABS, args.sk_slabs),
                             (csg.SYMM_OPT_SK_ENGINE, args.sk_engine), (csg.SYMM_OPT_SK_CTAS_PER_SM, args.sk_cps),
                             (csg.SYMM_OPT_SK_GRID, args.sk_grid), (csg.SYMM_OPT_DYN_SPLITS, args.dyn_splits),
                             (csg.SYMM_OPT_NORM_PDL, args.norm_pdl), (csg.SYMM_OPT_CHAIN, int(args.chain)),
                             (csg.SYMM_OPT_DYN_CLUSTER, args.dyn_cluster)):
                csg.symm_set_option(ws_.h, opt, val)
            return ws_

        ws = gemv_ws(False)
        plan = csg.symm_gemv_plan(ws.h, N, K, B)
        # Packed weights (made once by symm_pack_w, as at model load) wherever
        # the call runs on the persistent kernel, the only one that reads them;
        # the row-major weights are kept and timed beside them.
        ws_rm = None
        if args.w_layout == "packed" and plan["path"] == csg.GEMV_PATH_DYN:
            ws_rm, ws = ws, gemv_ws(True)
        for c in range(copies):
            ws.load_W(W, copy=c)
            if ws_rm is not None:
                ws_rm.load_W(W, copy=c)
        ws.load_x(x)
        if ws_rm is not None:
            ws_rm.load_x(x)
        mode = {"gemv": "all_reduce", "gemv_rs": "reduce_scatter", "gemv_rmsnorm": "bias_rmsnorm"}[kind]
        eps = w.get("eps", 1e-6)
        if kind == "gemv_rmsnorm":
            ws.load_vectors(*synth.norm_vectors(N, w["seed"]))
            if ws_rm is not None:
                ws_rm.load_vectors(*synth.norm_vectors(N, w["seed"]))
            # the planner reserves z at the top of the scratch region; the plan
            # shown is that of the all-reduce form of the same shape
        kernel = kernel_name(plan) + ("+rmsnorm_rows_kernel<z>" if kind == "gemv_rmsnorm" else "")
        out_rows = B // R if kind == "gemv_rs" else B
        # The layer's input written by a kernel of another library just before
        # the call (as the previous layer's kernel would): one strided copy of
        # the same bytes into every rank's x.
        import numpy as np
        import torch

        dev = torch.device("cuda", local_rank)
        span = (R - 1) * ws.stride + ws.x_off + ws.x_bytes
        slots_u8 = torch.as_tensor(csg.DeviceView(ws.base, (span,)), device=dev)
        x_slots = torch.as_strided(slots_u8, (R, ws.x_bytes), (ws.stride, 1), ws.x_off)
        x_src = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8).reshape(R, -1)).to(dev)
        return {
            "ws": ws, "W": W, "copies": copies, "per_copy": W.nbytes, "kernel": kernel,
            "step": lambda i: ws.run(stream, copy=i % copies, mode=mode, eps=eps),
            "run0": lambda: ws.run(stream, copy=0, mode=mode, eps=eps),
            "ws_rm": ws_rm,
            "rm_step": (None if ws_rm is None else lambda i: ws_rm.run(stream, copy=i % copies, mode=mode, eps=eps)),
            # e2e: per-step inputs are x_r (W_r are resident model weights); result y
            "in_host": _pinned(x), "in_dst": ws.x_ptr(), "in_bytes": ws.x_bytes,
            "out_src": ws.y_ptr(), "out_bytes": out_rows * N * 2,
            "read_out": ws.read_y_rs if kind == "gemv_rs" else ws.read_y,
            "producer": lambda: x_slots.copy_(x_src),
            "launches_per_step": 2 if kind == "gemv_rmsnorm" else 1,
            "config": {"R": R, "N": N, "K": K, "K_per_rank": K // R, "B": B, "plan": plan,
                       "w_layout": ("packed (symm_pack_w once at load, untimed; the same bytes per call)"
                                    if ws.packed else "row-major N x K/R per slot"),
                       "chain_option": bool(args.chain),
                       **({"eps": eps, "norm_pdl": args.norm_pdl} if kind == "gemv_rmsnorm" else {})},
        }
    if kind == "allreduce":
        n, op = w["n"], args.ar_op
        inp = synth.allreduce_inputs(R, n, w["seed"])
        copies = _copies_for(inp.nbytes * 2)    # R inputs read + R outputs written, both rotated
        ws = AllReduceWorkspace(R, n, device=local_rank, copies=copies)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_AR_CTAS_PER_SM, args.ar_cps)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_AR_KERNEL, args.ar_kernel)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, int(args.chain))
        for c in range(copies):
            ws.load_in(inp, copy=c)
        out_n = n // R if op == "reduce_scatter" else n
        staged = args.ar_kernel == csg.AR_KERNEL_STAGED   # the library's automatic choice is per-thread
        kernel = {"one_shot": "one_shot_ar_staged_kernel" if staged else "one_shot_ar_kernel",
                  "reduce_scatter": "reduce_scatter_kernel",
                  "two_shot": "reduce_scatter_kernel+all_gather_blocks_kernel"}[op]
        return {
            "ws": ws, "copies": copies, "per_copy": inp.nbytes * 2, "kernel": kernel,
            "step": lambda i: ws.run(stream, copy=i % copies, op=op),
            "run0": lambda: ws.run(stream, copy=0, op=op),
            "in_host": _pinned(inp), "in_dst": ws.base + ws.in_offs[0], "in_bytes": ws.bytes,
            "out_src": ws.base + ws.out_offs[0], "out_bytes": out_n * 2,
            "read_out": lambda: ws.read_out(copy=0, count=out_n),
            "launches_per_step": 2 if op == "two_shot" else 1,
            "chainable": True,
            "config": {"R": R, "n": n, "op": op, **({"ar_kernel": "staged" if staged else "per_thread"}
                                                    if op == "one_shot" else {})},
        }
    if kind == "ar_rmsnorm":
        rows, H, eps = w["rows"], w["H"], w["eps"]
        inp, bias, gamma = synth.rmsnorm_inputs(R, rows, H, w["seed"])
        copies = _copies_for(inp.nbytes * 2)
        ws = RmsNormWorkspace(R, rows, H, copies=copies, device=local_rank)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, int(args.chain))
        for c in range(copies):
            ws.load(inp, bias, gamma, copy=c)
        return {
            "ws": ws, "copies": copies, "per_copy": inp.nbytes * 2, "kernel": "rmsnorm_rows_kernel<slots>",
            "step": lambda i: ws.run(stream, copy=i % copies, eps=eps),
            "run0": lambda: ws.run(stream, copy=0, eps=eps),
            "in_host": _pinned(inp), "in_dst": ws.base + ws.in_offs[0], "in_bytes": ws.bytes,
            "out_src": ws.base + ws.out_offs[0], "out_bytes": ws.bytes,
            "read_out": lambda: ws.read_out(copy=0),
            "launches_per_step": 1,
            "config": {"R": R, "rows": rows, "H": H, "eps": eps},
        }
    if kind == "tile":
        n = w["rows"]
        h = n // 2
        full = synth.tile_inputs(R, n, w["cols"], w["seed"])
        copies = _copies_for(full.nbytes)
        ws = TileWorkspace(R, n, w["cols"], h, w["cols"] // 2, copies=copies, device=local_rank)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, int(args.chain))
        for c in range(copies):
            ws.load_in(full, copy=c)
        tiles = [(0, 0), (0, h), (h, 0), (h, h)]
        roots = [0, 1, 2, 3]
        return {
            "ws": ws, "copies": copies, "per_copy": full.nbytes, "kernel": "tile_reduce_kernel",
            "step": lambda i: ws.run(tiles, roots, h, w["cols"] // 2, stream=stream, copy=i % copies),
            "run0": lambda: ws.run(tiles, roots, h, w["cols"] // 2, stream=stream, copy=0),
            "in_host": _pinned(full), "in_dst": ws.base + ws.in_offs[0], "in_bytes": ws.in_bytes,
            "out_src": ws.base + ws.out_offs[0], "out_bytes": ws.out_bytes,
            "launches_per_step": 1,
            "chainable": True,
            "config": {"R": R, "tensor": [n, w["cols"]], "tiles": "four quadrants", "roots": roots},
        }
    raise SystemExit(f"unknown workload kind {kind!r}")


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import __graft_entry__
    import collective_split_gemv_gb300 as csg

    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()   # the other ranks load what rank 0 built
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = str(local_rank) if not visible else visible.split(",")[local_rank].strip()
    w = workload(args.workload)
    nbytes = workload_bytes(w, args.ar_op)
    stream = torch.cuda.Stream(device=dev)
    R = w["R"]

    c = make_case(args, w, local_rank, stream)
    ws, step, run0, kernel = c["ws"], c["step"], c["run0"], c["kernel"]
    in_host, in_dst, in_bytes = c["in_host"], c["in_dst"], c["in_bytes"]
    out_src, out_bytes = c["out_src"], c["out_bytes"]
    config_extra, per_copy, copies, W = c["config"], c["per_copy"], c["copies"], c.get("W")

    working_set = copies * per_copy
    flush = working_set < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    # Every call chains (the library default); region timing is used only
    # where no L2 flush sits between the launches.
    chained = args.chain and flush_buf is None and (W is not None or c.get("chainable", False))
    # Chained calls are timed over the region only: an event between two
    # launches would separate them on the stream.
    step_ms, launch_ms, clocks = timed_loop(step, args.steps, args.warmup, stream, dev, world, flush_buf, gpu_id,
                                            per_launch=not chained)
    floor_ms = empty_launch_floor(stream, dev, flush_buf)
    unchained = None
    spread = None
    if chained:
        # the spread of chained calls: the same calls timed in chunks
        chunk_ms, chunk = chunked_spread(step, args.steps, stream, dev, world)
        spread = (max_over_ranks(chunk_ms, world, dev), chunk)
        # the same calls in plain stream order, each bracketed by events
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 0)
        u_step, u_launch, _ = timed_loop(step, args.steps, args.warmup, stream, dev, world, flush_buf, gpu_id)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        unchained = (u_step, statistics.mean(u_launch), statistics.median(u_launch), _p10_p90(u_launch))
    in_step = None
    if chained and c.get("producer") is not None:
        # The call inside a step: another library's kernel writes the layer's
        # input x into the R slots, then the call (chained, the library
        # default; the producer does not release it early, so the call pays
        # its own start-up).  Its cost is the step's time minus the
        # producer's alone, both as the GPU runs the steps back to back (no
        # event between launches, and not paced by the host's launches).
        prod = c["producer"]
        n_in = min(args.steps, 200)
        with torch.cuda.stream(stream):
            for i in range(min(args.warmup, 10)):
                prod()
                step(i)
        ps_ms, host_a = gpu_bound_region(lambda i: (prod(), step(i)), n_in, stream, dev, world)
        p_ms, host_b = gpu_bound_region(lambda i: prod(), n_in, stream, dev, world)
        in_step = (ps_ms, p_ms, n_in, host_a or host_b)
    code, _, _ = csg.symm_status(ws.h, stream)
    if code != csg.SYMM_OK:
        raise SystemExit(f"protocol error in the timed region: {csg.symm_last_error()}")
    row_major = None
    if c.get("rm_step") is not None:
        # the same calls on the row-major weights (chained like the main leg)
        rm_step_ms, rm_launch, _ = timed_loop(c["rm_step"], args.steps, args.warmup, stream, dev, world, flush_buf,
                                              gpu_id, per_launch=not chained)
        code, _, _ = csg.symm_status(c["ws_rm"].h, stream)
        if code != csg.SYMM_OK:
            raise SystemExit(f"protocol error in the row-major leg: {csg.symm_last_error()}")
        row_major = statistics.mean(rm_launch)
        c["ws_rm"].close()
    unfused = None
    if w["kind"] == "gemv" and c.get("ws") is not None and csg.symm_gemv_plan(ws.h, w["N"], w["K"], w["B"])["path"] == \
            csg.GEMV_PATH_DYN:
        # What fusion buys: the same calls unfused (the GEMV storing every
        # rank's fp32 partials, then a separate all-reduce kernel of them),
        # timed like the main leg.
        # (The unfused form has no tile reduction, so no cluster epilogue either.)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, 1)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, -1)
        uf_step, uf_launch, _ = timed_loop(step, args.steps, args.warmup, stream, dev, world, flush_buf, gpu_id,
                                           per_launch=not chained)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, 0)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, args.dyn_cluster)
        code, _, _ = csg.symm_status(ws.h, stream)
        if code != csg.SYMM_OK:
            raise SystemExit(f"protocol error in the unfused leg: {csg.symm_last_error()}")
        unfused = statistics.mean(uf_launch)

    # ---- e2e: the same call through the ABI with host buffers every step ----
    # Each step: one strided copy of the step's inputs from pinned host memory
    # into the R slots, the call, one copy of the result (slot 0) back, and a
    # stream synchronisation.  The library copies pinned buffers with a kernel
    # (the SMs read and write host memory over the CPU-GPU link), so a step is
    # a chain of three kernels; --copy-engine 1 takes copy-engine copies.
    csg.symm_set_option(ws.h, csg.SYMM_OPT_COPY_ENGINE, args.copy_engine)
    out_host = torch.empty(max(out_bytes, 1), dtype=torch.uint8).pin_memory()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step(extra=None):
        if extra is not None:
            extra()
        csg.symm_copy_to_slots(ws.h, in_dst, in_host.data_ptr(), in_bytes, R, stream)
        run0()
        csg.symm_copy_from_slots(ws.h, out_host.data_ptr(), out_src, out_bytes, 1, stream)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    tt = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - tt) * 1e3 / e2e_steps
    h2d = in_bytes * R
    eager_out = out_host.clone()

    # The same step captured once into a CUDA graph (copy in, call, copy
    # out) and replayed: one graph launch per step instead of three calls.
    # The fused calls keep their protocol state in the signal pad, so the
    # replays are ordinary launches of the protocol.
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph, stream=stream):
        csg.symm_copy_to_slots(ws.h, in_dst, in_host.data_ptr(), in_bytes, R, stream)
        run0()
        csg.symm_copy_from_slots(ws.h, out_host.data_ptr(), out_src, out_bytes, 1, stream)
    out_host.zero_()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
            stream.synchronize()
        torch.cuda.synchronize(dev)
        tt = time.perf_counter()
        for i in range(e2e_steps):
            graph.replay()
            stream.synchronize()
        e2e_graph_ms = (time.perf_counter() - tt) * 1e3 / e2e_steps
    if not torch.equal(out_host, eager_out):
        raise SystemExit("the replayed step's result differs from the eager step's")
    del graph

    ew = None
    if W is not None:
        # weights streamed from the host as well (every step copies all W_r)
        W_host = _pinned(W)
        w_bytes = W.nbytes // R
        ew_steps = max(3, min(args.steps, 10))
        torch.cuda.synchronize(dev)
        tt = time.perf_counter()
        if ws.packed:   # the row-major weights into the staging copy, then packed, every step
            def put_w():
                csg.symm_copy_to_slots(ws.h, ws.W_rowmajor_ptr(), W_host.data_ptr(), w_bytes, R, stream)
                ws.pack(0, stream)
        else:
            def put_w():
                csg.symm_copy_to_slots(ws.h, ws.W_ptr(0), W_host.data_ptr(), w_bytes, R, stream)
        for i in range(ew_steps):
            e2e_step(put_w)
        ew = (time.perf_counter() - tt) * 1e3 / ew_steps
    code, _, _ = csg.symm_status(ws.h, stream)
    assert code == csg.SYMM_OK

    (step_ms, e2e_ms, ew_ms, mean_launch_ms, u_step_ms, u_launch_ms, e2e_graph_ms, rm_ms, uf_ms, ps_ms,
     p_ms) = max_over_ranks(
        [step_ms, e2e_ms, ew if ew is not None else 0.0, statistics.mean(launch_ms),
         unchained[0] if unchained else 0.0, unchained[1] if unchained else 0.0, e2e_graph_ms,
         row_major if row_major is not None else 0.0, unfused if unfused is not None else 0.0,
         in_step[0] if in_step else 0.0, in_step[1] if in_step else 0.0], world, dev)
    # the last call's result (every slot; all legs computed it from the same
    # inputs), for the oracle leg's check -- read before the handle is freed
    gpu_out = None
    if rank == 0 and not args.no_cpu_baseline and c.get("read_out") is not None:
        gpu_out = c["read_out"]()
    ws.close()
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes / (mean_launch_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(throughput_gbs(nbytes, step_ms, world), 2),
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
        "data": DATA,
        "config": {
            "workload": args.workload, **config_extra,
            "algorithmic_bytes_per_call": nbytes,
            "l2": (f"L2 flushed (2x{L2_BYTES // 10**6} MB write) between launches; step time = kernel time"
                   if flush else
                   f"inputs larger than L2: {copies} rotating copies ({working_set / 1e9:.2f} GB)"),
            "parallelism": "R ranks as symmetric slots on one GPU" + (f"; {world} independent replicas"
                                                                     if world > 1 else ""),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": kernel,
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": ("measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "fallback 6.8 TB/s"),
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(kernel, args.workload, kernel_source_sha(kernel)),
            "mean_launch_us": round(mean_launch_ms * 1e3, 3),
            "median_launch_us": round(statistics.median(spread[0] if spread else launch_ms) * 1e3, 3),
            "p10_p90_launch_us": [round(q * 1e3, 3) for q in _p10_p90(spread[0] if spread else launch_ms)],
            "empty_launch_us": round(floor_ms * 1e3, 3),
            "timing": ((f"chained calls: region time / steps (events around the region only); median and "
                        f"p10 / p90 over {len(spread[0])} chunks of {spread[1]} chained calls timed again "
                        f"(an event after each chunk)") if chained
                       else "CUDA events around every launch on the launching stream"),
        },
        "clocks": clocks,
        "e2e": {
            "value": round(throughput_gbs(nbytes, e2e_ms, world), 2), "unit": "GB/s",
            "us_per_call": round(e2e_ms * 1e3, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_bytes,
            "what": ("per step: the inputs H2D from pinned memory into the R slots (symm_copy_to_slots), the "
                     "call, the result (slot 0) D2H (symm_copy_from_slots), stream synchronised; the copies "
                     + ("by the copy engine" if args.copy_engine else
                        "by a kernel reading / writing the pinned buffers over the CPU-GPU link")
                     + ("; W_r resident (model weights)" if W is not None else "")),
        },
        "e2e_graph": {
            "value": round(throughput_gbs(nbytes, e2e_graph_ms, world), 2), "unit": "GB/s",
            "us_per_call": round(e2e_graph_ms * 1e3, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_bytes,
            "what": ("the e2e step (copy in, call, copy out) captured once into a CUDA graph and replayed "
                     "each step, stream synchronised; result checked equal to the eager step's"),
        },
        "gpu_launches": args.steps * c["launches_per_step"],
    }
    if unchained is not None:
        line["unchained"] = {
            "what": "the same calls in plain stream order (SYMM_OPT_CHAIN 0), events around every launch",
            "us_per_call": round(u_step_ms * 1e3, 3), "mean_launch_us": round(u_launch_ms * 1e3, 3),
            "median_launch_us": round(unchained[2] * 1e3, 3),
            "p10_p90_launch_us": [round(q * 1e3, 3) for q in unchained[3]],
            "achieved": round(nbytes / (u_launch_ms * 1e-3) / 1e9, 1),
            "frac": round(nbytes / (u_launch_ms * 1e-3) / 1e9 / peak, 4),
        }
    if in_step is not None:
        call_ms = ps_ms - p_ms
        line["in_step"] = {
            "what": ("each step: one kernel of another library writes the layer's input x into the R slots "
                     "(as the previous layer's kernel would), then the call; per call = the step's time minus "
                     "the producer's alone, each over a region of steps the GPU runs back to back (enqueued "
                     "behind a sleep kernel; no event between launches)"),
            "steps": in_step[2], "host_fell_behind": in_step[3],
            "us_per_call": round(call_ms * 1e3, 3), "producer_us": round(p_ms * 1e3, 3),
            "achieved": round(nbytes / (call_ms * 1e-3) / 1e9, 1),
            "frac": round(nbytes / (call_ms * 1e-3) / 1e9 / peak, 4),
        }
    if row_major is not None:
        line["row_major_w"] = {
            "what": "the same calls with W_r row-major (no symm_pack_w), timed like the main leg",
            "us_per_call": round(rm_ms * 1e3, 3),
            "achieved": round(nbytes / (rm_ms * 1e-3) / 1e9, 1),
            "frac": round(nbytes / (rm_ms * 1e-3) / 1e9 / peak, 4),
        }
    if unfused is not None:
        line["unfused"] = {
            "what": ("the same calls unfused (SYMM_OPT_UNFUSED: the GEMV kernel storing every rank's fp32 partials, "
                     "then a separate all-reduce kernel over them; the same bits), timed like the main leg"),
            "us_per_call": round(uf_ms * 1e3, 3),
            "fused_saving_pct": round(100.0 * (uf_ms - mean_launch_ms) / uf_ms, 2),
            "pages_claim": "13-22 % lower execution time for the fused GEMV + AllReduce (hardware not named)",
        }
    if ew is not None:
        line["e2e_weights_from_host"] = {
            "value": round(throughput_gbs(nbytes, ew_ms, world), 2), "unit": "GB/s",
            "us_per_call": round(ew_ms * 1e3, 2),
            "h2d_bytes_per_step": W.nbytes + h2d, "d2h_bytes_per_step": out_bytes,
            "what": ("the e2e step with every rank's W_r copied from pinned host memory into the slots as well"
                     + (", then packed (symm_pack_w)" if ws.packed else "")),
        }
    if not args.no_cpu_baseline:
        cb = cpu_baseline(args.workload, budget_s=args.cpu_seconds, ar_op=args.ar_op, gpu_out=gpu_out)
        parity = cb.pop("parity", None)
        if cb["cores"] > 1:   # the same oracle on one core, a shorter sample
            one = cpu_baseline(args.workload, budget_s=min(args.cpu_seconds, 4.0), ar_op=args.ar_op, threads=1)
            cb["one_thread"] = {k: one[k] for k in ("value", "unit", "us_per_call_equiv", "cores", "sample")}
        line["cpu_baseline"] = cb
        if parity is not None:
            line["parity"] = parity
    return line


# ------------------------------------------------------------ CPU oracle


def cpu_baseline(name, budget_s=10.0, steps=None, warmup=0, ar_op="one_shot", threads=None, gpu_out=None):
    """Time the oracle (as it is) on this host's cores on the workload: with
    `steps` None, repeat the full call for about `budget_s` seconds; else run
    exactly `steps` calls, each on a row sample sized so that all of them fit
    in about `budget_s`.  Returns the cpu_baseline object (GB/s of algorithmic
    bytes, the time scaled to a full call).  `threads`: the oracle's threads
    where it is multithreaded (None: every host core); `cores` in the result
    is what the call actually used.  `gpu_out`: the GPU path's last result on
    the same inputs, every slot's words; the object then carries `parity`,
    that result checked against the oracle's on the sample (after the
    timing)."""
    import numpy as np

    import oracle
    import synth

    w = workload(name)
    threads = host_cores() if threads is None else threads
    used = threads
    nbytes = workload_bytes(w, ar_op)
    kind, R = w["kind"], w["R"]
    # make(rows) prepares a sample of the call's inputs (the first `rows`
    # rows, made contiguous: input preparation, outside the timed loop) and
    # returns the oracle call on it.
    if kind == "allreduce":
        inp = synth.allreduce_inputs(R, w["n"], w["seed"])
        full = inp.shape[1]
        if ar_op == "reduce_scatter":
            used = 1    # single-threaded oracle function

            def make(rows):   # rows: a multiple of R (rounded below)
                part = np.ascontiguousarray(inp[:, :rows])
                return lambda: oracle.reduce_scatter(part)
        else:   # the two-shot all-reduce reaches the all-reduce definition
            def make(rows):
                part = np.ascontiguousarray(inp[:, :rows])
                return lambda: oracle.one_shot_all_reduce(part, threads=threads)
        unit = "elements per slot"
    elif kind == "ar_rmsnorm":
        inp, bias, gamma = synth.rmsnorm_inputs(R, w["rows"], w["H"], w["seed"])
        full = w["rows"]
        used = 1

        def make(rows):
            part = np.ascontiguousarray(inp[:, :rows])
            return lambda: oracle.all_reduce_bias_rmsnorm(part, bias, gamma, w["eps"])
        unit = "rows"
    elif kind == "tile":
        used = 1
        h = w["rows"] // 2
        full_t = synth.tile_inputs(R, w["rows"], w["cols"], w["seed"])
        flat = full_t.reshape(R, -1)
        out = np.zeros((R, h * (w["cols"] // 2)), dtype=np.uint16)
        offs = [0, h, h * w["cols"], h * w["cols"] + h]
        full = h

        def make(rows):
            return lambda: oracle.tile_reduce(flat, out, offs, 0, [0, 1, 2, 3], rows, w["cols"] // 2, w["cols"],
                                              w["cols"] // 2)
        unit = "tile rows"
    else:
        W, x = synth.gemv_inputs(R, w["N"], w["K"], w["B"], w["seed"], w["w_std"], w["x"])
        full = w["N"]
        if kind == "gemv_rs":
            def make(rows):
                part = np.ascontiguousarray(W[:, :rows])
                return lambda: oracle.gemv_reduce_scatter(part, x, threads=threads)
        elif kind == "gemv_rmsnorm":
            bias, gamma = synth.norm_vectors(w["N"], w["seed"])

            def make(rows):
                part = np.ascontiguousarray(W[:, :rows])
                return lambda: oracle.gemv_bias_rmsnorm(part, x, bias[:rows], gamma[:rows], w["eps"],
                                                        threads=threads)
        else:
            def make(rows):
                part = np.ascontiguousarray(W[:, :rows])
                return lambda: oracle.gemv_all_reduce(part, x, threads=threads)
        unit = "rows"
    call = make(full)
    t = time.perf_counter()
    call()                                      # calibration: one full call
    t_full = max(time.perf_counter() - t, 1e-6)
    if steps is None:
        rows = full if t_full <= budget_s else max(1, int(full * budget_s / t_full))
        reps = max(1, int(budget_s / (t_full * rows / full)))
    else:
        per_step = budget_s / max(1, steps + warmup)
        rows = max(1, min(full, int(full * per_step / t_full)))
        reps = steps
    if kind == "allreduce" and ar_op == "reduce_scatter":
        rows = min(full, max(R, rows // R * R))   # whole owner blocks
    if rows != full:
        call = make(rows)
    if steps is not None:
        for _ in range(warmup):
            call()
    t = time.perf_counter()
    for _ in range(reps):
        call()
    el = time.perf_counter() - t
    parity = None
    if gpu_out is not None:
        parity = parity_check(kind, ar_op, call(), np.asarray(gpu_out), rows, full, R, unit)
    sec_per_call = el / reps * full / rows
    return {
        "value": round(nbytes / sec_per_call / 1e9, 4),
        "unit": "GB/s",
        "us_per_call_equiv": round(sec_per_call * 1e6, 1),
        "cores": used,
        "kind": "oracle",
        "sample": (f"{rows} of {full} {unit} of {name}, {reps} repetitions, {el:.3f} s wall time on {used} "
                   f"thread{'s' if used != 1 else ''}; time scaled to the full call"),
        **({"parity": parity} if parity is not None else {}),
    }


# The accuracy bar of the fused call: |y - y_ref| <= REL |y_ref| + ABS rms(y_ref),
# y_ref the oracle's fp64 value before rounding.
TOL_REL, TOL_ABS = 4e-3, 1e-3


def _bf16_f64(words):
    import numpy as np

    return (np.asarray(words, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_distance(a, b):
    """Units in the last place between bf16 words, through their ordering
    as sign-magnitude integers (+0 and -0 are 0 apart)."""
    import numpy as np

    def key(w):
        w = np.asarray(w, dtype=np.uint16).astype(np.int64)
        return np.where(w & 0x8000, -(w & 0x7FFF), w)

    return np.abs(key(a) - key(b))


def tolerance_ratio(y, y_ref):
    """max over outputs of |y - y_ref| / (REL |y_ref| + ABS rms(y_ref))."""
    import numpy as np

    y_ref = np.asarray(y_ref, dtype=np.float64)
    if y_ref.size == 0:
        return 0.0
    bound = TOL_REL * np.abs(y_ref) + TOL_ABS * float(np.sqrt(np.mean(y_ref * y_ref)))
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    return float(np.max(r))


def parity_check(kind, ar_op, ref, gpu_out, rows, full, R, unit):
    """The GPU result (every slot's words) against the oracle's (y_ref fp64,
    words) on the first `rows` rows: the worst error over the tolerance, the
    fraction of outputs equal to the oracle's correctly rounded words, and
    whether the R replicas are bitwise identical.  None where a row sample of
    the form is not a sample of the full result (a normalisation over the
    whole row, a reduce-scatter's owner blocks)."""
    import numpy as np

    y_ref, words = ref
    replicas = None
    if kind in ("gemv", "gemv_rmsnorm"):
        if kind == "gemv_rmsnorm" and rows != full:
            return None
        got = gpu_out[:, :, :rows]
        replicas = bool(all(np.array_equal(got[r], got[0]) for r in range(R)))
        y, want = got[0], words[0]
    elif kind == "gemv_rs":
        got = gpu_out[:, :, :rows]                      # slot s: batch rows s*B/R ... of the sum
        y, want = got.reshape(-1, rows), np.asarray(words).reshape(-1, rows)
    elif kind == "allreduce" and ar_op != "reduce_scatter":
        got = gpu_out[:, :rows]
        replicas = bool(all(np.array_equal(got[r], got[0]) for r in range(R)))
        y, want = got[0], words[0]
    elif kind == "allreduce" and rows == full:
        y, want = gpu_out.reshape(-1), np.asarray(words).reshape(-1)
    elif kind == "ar_rmsnorm":
        got = gpu_out[:, :rows]
        replicas = bool(all(np.array_equal(got[r], got[0]) for r in range(R)))
        y, want = got[0], words[0]
    else:
        return None
    ref_v = np.asarray(y_ref).reshape(np.shape(y))
    ratio = tolerance_ratio(_bf16_f64(y), ref_v)
    ulps = ulp_distance(y, want)
    big = np.abs(ref_v) >= 0.1 * float(np.sqrt(np.mean(ref_v * ref_v)))   # outside the cancellation zone
    return {
        "checked": f"{rows} of {full} {unit}, every output of those, against the oracle (fp64)",
        "tolerance": "|y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(y_ref), y_ref before rounding",
        "max_tol_ratio": round(ratio, 4),
        "bit_equal_frac": round(float(np.mean(np.asarray(y) == np.asarray(want))), 6),
        "max_ulp": int(ulps.max(initial=0)),
        "max_ulp_where_abs_ge_0.1_rms": int(ulps[big].max(initial=0)),
        "replicas_identical": replicas,
        "passed": bool(ratio <= 1.0 and replicas is not False),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = workload(args.workload)
    cb = cpu_baseline(args.workload, budget_s=min(120.0, 2.0 * (args.steps + args.warmup)),
                      steps=args.steps, warmup=args.warmup, ar_op=args.ar_op)
    sec = cb["us_per_call_equiv"] * 1e-6
    cfg = {k: w[k] for k in ("R", "N", "K", "B", "n", "rows", "cols", "H") if k in w}
    if w["kind"] == "allreduce":
        cfg["op"] = args.ar_op
    return {
        "metric": METRIC, "impl": "reference", "value": cb["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": {"workload": args.workload, **cfg, "algorithmic_bytes_per_call": workload_bytes(w, args.ar_op)},
        "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=100)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="mlp_down_decode",
                   help="a named workload (synth.WORKLOADS) or gemv:R,N,K,B for the fused GEMV of any shape")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--gemv-path", choices=("auto", "ffma", "dyn", "cluster"), default="auto",
                   help="force one kernel (measurement only)")
    p.add_argument("--sk-slabs", type=int, default=0, choices=(0, 1, 2, 3, 4),
                   help="TMA kernels: slabs per pipeline stage (0 = library default)")
    p.add_argument("--sk-cps", type=int, default=0, choices=(0, 1, 2, 3),
                   help="TMA kernels: resident CTAs per SM (0 = library default)")
    p.add_argument("--sk-grid", type=int, default=0,
                   help="persistent kernel: grid in CTAs (0 = library default)")
    p.add_argument("--w-layout", choices=("packed", "row_major"), default="packed",
                   help="GEMV weights: packed (symm_pack_w, where the call runs on the persistent kernel) or "
                        "row-major")
    p.add_argument("--dyn-splits", type=int, default=0,
                   help="persistent kernel: K splits per (tile, rank) (0 = library default)")
    p.add_argument("--dyn-cluster", type=int, default=-1, choices=(-1, 0, 1),
                   help="persistent kernel: cluster epilogue -1 auto, 0 off, 1 on (SYMM_OPT_DYN_CLUSTER)")
    p.add_argument("--sk-engine", type=int, default=-1, choices=(-1, 0),
                   help="persistent kernel's engine: -1 auto, 0 tcgen05 (the only one)")
    p.add_argument("--ar-cps", type=int, default=0,
                   help="allreduce workload: grid cap in CTAs per SM (0 = library default)")
    p.add_argument("--copy-engine", type=int, default=0, choices=(0, 1),
                   help="end-to-end legs: 0 library default (pinned host buffers copied by a kernel), "
                        "1 the copy engine (SYMM_OPT_COPY_ENGINE)")
    p.add_argument("--ar-kernel", type=int, default=0, choices=(0, 1, 2),
                   help="allreduce workload, one-shot: 0 library default, 1 per-thread loads/stores, "
                        "2 staged through shared memory by bulk copies")
    p.add_argument("--ar-op", choices=("one_shot", "two_shot", "reduce_scatter"), default="one_shot",
                   help="allreduce workload: which collective one step calls")
    p.add_argument("--no-chain", dest="chain", action="store_false",
                   help="GEMV workloads: launch every call in plain stream order (SYMM_OPT_CHAIN 0) instead of "
                        "as a programmatic dependent of the previous call (the library default)")
    p.add_argument("--norm-pdl", type=int, default=1, choices=(0, 1),
                   help="bias + RMSNorm form: launch the normalisation stage as a programmatic dependent")
    args = p.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main():
    args = parse_args()
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
