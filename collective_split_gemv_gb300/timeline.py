"""Per-phase timeline of one launch, from the timeline build of the library.

    python -m collective_split_gemv_gb300.timeline --workload attn_out_proj [--reps 20]

Builds ``libsymm_gemv_timeline.so`` (the kernels with %globaltimer stamps at
their phase boundaries), runs the workload's call ``--reps`` times in plain
stream order with L2 flushed before each launch (or, for GEMV workloads
whose weights exceed L2, on rotating weight copies), and prints a Markdown
summary: the CUDA-event time of the launch, that of an empty kernel launched
the same way (``torch.cuda._sleep(0)``: the floor of launch and completion
outside any CTA), the span between the first CTA's entry and the last CTA's
exit, and for each phase the time after the first
CTA entry at which the CTAs reached it (min / median / max over CTAs, median
over the repetitions).  The stamps cost a few global stores per CTA, so the
times are those of a slightly slower kernel than the product build's.

Workloads are those of ``synth.WORKLOADS``; GEMV weights are packed where the
call runs on the persistent kernel, as in the bench.
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

os.environ["SYMM_GEMV_VARIANT"] = "timeline"

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1000 * 1000

# slot -> phase, per kernel (the slot lists in the kernels' sources)
PHASES = {
    "gemv_ar_ffma_kernel": {0: "entry", 1: "x staged in shared memory", 2: "dot products done",
                            3: "partial and flag stored and fenced", 4: "ticket taken",
                            5: "reducer: first loads out, launch bookkeeping done", 6: "reducer: flags checked, tile summed and stored",
                            7: "exit"},
    "gemv_ar_dyn_kernel": {0: "entry", 1: "set-up done (mbarriers, TMEM)", 2: "first W load issued",
                           3: "producer passed the dependency wait", 4: "MMA: first stage full",
                           5: "epilogue: first accumulator ready", 12: "producer: last stage issued",
                           13: "producer: end of work seen", 6: "epilogue: last accumulator ready",
                           7: "last unit published (not reduced here)", 8: "last tile reduction done",
                           14: "cluster epilogue: partials published (cluster barrier passed)",
                           15: "cluster epilogue: share of the tile stored", 9: "exit"},
    "gemv_ar_cluster_kernel": {0: "entry", 1: "dot products done, partial in shared memory",
                               2: "partials published (first cluster barrier passed)",
                               3: "share of the tile summed and stored", 4: "exit"},
    "rmsnorm_rows_kernel": {0: "entry", 1: "gamma / bias loads issued", 2: "dependency wait passed",
                            3: "row loaded, squares summed", 4: "first cluster barrier passed",
                            5: "second cluster barrier passed", 6: "stores issued"},
}
# The slot that marks a CTA's first data (for the chained view).
FIRST_DATA = {"gemv_ar_dyn_kernel": 4, "gemv_ar_ffma_kernel": 1, "gemv_ar_cluster_kernel": 1,
              "rmsnorm_rows_kernel": 3}
COUNTS = {"gemv_ar_ffma_kernel": {8: "tiles reduced"},
          "gemv_ar_dyn_kernel": {10: "units computed", 11: "tile reductions"}}


def _pct(v, q):
    v = sorted(v)
    return v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--workload", default="attn_out_proj")
    p.add_argument("--reps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--w-layout", choices=("packed", "row_major"), default="packed")
    p.add_argument("--chain", type=int, default=0,
                   help="also time this many calls chained back to back (SYMM_OPT_CHAIN 1), one timeline "
                        "buffer each, and report how consecutive launches overlap")
    p.add_argument("--opt", action="append", default=[],
                   help="handle option NAME=VALUE (e.g. SYMM_OPT_GEMV_PATH=1), repeatable")
    args = p.parse_args(argv)

    import numpy as np
    import torch

    import collective_split_gemv_gb300 as csg
    import synth
    from collective_split_gemv_gb300 import _build
    from collective_split_gemv_gb300.workspace import GemvWorkspace, RmsNormWorkspace

    _build.build(variant="timeline")
    synth.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    opts = []
    for o in args.opt:
        name, val = o.split("=")
        opts.append((getattr(csg, name), int(val)))

    def set_opts(h):
        for k, v in opts:
            csg.symm_set_option(h, k, v)

    w = dict(synth.WORKLOADS[args.workload])
    kind, R = w["kind"], w["R"]
    if kind == "gemv":
        N, K, B = w["N"], w["K"], w["B"]
        W, x = synth.gemv_inputs(R, N, K, B, w["seed"], w["w_std"], w["x"])
        copies = max(1, min(8, -(-3 * L2_BYTES // max(W.nbytes, 1))))
        probe = GemvWorkspace(R, N, K, B)
        set_opts(probe.h)
        plan = csg.symm_gemv_plan(probe.h, N, K, B)
        probe.close()
        packed = args.w_layout == "packed" and plan["path"] == csg.GEMV_PATH_DYN
        ws = GemvWorkspace(R, N, K, B, copies=copies, packed=packed)
        set_opts(ws.h)
        for c in range(copies):
            ws.load_W(W, copy=c)
        ws.load_x(x)
        kernel = {csg.GEMV_PATH_FFMA: "gemv_ar_ffma_kernel", csg.GEMV_PATH_DYN: "gemv_ar_dyn_kernel",
                  csg.GEMV_PATH_CLUSTER: "gemv_ar_cluster_kernel"}[plan["path"]]
        ctas = plan["grid"]
        run = lambda i: ws.run(stream, copy=i % copies)
        flush = copies * W.nbytes < 2 * L2_BYTES
        desc = (f"R={R} N={N} K={K} (K/R={K // R}) B={B}; plan {plan}; "
                f"W {'packed' if packed else 'row-major'}, {copies} rotating copies")
    elif kind == "ar_rmsnorm":
        rows, H, eps = w["rows"], w["H"], w["eps"]
        inp, bias, gamma = synth.rmsnorm_inputs(R, rows, H, w["seed"])
        ws = RmsNormWorkspace(R, rows, H)
        set_opts(ws.h)
        ws.load(inp, bias, gamma)
        kernel = "rmsnorm_rows_kernel"
        ctas = 8 * rows
        run = lambda i: ws.run(stream, eps=eps)
        flush = True
        copies = 1
        desc = f"R={R} rows={rows} H={H}"
    else:
        raise SystemExit(f"no timeline for workload kind {kind!r}")

    slots = csg.TIMELINE_SLOTS
    tl = torch.zeros(ctas * slots, dtype=torch.int64, device=dev)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 0)
    csg.symm_set_timeline(ws.h, tl.data_ptr(), tl.numel() * 8)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    phases = PHASES[kernel]
    per_rep = {s: [] for s in phases}          # [rep] -> (min, median, max) over CTAs, µs after first entry
    counts = {s: [] for s in COUNTS.get(kernel, {})}
    event_us, span_us, entry_spread, empty_us = [], [], [], []

    def prelude(i):
        # Keep the GPU busy while the host enqueues the launch, so that the
        # events time the GPU side only: the L2 flush where the inputs fit
        # in L2, else a ~50 us sleep kernel.
        if flush_buf is not None:
            flush_buf.fill_(i & 0xFF)
        else:
            torch.cuda._sleep(100_000)

    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.reps):
            # the floor: an empty kernel between the same events
            prelude(i)
            ev0.record(stream)
            torch.cuda._sleep(0)
            ev1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                empty_us.append(ev0.elapsed_time(ev1) * 1e3)
            tl.zero_()
            prelude(i)
            ev0.record(stream)
            run(i)
            ev1.record(stream)
            stream.synchronize()
            if i < args.warmup:
                continue
            event_us.append(ev0.elapsed_time(ev1) * 1e3)
            t = tl.view(ctas, slots).cpu().numpy().astype(np.int64)
            entry = t[:, 0][t[:, 0] > 0]
            t0 = int(entry.min())
            last = int(t[t > 10**12].max()) if np.any(t > 10**12) else t0
            span_us.append((last - t0) / 1e3)
            entry_spread.append((int(entry.max()) - t0) / 1e3)
            for s in phases:
                col = t[:, s]
                col = col[col > 10**12]      # stamps, not unset slots
                if col.size:
                    d = (col - t0) / 1e3
                    per_rep[s].append((float(d.min()), float(np.median(d)), float(d.max()), int(col.size)))
            for s in counts:
                col = t[:, s]
                counts[s].append((int(col.min()), float(np.mean(col)), int(col.max()), int(col.sum())))
    chain_rows = []
    if args.chain > 1:
        # Calls chained back to back (each a programmatic dependent of the
        # one before), one buffer per call; the stamps share one clock.
        bufs = [torch.zeros(ctas * slots, dtype=torch.int64, device=dev) for _ in range(args.chain)]
        first_data = FIRST_DATA.get(kernel, 1)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        with torch.cuda.stream(stream):
            for rep_i in range(3):
                for b in bufs:
                    b.zero_()
                prelude(rep_i)
                for k, b in enumerate(bufs):
                    csg.symm_set_timeline(ws.h, b.data_ptr(), b.numel() * 8)
                    run(k)
                stream.synchronize()
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 0)
        ts = [b.view(ctas, slots).cpu().numpy().astype(np.int64) for b in bufs]
        t0 = int(ts[0][:, 0][ts[0][:, 0] > 0].min())
        for k, t in enumerate(ts):
            entry = t[:, 0][t[:, 0] > 0]
            data = t[:, first_data][t[:, first_data] > 10**12]
            last = int(t[t > 10**12].max())
            chain_rows.append(((int(entry.min()) - t0) / 1e3, (float(np.median(data)) - t0) / 1e3 if data.size else
                               float("nan"), (int(entry.max()) - t0) / 1e3, (last - t0) / 1e3))
    code, _, _ = csg.symm_status(ws.h, stream)
    if code != csg.SYMM_OK:
        raise SystemExit(f"protocol error: {csg.symm_last_error()}")
    csg.symm_set_timeline(ws.h, None, 0)
    ws.close()

    med = statistics.median
    print(f"# {kernel} timeline — {args.workload}\n")
    print(f"{desc}; options {args.opt or 'none'}; {args.reps} launches in plain stream order"
          + ("; L2 flushed before each" if flush else "; a sleep kernel before each, so the host enqueues ahead")
          + "\n")
    print(f"- CUDA-event time of the launch: median {med(event_us):.2f} µs "
          f"(p10 {_pct(event_us, 0.1):.2f}, p90 {_pct(event_us, 0.9):.2f})")
    print(f"- CUDA-event time of an empty kernel (torch.cuda._sleep(0)) launched the same way: median "
          f"{med(empty_us):.2f} µs")
    print(f"- first CTA entry to last stamp: median {med(span_us):.2f} µs; "
          f"event time minus that span (launch and teardown outside the CTAs): "
          f"{med(event_us) - med(span_us):.2f} µs")
    print(f"- spread of CTA entries (last entry after the first): median {med(entry_spread):.2f} µs\n")
    print("| phase | CTAs | min µs | median µs | max µs |")
    print("|---|---|---|---|---|")
    for s, name in phases.items():
        v = per_rep[s]
        if not v:
            continue
        print(f"| {name} | {v[0][3]} | {med(a for a, _, _, _ in v):.2f} | {med(b for _, b, _, _ in v):.2f} | "
              f"{med(c for _, _, c, _ in v):.2f} |")
    for s, name in COUNTS.get(kernel, {}).items():
        v = counts[s]
        if v:
            print(f"\n- {name} per CTA: min {v[-1][0]}, mean {v[-1][1]:.2f}, max {v[-1][2]}, total {v[-1][3]}")
    print("\n(times: after the first CTA's entry, median over the launches of each CTA statistic)")
    if chain_rows:
        print(f"\n## {len(chain_rows)} calls chained back to back (the last of 3 repetitions)\n")
        print("Times after the first call's first CTA entry, µs; 'first data' is the median CTA's "
              f"'{phases.get(FIRST_DATA.get(kernel, 1), 'phase 1')}'.\n")
        print("| call | first CTA entry | first data (median CTA) | last CTA entry | last stamp | "
              "entry after the previous call's last stamp |")
        print("|---|---|---|---|---|---|")
        for k, (e0, fd, e1, end) in enumerate(chain_rows):
            gap = "" if k == 0 else f"{e0 - chain_rows[k - 1][3]:.2f}"
            print(f"| {k} | {e0:.2f} | {fd:.2f} | {e1:.2f} | {end:.2f} | {gap} |")
        per_call = (chain_rows[-1][3] - chain_rows[0][3]) / (len(chain_rows) - 1)
        print(f"\nLast stamp to last stamp: {per_call:.2f} µs per call.")


if __name__ == "__main__":
    main()
