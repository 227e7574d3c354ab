"""Host-side logic of bench.py, on the CPU: byte accounting against the
hand-computed per-call figures of the five workloads, argument defaults, and
the max-over-ranks aggregation of the multi-GPU replicas with two gloo ranks."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_match_hand_computed_values():
    # W + x + partials written and read back + R replicated outputs
    assert bench.algorithmic_bytes(2, 256, 512, 1) == 262_144 + 1_024 + 4_096 + 1_024
    assert bench.algorithmic_bytes(4, 8192, 8192, 8) == 136_970_240
    assert bench.algorithmic_bytes(8, 8192, 28672, 1) == 470_474_752
    assert bench.algorithmic_bytes(8, 16384, 53248, 16) == 1_767_505_920
    assert bench.allreduce_bytes(8, 4_194_304) == 134_217_728
    for name in ("tiny", "allreduce", "attn_out_proj", "mlp_down_decode", "mlp_down_large"):
        assert bench.workload_bytes(bench.workload(name)) > 0


def test_throughput_is_whole_job():
    assert bench.throughput_gbs(1e9, 1.0) == pytest.approx(1000.0)
    assert bench.throughput_gbs(1e9, 1.0, world=4) == pytest.approx(4000.0)


def test_default_arguments_time_the_decode_workload():
    a = bench.parse_args([])
    assert a.workload == "mlp_down_decode" and a.impl == "ours" and a.gpus == 1 and a.warmup >= 3
    assert bench.parse_args(["--warmup", "1"]).warmup == 3


def test_single_rank_aggregation_is_identity():
    assert bench.max_over_ranks([1.5, 2.0], 1) == [1.5, 2.0]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], world)
        queue.put((rank, vals))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0, 3.0]


def test_traffic_entries_name_known_kernels_and_workloads():
    """Every profiled traffic entry names a kernel the bench reports and a
    workload it runs, with positive bytes and a 16-hex-digit source hash."""
    import json
    import re
    import synth
    d = json.load(open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                                    "traffic.json")))
    for kernel, per in d.items():
        if kernel.startswith("_"):
            continue
        for part in kernel.split("+"):
            assert part.split("<")[0] in bench.KERNEL_SOURCES, kernel
        for workload, entry in per.items():
            assert workload in synth.WORKLOADS, (kernel, workload)
            assert entry["dram_bytes_per_launch"] > 0
            assert re.fullmatch(r"[0-9a-f]{16}", entry["source_sha"])
            # a stale entry is reported as null, a current one as its bytes
            got = bench.profiled_traffic(kernel, workload, entry["source_sha"])
            assert got == entry["dram_bytes_per_launch"]
            assert bench.profiled_traffic(kernel, workload, "0" * 16) is None


@pytest.mark.parametrize("workload,threads", [("tiny", None), ("ar_bias_rmsnorm", 1)])
def test_reference_arm_line_follows_the_contract(workload, threads):
    """`bench.py --impl reference` (the oracle on the host cores): the keys of
    the JSON line, a zero-copy e2e object, no GPU launches, and `cores` as the
    threads the oracle function used (the RMSNorm oracle is single-threaded)."""
    args = bench.parse_args(["--impl", "reference", "--workload", workload, "--steps", "2", "--warmup", "1"])
    line = bench.run_reference(args, 0, 1)
    for key in ("metric", "impl", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["gpu_launches"] == 0
    assert line["config"]["workload"] == workload and line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["sample"]
    assert cb["cores"] == (threads if threads is not None else bench.host_cores())
    assert bench.run_reference(args, 1, 2) is None   # other ranks print nothing


@pytest.mark.parametrize("workload", ["tiny", "allreduce"])
def test_parity_object_of_the_oracle_leg(workload):
    """The bench's parity check: the oracle's own words pass (their ratio is
    their rounding, at most half a bf16 ulp, so below 1) with every output
    bit-equal; a large change in one output (every replica) fails the
    tolerance; one replica that differs is reported."""
    import numpy as np

    import oracle
    import synth

    w = bench.workload(workload)
    if workload == "tiny":
        W, x = synth.gemv_inputs(w["R"], w["N"], w["K"], w["B"], w["seed"], w["w_std"], w["x"])
        y_ref, words = oracle.gemv_all_reduce(W, x)
        at = (slice(None), *np.unravel_index(np.argmax(np.abs(y_ref)), y_ref.shape))
        first = (1, 0, 0)
    else:
        inp = synth.allreduce_inputs(w["R"], w["n"], w["seed"])
        y_ref, words = oracle.one_shot_all_reduce(inp)
        at = (slice(None), int(np.argmax(np.abs(y_ref))))
        first = (1, 0)
    p = bench.cpu_baseline(workload, budget_s=0.5, gpu_out=words)["parity"]
    assert p["passed"] and p["max_tol_ratio"] <= 1.0 and p["bit_equal_frac"] == 1.0 and p["replicas_identical"]
    assert p["max_ulp"] == 0 and p["max_ulp_where_abs_ge_0.1_rms"] == 0
    bad = words.copy()
    bad[at] ^= 0x0040                       # the largest output changed by a quarter or more
    p = bench.cpu_baseline(workload, budget_s=0.5, gpu_out=bad)["parity"]
    assert not p["passed"] and p["max_tol_ratio"] > 1 and p["max_ulp"] == 0x40
    odd = words.copy()
    odd[first] ^= 1                         # one ulp in one replica
    p = bench.cpu_baseline(workload, budget_s=0.5, gpu_out=odd)["parity"]
    assert p["replicas_identical"] is False and not p["passed"]


def test_parity_check_of_every_form():
    """parity_check on small oracle results of each form: the oracle's own
    words pass; the largest output changed by a quarter or more (alike in
    every replica) fails; the forms whose row sample is no sample of the
    call (a normalisation over the whole row on a partial sample, a
    reduce-scatter's blocks on a prefix) are skipped."""
    import numpy as np

    import oracle
    import synth

    R, N, Kr, B = 4, 64, 32, 8
    W, x = synth.gemv_inputs(R, N, R * Kr, B, seed=5, w_std=0.05, x="normal")
    bias, gamma = synth.norm_vectors(N, 5)
    inp = synth.allreduce_inputs(R, 256, 6)
    rin, rbias, rgamma = synth.rmsnorm_inputs(R, 3, 64, 7)
    # (kind, op, oracle result, rows = full, does every slot hold a replica)
    cases = [
        ("gemv", "one_shot", oracle.gemv_all_reduce(W, x), N, True),
        ("gemv_rs", "one_shot", oracle.gemv_reduce_scatter(W, x), N, False),
        ("gemv_rmsnorm", "one_shot", oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6), N, True),
        ("allreduce", "reduce_scatter", oracle.reduce_scatter(inp), 256, False),
        ("ar_rmsnorm", "one_shot", oracle.all_reduce_bias_rmsnorm(rin, rbias, rgamma, 1e-6), 3, True),
    ]
    for kind, op, ref, rows, replicated in cases:
        y_ref, words = ref
        p = bench.parity_check(kind, op, ref, np.asarray(words), rows, rows, R, "rows")
        assert p is not None and p["passed"] and p["max_ulp"] == 0, (kind, p)
        at = int(np.argmax(np.abs(np.asarray(y_ref)).reshape(-1)))
        bad = np.array(words, copy=True)
        if replicated:          # the same output of every replica
            per = bad.reshape(R, -1)
            per[:, at] ^= 0x0040
        else:                   # the slots' blocks, in order, are the whole result
            bad.reshape(-1)[at] ^= 0x0040
        p = bench.parity_check(kind, op, ref, bad, rows, rows, R, "rows")
        assert not p["passed"] and p["max_tol_ratio"] > 1, (kind, p)
    # a row sample that is no sample of the form
    assert bench.parity_check("gemv_rmsnorm", "one_shot", cases[2][2], cases[2][2][1], N // 2, N, R, "rows") is None
    assert bench.parity_check("allreduce", "reduce_scatter", cases[3][2], cases[3][2][1], 128, 256, R, "rows") \
        is None
    assert bench.parity_check("tile", "one_shot", cases[0][2], cases[0][2][1], N, N, R, "rows") is None


def test_workload_of_any_gemv_shape():
    """--workload gemv:R,N,K,B names the fused GEMV of that shape; shapes
    the call refuses, malformed names and unknown names are refused."""
    w = bench.workload("gemv:8,8192,28672,4")
    assert (w["kind"], w["R"], w["N"], w["K"], w["B"]) == ("gemv", 8, 8192, 28672, 4)
    assert bench.workload_bytes(w) == bench.algorithmic_bytes(8, 8192, 28672, 4)
    # K not a multiple of R, B above 16, not integers, too few numbers, unknown, K/R not a multiple of 8
    for bad in ("gemv:8,8192,28671,4", "gemv:8,8192,28672,17", "gemv:8,8192,8*4,1", "gemv:8,8192", "nonesuch",
                "gemv:8,8192,96,1"):
        with pytest.raises(SystemExit):
            bench.workload(bad)
