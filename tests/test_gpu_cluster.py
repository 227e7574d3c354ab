"""The cluster kernel for small layers (path 5): one thread-block cluster of
R CTAs per 16-row tile, the ranks' partials exchanged through distributed
shared memory.  Against the oracle: small-integer inputs bit-exact, normal
inputs within the parity tolerance, every rank count 1..8 and batch width
1..4 on ragged shapes; bitwise the CUDA-core per-tile kernel's results
(the same per-rank sums in the same order); every output form; chained and
captured calls; the limits it rejects."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu, run_gemv
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu

CLUSTER = csg.GEMV_PATH_CLUSTER


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ints(R, N, Kr, B, seed):
    rng = np.random.default_rng(seed)
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    return W, x


CASES = [(R, N, Kr, B) for R in (1, 2, 3, 5, 8) for N, Kr, B in ((1, 8, 1), (17, 24, 4), (256, 256, 1), (100, 1032, 3),
                                                                  (33, 4096, 2))]


@pytest.mark.parametrize("case", CASES, ids=[f"R{a}N{b}Kr{c}B{d}" for a, b, c, d in CASES])
def test_cluster_kernel_against_the_oracle(case):
    R, N, Kr, B = case
    W, x = _ints(R, N, Kr, B, seed=sum(case))
    (y,), status = run_gemv(W, x, path=CLUSTER)
    assert status[0] == csg.SYMM_OK
    check_gemv(W, x, y, exact=True)
    Wn, xn = synth.gemv_inputs(R, N, R * Kr, B, seed=N + Kr, w_std=0.02, x="normal")
    outs, status = run_gemv(Wn, xn, path=CLUSTER, repeat=2)
    assert status[0] == csg.SYMM_OK
    assert np.array_equal(outs[0], outs[1]), "a second run changed bits"
    check_gemv(Wn, xn, outs[0])
    # the CUDA-core per-tile kernel sums each rank's products and the ranks
    # in the same order (one pass over K/R here): the same bits
    ref, _ = run_gemv(Wn, xn, path=csg.GEMV_PATH_FFMA)
    assert np.array_equal(outs[0], ref[0])


def test_tiny_layer_is_planned_on_the_cluster_kernel():
    w = synth.WORKLOADS["tiny"]
    ws = GemvWorkspace(w["R"], w["N"], w["K"], w["B"])
    try:
        plan = csg.symm_gemv_plan(ws.h, w["N"], w["K"], w["B"])
        assert plan["path"] == CLUSTER and plan["grid"] == w["R"] * (w["N"] // 16)
    finally:
        ws.close()
    W, x = synth.gemv_inputs(w["R"], w["N"], w["K"], w["B"], w["seed"], w["w_std"], w["x"])
    (y,), status = run_gemv(W, x)
    assert status[0] == csg.SYMM_OK
    ratio, eq, ulp = check_gemv(W, x, y)
    assert ulp <= 1


@pytest.mark.parametrize("form", ["reduce_scatter", "bias_rmsnorm"])
def test_cluster_kernel_other_forms(form):
    R, N, K, B = 4, 264, 4 * 136, 4
    W, x = synth.gemv_inputs(R, N, K, B, seed=3, w_std=0.05, x="normal")
    bias, gamma = synth.norm_vectors(N, 3)
    outs = {}
    for path in (CLUSTER, csg.GEMV_PATH_FFMA):
        ws = GemvWorkspace(R, N, K, B)
        try:
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
            ws.load_W(W)
            ws.load_x(x)
            ws.load_vectors(bias, gamma)
            ws.fill_y(0xFF)
            ws.run(torch.cuda.current_stream(), mode=form, eps=1e-6)
            assert csg.symm_status(ws.h, None)[0] == csg.SYMM_OK
            outs[path] = ws.read_y_rs() if form == "reduce_scatter" else ws.read_y()
            assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        finally:
            ws.close()
    assert np.array_equal(outs[CLUSTER], outs[csg.GEMV_PATH_FFMA])
    if form == "reduce_scatter":
        y_ref, _ = oracle.gemv_reduce_scatter(W, x)
        got = outs[CLUSTER]
        for s in range(R):
            rows = slice(s * (B // R), (s + 1) * (B // R))
            assert tolerance_ratio(words_to_f64(got[s]), y_ref[rows]) <= 1.0
    else:
        y_ref, want = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6)
        got = outs[CLUSTER]
        assert tolerance_ratio(words_to_f64(got[0]), y_ref) <= 1.0
        rms = float(np.sqrt(np.mean(y_ref * y_ref)))
        big = np.abs(y_ref) >= 0.1 * rms
        assert int(ulp_distance(got[0][big], want[0][big]).max(initial=0)) <= 1


def _chain_and_capture(chain):
    """Chained calls, each reading the previous call's y as its x, then the
    same call captured into a CUDA graph and replayed: the eager call's bits."""
    R, N, K, B = 2, 512, 2 * 256, 1
    W, x = synth.gemv_inputs(R, N, K, B, seed=11, w_std=0.06, x="normal")
    ws = GemvWorkspace(R, 2 * N, K, B)   # y (B x 2N per slot) is wide enough to hold x (B x K/R)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, CLUSTER)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        Wfull = np.zeros((R, 2 * N, K // R), dtype=np.uint16)
        Wfull[:, :N] = W
        ws.load_W(Wfull)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for _ in range(6):
            ws.run(s)
            for r in range(R):   # y's first K/R elements of each rank become its next x
                ws.x_view(r).copy_(ws.y_view(r)[: ws.x_bytes])
        got = ws.read_y()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ws.run(torch.cuda.current_stream())
        ws.fill_y(0xFF)
        g.replay()
        replayed = ws.read_y()
        ws.fill_y(0xFF)
        ws.run(s)
        eager = ws.read_y()
        assert np.array_equal(replayed, eager)
        del g
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        return got
    finally:
        ws.close()


def test_cluster_chain_and_capture_match_plain_order():
    assert np.array_equal(_chain_and_capture(1), _chain_and_capture(0))


def test_cluster_kernel_limits():
    for R, B in ((9, 1), (2, 5)):
        ws = GemvWorkspace(R, 64, R * 64, B)
        try:
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, CLUSTER)
            with pytest.raises(csg.SymmError) as e:
                ws.run(torch.cuda.current_stream())
            assert e.value.code == csg.SYMM_EINVAL
            with pytest.raises(csg.SymmError):
                csg.symm_gemv_plan(ws.h, 64, R * 64, B)
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_AUTO)
            assert csg.symm_gemv_plan(ws.h, 64, R * 64, B)["path"] != CLUSTER
        finally:
            ws.close()
