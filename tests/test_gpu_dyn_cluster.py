"""The persistent kernel's cluster epilogue (SYMM_OPT_DYN_CLUSTER): one
(row tile, rank) unit per CTA, the R units of a tile one thread-block cluster,
the partials summed through distributed shared memory instead of the
global-memory protocol.  It adds in the same rank order as the global-memory
reducer, so it must give that path's bits on every shape, batch, weight layout
and output form, the oracle's words on small-integer inputs, and leave the
signal pad's protocol state usable by the calls that follow it."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu
from helpers import f64_to_words_via_f32, tolerance_ratio, words_to_f64

pytestmark = pytest.mark.gpu

ON, OFF, AUTO = 1, 0, -1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ws(W, x, cluster, packed=False, slabs=0, chain=1, splits=0):
    R, N, Kr = W.shape
    ws = GemvWorkspace(R, N, R * Kr, x.shape[1], packed=packed)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, cluster)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_SLABS, slabs)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
    csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, splits)
    ws.load_W(W)   # (packed: packs on the current stream)
    ws.load_x(x)
    return ws


def _run(W, x, cluster, mode="all_reduce", bias=None, gamma=None, eps=1e-6, repeat=2, **kw):
    """`repeat` calls; returns the outputs of each (all slots) and the plan."""
    ws = _ws(W, x, cluster, **kw)
    try:
        R, N, Kr = W.shape
        plan = csg.symm_gemv_plan(ws.h, N, R * Kr, x.shape[1])
        ws.load_vectors(bias, gamma)
        s = torch.cuda.current_stream()
        outs = []
        for _ in range(repeat):
            ws.fill_y(0xFF)
            ws.run(s, mode=mode, eps=eps, bias=bias is not None, gamma=gamma is not None)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            outs.append(ws.read_y_rs() if mode == "reduce_scatter" else ws.read_y())
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        return outs, plan
    finally:
        ws.close()


# (R, N, K, B): ragged last tiles, N % 4 != 0 (scalar sums), one-tile layers,
# every batch width class, 8 ranks (the largest portable cluster)
SHAPES = [(4, 1024, 4 * 1024, 8), (2, 300, 2 * 512, 1), (3, 257, 3 * 136, 3), (8, 130, 8 * 264, 16),
          (4, 128, 4 * 64, 2), (8, 1000, 8 * 512, 5), (2, 2 * 128 + 4, 2 * 1040, 16)]


@pytest.mark.parametrize("packed", [False, True], ids=["rowmajor", "packed"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"R{a}N{b}K{c}B{d}" for a, b, c, d in SHAPES])
def test_cluster_epilogue_gives_the_protocol_bits(packed, shape):
    R, N, K, B = shape
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + B, w_std=0.02, x="normal")
    ref, p_off = _run(W, x, OFF, packed=packed, splits=1)
    got, p_on = _run(W, x, ON, packed=packed)
    assert p_on["cluster"] == R and p_on["splits"] == 1 and p_on["grid"] == p_on["tiles"] * R
    assert p_off["cluster"] == 0
    for y in ref + got:
        assert np.array_equal(y, ref[0])
    check_gemv(W, x, got[0])


# (R, N, K, B, splits) with R x splits <= 8: a cluster holds every rank's K splits of a tile
SPLIT_SHAPES = [(2, 300, 2 * 1024, 3, 4), (4, 1024, 4 * 1024, 8, 2), (2, 257, 2 * 520, 16, 3), (3, 128, 3 * 384, 1, 2)]


@pytest.mark.parametrize("packed", [False, True], ids=["rowmajor", "packed"])
@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[f"R{a}N{b}K{c}B{d}S{e}" for a, b, c, d, e in SPLIT_SHAPES])
def test_cluster_epilogue_with_k_splits_gives_the_protocol_bits(packed, shape):
    R, N, K, B, S = shape
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + S, w_std=0.02, x="normal")
    ref, p_off = _run(W, x, OFF, packed=packed, splits=S)
    got, p_on = _run(W, x, ON, packed=packed, splits=S)
    assert p_off["splits"] == S and p_on["splits"] == S and p_on["cluster"] == R * S
    assert p_on["grid"] == p_on["tiles"] * R * S
    for y in ref + got:
        assert np.array_equal(y, ref[0])
    check_gemv(W, x, got[0])


def test_cluster_epilogue_with_k_splits_integers_bit_exact():
    rng = np.random.default_rng(21)
    R, N, Kr, B = 4, 300, 512, 5
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    (y, y2), plan = _run(W, x, ON, splits=2)
    assert plan["cluster"] == 8
    check_gemv(W, x, y, exact=True)
    assert np.array_equal(y, y2)


@pytest.mark.parametrize("slabs", [1, 2, 3])
@pytest.mark.parametrize("chain", [0, 1])
def test_cluster_epilogue_small_integers_bit_exact(slabs, chain):
    rng = np.random.default_rng(11 + slabs)
    R, N, Kr, B = 4, 300, 264, 7
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    (y, y2), _ = _run(W, x, ON, slabs=slabs, chain=chain)
    check_gemv(W, x, y, exact=True)
    assert np.array_equal(y, y2)


@pytest.mark.parametrize("R,N,Kr,B", [(2, 300, 64, 2), (4, 129, 128, 8), (8, 1000, 256, 16)])
def test_cluster_epilogue_reduce_scatter(R, N, Kr, B):
    rng = np.random.default_rng(R * N)
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    _, want = oracle.gemv_reduce_scatter(W, x)
    (out, _), plan = _run(W, x, ON, mode="reduce_scatter")
    assert plan["cluster"] == R
    assert np.array_equal(out, want)


@pytest.mark.parametrize("R,N,K,B", [(2, 256, 512, 1), (4, 1000, 2048, 3), (8, 1024, 8 * 256, 2)])
def test_cluster_epilogue_bias_rmsnorm(R, N, K, B):
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + B, w_std=0.05)
    bias, gamma = synth.norm_vectors(N, seed=N)
    ref, _ = _run(W, x, OFF, mode="bias_rmsnorm", bias=bias, gamma=gamma, eps=1e-5, repeat=1, splits=1)
    got, plan = _run(W, x, ON, mode="bias_rmsnorm", bias=bias, gamma=gamma, eps=1e-5, repeat=1)
    assert plan["cluster"] == R
    assert np.array_equal(got[0], ref[0])
    y_ref, _ = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-5)
    assert tolerance_ratio(words_to_f64(got[0][0]), y_ref) <= 1.0


def test_cluster_epilogue_automatic_choice():
    """attn_out_proj (64 tiles x 4 ranks = 256 units) fits the persistent
    grid in one wave and takes the cluster epilogue, and so do layers of any
    unit count whose units are long (K/R >= 3072: the decode, the large
    layer); layers of many short units, one CTA per SM, K splits, the
    unfused form and a single rank keep the global-memory protocol."""
    ws = GemvWorkspace(4, 4 * 8192, 4 * 64, 8)    # scratch and pad for up to 256 row tiles at B = 8
    try:
        h = ws.h
        csg.symm_set_option(h, csg.SYMM_OPT_DYN_CLUSTER, OFF)
        if csg.symm_gemv_plan(h, 8192, 8192, 8)["grid"] < 256:
            pytest.skip("fewer than 256 CTA slots on this GPU")
        csg.symm_set_option(h, csg.SYMM_OPT_DYN_CLUSTER, AUTO)
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["cluster"] == 4
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["grid"] == 256
        assert csg.symm_gemv_plan(h, 4 * 8192, 8192, 8)["cluster"] == 0     # 1024 units of K/R = 2048
        long_units = csg.symm_gemv_plan(h, 4 * 8192, 4 * 3072, 8)            # 1024 units of K/R = 3072
        assert long_units["cluster"] == 4 and long_units["grid"] == 1024
        csg.symm_set_option(h, csg.SYMM_OPT_SK_CTAS_PER_SM, 1)
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["cluster"] == 0
        csg.symm_set_option(h, csg.SYMM_OPT_SK_CTAS_PER_SM, 0)
        csg.symm_set_option(h, csg.SYMM_OPT_DYN_SPLITS, 2)
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["cluster"] == 0
        csg.symm_set_option(h, csg.SYMM_OPT_DYN_SPLITS, 0)
        csg.symm_set_option(h, csg.SYMM_OPT_UNFUSED, 1)
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["cluster"] == 0
        csg.symm_set_option(h, csg.SYMM_OPT_UNFUSED, 0)
        csg.symm_set_option(h, csg.SYMM_OPT_DYN_CLUSTER, OFF)
        assert csg.symm_gemv_plan(h, 8192, 8192, 8)["cluster"] == 0
    finally:
        ws.close()


def test_cluster_epilogue_rejections():
    W, x = synth.gemv_inputs(2, 256, 2 * 256, 2, seed=1, w_std=0.02, x="normal")
    ws = _ws(W, x, ON)
    try:
        s = torch.cuda.current_stream()
        for opt, val in ((csg.SYMM_OPT_SK_CTAS_PER_SM, 1), (csg.SYMM_OPT_UNFUSED, 1)):
            csg.symm_set_option(ws.h, opt, val)
            with pytest.raises(csg.SymmError) as e:
                ws.run(s)
            assert e.value.code == csg.SYMM_EINVAL
            csg.symm_set_option(ws.h, opt, 0)
        ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        for bad in (-2, 2):
            with pytest.raises(csg.SymmError) as e:
                csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, bad)
            assert e.value.code == csg.SYMM_EINVAL
    finally:
        ws.close()
    # R x splits above a portable cluster
    W, x = synth.gemv_inputs(4, 256, 4 * 768, 2, seed=2, w_std=0.02, x="normal")
    ws = _ws(W, x, ON, splits=3)
    try:
        with pytest.raises(csg.SymmError) as e:
            ws.run(torch.cuda.current_stream())
        assert e.value.code == csg.SYMM_EINVAL
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, 2)
        assert csg.symm_gemv_plan(ws.h, 256, 4 * 768, 2)["cluster"] == 8
    finally:
        ws.close()
    ws = GemvWorkspace(9, 64, 9 * 64, 1)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, ON)
        with pytest.raises(csg.SymmError) as e:     # more ranks than a portable cluster holds
            csg.symm_gemv_plan(ws.h, 64, 9 * 64, 1)
        assert e.value.code == csg.SYMM_EINVAL
    finally:
        ws.close()


def test_cluster_and_drawn_launches_alternate_on_one_handle():
    """The cluster epilogue touches neither the launch epoch nor the work
    counters: cluster, drawn and K-split launches alternate, chained, with no
    reset in between, and every one is right."""
    R, N, K, B = 4, 1024, 4 * 1024, 4
    W, x = synth.gemv_inputs(R, N, K, B, seed=3, w_std=0.02, x="normal")
    ws = _ws(W, x, ON)
    try:
        s = torch.cuda.current_stream()
        ref = None
        for i in range(12):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, (ON, OFF, OFF)[i % 3])
            csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, (0, 1, 3)[i % 3])
            ws.fill_y(0xFF)
            ws.run(s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            y = ws.read_y()
            if i % 3 != 2:                            # K splits add in another order
                if ref is None:
                    ref = y
                assert np.array_equal(y, ref)
            check_gemv(W, x, y)
    finally:
        ws.close()


def test_cluster_epilogue_beyond_one_wave():
    """Forced on a layer with more units than CTA slots (8 x 128 tiles =
    1024 units), the clusters run in several waves: still the protocol's bits."""
    R, N, K, B = 8, 128 * 128, 8 * 128, 2
    W, x = synth.gemv_inputs(R, N, K, B, seed=7, w_std=0.02, x="normal")
    ref, _ = _run(W, x, OFF, repeat=1, splits=1)
    got, plan = _run(W, x, ON, repeat=1)
    assert plan["grid"] == 1024 and plan["cluster"] == 8
    assert np.array_equal(got[0], ref[0])
    check_gemv(W, x, got[0])


def test_cluster_epilogue_graph_replay():
    """A captured cluster-epilogue call replays to the eager call's bits."""
    R, N, K, B = 4, 1024, 4 * 2048, 8
    W, x = synth.gemv_inputs(R, N, K, B, seed=5, w_std=0.02, x="normal")
    ws = _ws(W, x, ON, packed=True)
    try:
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            ws.run(s)
        s.synchronize()
        eager = ws.read_y()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ws.run(s)
        for _ in range(3):
            ws.fill_y(0xFF)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(ws.read_y(), eager)
        assert csg.symm_status(ws.h, torch.cuda.current_stream())[0] == csg.SYMM_OK
        check_gemv(W, x, eager)
    finally:
        ws.close()


def test_cluster_epilogue_attn_out_proj_full_size():
    """The workload the epilogue is chosen for, at full size, automatic plan,
    packed weights: sampled against the oracle, replicas identical, and the
    same bits as the global-memory protocol."""
    W, x = synth.workload_inputs("attn_out_proj")
    got, plan = _run(W, x, AUTO, packed=True, repeat=1)
    if plan["cluster"] == 0:
        pytest.skip("the automatic plan did not take the cluster epilogue on this GPU")
    ref, _ = _run(W, x, OFF, packed=True, repeat=1, splits=1)
    assert np.array_equal(got[0], ref[0])
    check_gemv(W, x, got[0])


def test_long_chain_of_cluster_launches():
    """Hundreds of chained cluster-epilogue calls (each a programmatic
    dependent of the one before, every CTA a cluster member), alternating two
    activations: the last result is the oracle's for the last inputs and the
    status stays clean."""
    R, N, K, B = 8, 2048, 8 * 3072, 1          # long units: the automatic plan takes clusters
    W, x0 = synth.gemv_inputs(R, N, K, B, seed=31, w_std=0.02, x="normal")
    _, x1 = synth.gemv_inputs(R, N, K, B, seed=32, w_std=0.02, x="normal")
    ws = GemvWorkspace(R, N, K, B, copies=1, packed=True)
    try:
        plan = csg.symm_gemv_plan(ws.h, N, K, B)
        assert plan["path"] == csg.GEMV_PATH_DYN and plan["cluster"] == R
        ws.load_W(W)
        s = torch.cuda.current_stream()
        for i in range(400):
            if i % 100 == 0:
                ws.load_x(x0 if (i // 100) % 2 == 0 else x1)   # stream-ordered rewrite of x between runs of calls
            ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x1, ws.read_y())
    finally:
        ws.close()


def test_twenty_thousand_chained_calls_across_endings():
    """20,000 chained calls on one handle, switching every 500 calls between
    drawn units (the launch epoch, flags, tickets and work counters advance
    every launch), the cluster epilogue, K splits and the unfused form: the
    protocol state the pad carries stays consistent (clean status) and the
    last result is the oracle's."""
    R, N, K, B = 8, 2048, 8 * 512, 2
    W, x = synth.gemv_inputs(R, N, K, B, seed=44, w_std=0.02, x="normal")
    ws = GemvWorkspace(R, N, K, B, packed=True)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        modes = [(OFF, 0, 0), (ON, 0, 0), (OFF, 2, 0), (OFF, 0, 1)]   # (cluster, splits, unfused)
        for i in range(20000):
            if i % 500 == 0:
                cl, sp, uf = modes[(i // 500) % len(modes)]
                csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, cl)
                csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, sp)
                csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, uf)
            ws.run(s)
            if i % 5000 == 4999:
                assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK, i
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


@pytest.mark.parametrize("shape,want", [
    # (R, N, K, B): (path, CTAs per cluster, K splits) of the automatic plan
    ((2, 256, 512, 1), (csg.GEMV_PATH_CLUSTER, 2, 1)),            # the tiny layer: cluster kernel
    ((8, 1024, 8 * 512, 1), (csg.GEMV_PATH_CLUSTER, 8, 1)),       # 512 CTAs x B = 1: still the cluster kernel
    ((8, 4096, 2048, 4), (csg.GEMV_PATH_DYN, 8, 1)),              # small W, 8192 CTAs x B: persistent kernel
    ((16, 256, 16 * 256, 1), (csg.GEMV_PATH_FFMA, 0, 1)),         # R > 8, 256 CTAs: per-tile kernel
    ((16, 1024, 16 * 512, 1), (csg.GEMV_PATH_DYN, 0, 1)),         # R > 8, 1024 CTAs: persistent, drawn units
    ((2, 8192, 28672, 1), (csg.GEMV_PATH_DYN, 4, 2)),             # half-empty wave: K split inside clusters
    ((1, 8192, 28672, 1), (csg.GEMV_PATH_DYN, 4, 4)),             # one rank: the splits are the cluster
    ((4, 8192, 8192, 8), (csg.GEMV_PATH_DYN, 4, 1)),              # attn_out_proj: one wave, no split
    ((8, 8192, 28672, 1), (csg.GEMV_PATH_DYN, 8, 1)),             # the decode layer
], ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) and len(v) == 4 else None)
def test_automatic_plans(shape, want):
    """The automatic plan of representative layers on a GPU of 152 SMs (two
    persistent CTAs per SM): which kernel, the cluster size and the K splits
    that measured fastest."""
    if torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count != 152:
        pytest.skip("the plans were measured on 152 SMs")
    R, N, K, B = shape
    ws = GemvWorkspace(R, N, K, B)
    try:
        plan = csg.symm_gemv_plan(ws.h, N, K, B)
        assert (plan["path"], plan["cluster"], plan["splits"]) == want, plan
    finally:
        ws.close()
