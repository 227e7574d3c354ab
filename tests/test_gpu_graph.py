"""Fused calls captured into a CUDA graph and replayed.

The launch epoch, the tile tickets, the tiles-done count and the persistent
kernel's work counters live in the signal pad and are advanced by the kernels
(every counter is back at zero when a launch ends), so a captured call can be
replayed any number of times, and eager calls of other geometries may run on
the same handle between replays.  Checked on the GPU, through the C ABI, for
every kernel path: the pad's state after each launch, replays against eager
calls bit for bit and against the oracle, a captured decode-like chain, and the
stateless collectives captured with their programmatic dependents."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import synth
from collective_split_gemv_gb300 import DeviceView
from collective_split_gemv_gb300.workspace import AllReduceWorkspace, GemvWorkspace, RmsNormWorkspace
from gpu_common import check_gemv, require_gpu

pytestmark = pytest.mark.gpu

PATHS = {"ffma": csg.GEMV_PATH_FFMA, "dyn": csg.GEMV_PATH_DYN}
WORK_OFF, EPOCH_OFF, DONE_OFF = 64, 96, 112   # slot 0's pad: work[2], epoch, tiles_done


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _pad_words(ws, nbytes):
    torch.cuda.synchronize()
    v = torch.as_tensor(DeviceView(ws.pads[0], (nbytes // 4,), "<i4"), device=ws.device)
    return v.cpu().numpy().astype(np.int64)


def _counters(ws, tiles):
    info = csg.symm_info(ws.h)
    off = 128 + -(-4 * info["max_tiles"] // 128) * 128
    torch.cuda.synchronize()
    v = torch.as_tensor(DeviceView(ws.pads[0] + off, (tiles,), "<i4"), device=ws.device)
    return v.cpu().numpy()


def _case(R=4, N=576, K=2048, B=2, seed=41):
    W, x = synth.gemv_inputs(R, N, K, B, seed=seed, w_std=1.0 / np.sqrt(K), x="normal")
    return W, x


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("B", [2, 8])
def test_pad_is_clean_after_every_launch(path, B):
    """The global-memory protocol (per-tile kernel, and the persistent
    kernel drawing units): after launch e the epoch word holds e, tiles_done
    and every tile counter are zero, and the work counter the next launch
    draws from (work[(e + 1) & 1]) is zero."""
    R, N, K = 4, 576, 2048
    W, x = _case(R, N, K, B)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, PATHS[path])
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_CLUSTER, 0)
        ws.load_W(W)
        ws.load_x(x)
        plan = csg.symm_gemv_plan(ws.h, N, K, B)
        s = torch.cuda.current_stream()
        for e in range(1, 5):
            ws.run(s)
            words = _pad_words(ws, 128)
            assert words[EPOCH_OFF // 4] == e
            assert words[DONE_OFF // 4] == 0
            assert words[WORK_OFF // 4 + ((e + 1) & 1)] == 0
            assert not _counters(ws, plan["tiles"]).any()
            if path == "dyn":
                units = plan["tiles"] * R * plan["splits"]
                assert words[WORK_OFF // 4 + (e & 1)] == units   # every unit drawn, plus one stop per CTA
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


@pytest.mark.parametrize("B", [2, 8])
def test_cluster_epilogue_leaves_the_pad_untouched(B):
    """The persistent kernel's cluster epilogue (the automatic plan of this
    small layer: K split inside the clusters) draws nothing and publishes
    nothing: the epoch, work counters, tiles_done and tile counters stay
    zero launch after launch."""
    R, N, K = 4, 576, 2048
    W, x = _case(R, N, K, B)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        ws.load_W(W)
        ws.load_x(x)
        plan = csg.symm_gemv_plan(ws.h, N, K, B)
        assert plan["cluster"] == R * plan["splits"] and plan["splits"] > 1
        s = torch.cuda.current_stream()
        for _ in range(4):
            ws.run(s)
            words = _pad_words(ws, 128)
            assert not words[WORK_OFF // 4:WORK_OFF // 4 + 2].any()
            assert words[EPOCH_OFF // 4] == 0 and words[DONE_OFF // 4] == 0
            assert not _counters(ws, plan["tiles"]).any()
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("mode", ["all_reduce", "reduce_scatter", "bias_rmsnorm"])
def test_graph_replay_matches_eager(path, mode):
    """A captured call replayed with new x each time gives the eager call's
    bits, also with eager calls of another geometry on the handle in
    between (they change the tile count, the contributors per tile and the
    grid)."""
    R, N, K, B = 4, 576, 2048, 8
    W, x0 = _case(R, N, K, B)
    bias, gamma = synth.norm_vectors(N, 43)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, PATHS[path])
        ws.load_W(W)
        ws.load_x(x0)
        ws.load_vectors(bias, gamma)
        s = torch.cuda.current_stream()
        ws.run(s, mode=mode)             # first call outside the capture (attributes, descriptors)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ws.run(torch.cuda.current_stream(), mode=mode)
        read = ws.read_y_rs if mode == "reduce_scatter" else ws.read_y
        for i in range(4):
            _, x = synth.gemv_inputs(R, N, K, B, seed=100 + i, w_std=1.0, x="normal")
            ws.load_x(x)
            ws.fill_y(0xFF)
            g.replay()
            y_graph = read()
            ws.fill_y(0xFF)
            ws.run(s, mode=mode)
            y_eager = read()
            assert np.array_equal(y_graph, y_eager), f"replay {i}"
            if mode == "all_reduce":
                check_gemv(W, x, y_graph)
            # another geometry on the same handle between replays
            csg.gemv_all_reduce(ws.h, ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), R, 320 - 64 * i, K, 1 + i, s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK, f"replay {i}"
        del g
    finally:
        ws.close()


def test_captured_decode_chain():
    """R = 1, N = K: six fused calls, each reading the previous call's y as
    x (chained launches), the last one with the bias + RMSNorm epilogue,
    captured once and replayed with new inputs; the bits match the same chain
    issued eagerly."""
    N = K = 2048
    B, steps = 2, 6
    W, _ = synth.gemv_inputs(1, N, K, B, seed=47, w_std=1.0 / np.sqrt(K), x="normal")
    bias, gamma = synth.norm_vectors(N, 47)
    ws = GemvWorkspace(1, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        ws.load_W(W)
        ws.load_vectors(bias, gamma)
        vbytes = B * N * 2
        vstep = (vbytes + 255) // 256 * 256
        base = ws.W_ptr(1)

        def chain(stream):
            for i in range(steps - 1):
                csg.gemv_all_reduce(ws.h, ws.W_ptr(0), base + i * vstep, base + (i + 1) * vstep, 1, N, K, B, stream)
            csg.gemv_all_reduce_bias_rmsnorm(ws.h, ws.W_ptr(0), base + (steps - 1) * vstep, ws.base + ws.bias_off,
                                             ws.base + ws.gamma_off, base + steps * vstep, 1, N, K, B, 1e-6, stream)

        def load_v0(x):
            ws.view(0, ws.w_off[1], vbytes).copy_(torch.from_numpy(np.ascontiguousarray(x[0])).view(torch.uint8)
                                                  .reshape(-1))

        def region():
            torch.cuda.synchronize()
            return ws.view(0, ws.w_off[1], (steps + 1) * vstep).cpu().numpy().copy()

        s = torch.cuda.current_stream()
        _, x = synth.gemv_inputs(1, N, K, B, seed=48, w_std=1.0, x="normal")
        load_v0(x)
        chain(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain(torch.cuda.current_stream())
        for i in range(3):
            _, x = synth.gemv_inputs(1, N, K, B, seed=50 + i, w_std=1.0, x="normal")
            load_v0(x)
            g.replay()
            got = region()
            load_v0(x)
            chain(s)
            want = region()
            assert np.array_equal(got, want), f"replay {i}"
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        del g
    finally:
        ws.close()


@pytest.mark.parametrize("op", ["one_shot", "two_shot", "reduce_scatter"])
def test_captured_collectives(op):
    """The all-reduce family (the two-shot's second phase is a programmatic
    dependent of the first) and the all-reduce + bias + RMSNorm, captured and
    replayed with new inputs: the eager call's bits."""
    R, n = 8, 8 * 4096 + 8 * 24
    aw = AllReduceWorkspace(R, n)
    nw = RmsNormWorkspace(R, 2, 4096)
    try:
        rng = np.random.default_rng(61)
        s = torch.cuda.current_stream()
        aw.load_in(synth.allreduce_inputs(R, n, 61))
        aw.run(s, op=op)
        x_n, bias, gamma = synth.rmsnorm_inputs(R, 2, 4096, 61)
        nw.load(x_n, bias, gamma)
        nw.run(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            aw.run(cs, op=op)
            nw.run(cs)
        count = n // R if op == "reduce_scatter" else n
        for i in range(3):
            seed = int(rng.integers(1 << 30))
            aw.load_in(synth.allreduce_inputs(R, n, seed))
            x_n, bias, gamma = synth.rmsnorm_inputs(R, 2, 4096, seed)
            nw.load(x_n, bias, gamma)
            g.replay()
            got = (aw.read_out(count=count), nw.read_out())
            aw.run(s, op=op)
            nw.run(s)
            want = (aw.read_out(count=count), nw.read_out())
            assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]), f"replay {i}"
        del g
    finally:
        aw.close()
        nw.close()
