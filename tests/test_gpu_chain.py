"""Chained fused calls (SYMM_OPT_CHAIN = 1): the persistent kernel launched as a
programmatic dependent of the previous call may start while that call drains,
loading W early and everything else only after the previous grid has
finished.  Checked on the GPU, through the C ABI: a chain whose every call
reads the previous call's output as x gives the same bits as the same chain
in plain stream order, back-to-back calls on one handle never trip the
protocol, and the first result matches the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dependent_chain(chain: int, steps: int, B: int):
    """R = 1, N = K: call i + 1 reads call i's y as its x, so a call that read
    x before its predecessor finished would see a stale vector.  The vectors
    v_0 = x, v_1, ..., v_steps live in the second W copy's region, so the calls
    follow one another on the stream with nothing in between.  Returns
    (W, x, every call's y as bf16 words (steps, 1, B, N))."""
    N = K = 2048
    W, x = synth.gemv_inputs(1, N, K, B, seed=17, w_std=1.0 / np.sqrt(K), x="normal")
    ws = GemvWorkspace(1, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        ws.load_W(W)
        vbytes = B * N * 2
        vstep = (vbytes + 255) // 256 * 256
        assert (steps + 1) * vstep <= ws.w_bytes
        base = ws.W_ptr(1)
        ws.view(0, ws.w_off[1], vbytes).copy_(torch.from_numpy(np.ascontiguousarray(x[0])).view(torch.uint8).reshape(-1))
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for i in range(steps):
            csg.gemv_all_reduce(ws.h, ws.W_ptr(0), base + i * vstep, base + (i + 1) * vstep, 1, N, K, B, s)
        code, _, _ = csg.symm_status(ws.h, s)
        assert code == csg.SYMM_OK
        region = ws.view(0, ws.w_off[1], (steps + 1) * vstep).cpu().numpy()
        outs = np.stack([region[(i + 1) * vstep:(i + 1) * vstep + vbytes].view(np.uint16).reshape(1, B, N)
                         for i in range(steps)])
        return W, x, outs
    finally:
        ws.close()


@pytest.mark.parametrize("B", [1, 2, 8])
def test_dependent_chain_matches_plain_stream_order(B):
    W, x, plain = _dependent_chain(0, 12, B)
    _, _, chained = _dependent_chain(1, 12, B)
    assert np.array_equal(chained, plain)
    # the first call against the oracle
    check_gemv(W, x, plain[0])


def test_back_to_back_calls_on_one_handle():
    w = synth.WORKLOADS["mlp_down_decode"]
    R, N, K, B = w["R"], w["N"], w["K"], w["B"]
    W, x = synth.gemv_inputs(R, N, K, B, w["seed"], w["w_std"], w["x"])
    ws = GemvWorkspace(R, N, K, B, copies=2)
    try:
        for c in range(2):
            ws.load_W(W, copy=c)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        results = {}
        for chain in (0, 1):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
            ws.fill_y(0xFF)
            for i in range(40):
                ws.run(s, copy=i % 2)
            code, rank, tile = csg.symm_status(ws.h, s)
            assert code == csg.SYMM_OK, (chain, rank, tile)
            results[chain] = ws.read_y()
        assert np.array_equal(results[0], results[1])
        check_gemv(W, x, results[1])
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


def test_chained_call_after_rmsnorm_and_allreduce():
    # a chained launch that follows kernels of other calls on the stream
    R, N, K, B = 4, 1024, 4096, 2
    W, x = synth.gemv_inputs(R, N, K, B, seed=21, w_std=0.05)
    bias, gamma = synth.norm_vectors(N, 21)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        ws.load_W(W)
        ws.load_x(x)
        ws.load_vectors(bias, gamma)
        s = torch.cuda.current_stream()
        ws.run(s, mode="bias_rmsnorm")
        ws.run(s)
        csg.one_shot_all_reduce(ws.h, ws.y_ptr(), ws.base + ws.bias_off, R, N, s)   # an unrelated kernel
        ws.run(s)
        code, _, _ = csg.symm_status(ws.h, s)
        assert code == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


def _weights_from_previous_output(chain: int):
    """Call A writes y (B x N); call B uses that same memory as its W
    (N x K with K = B).  A chained launch of B would read W early, so the
    library launches B in plain stream order; the result must not depend on
    the option."""
    R, N, K, B = 1, 512, 8, 8
    W, x = synth.gemv_inputs(R, N, K, B, seed=23, w_std=0.3, x="normal")
    ws = GemvWorkspace(R, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        y_a = ws.W_ptr(1)                       # A's output, B's weights (8 KB, the W copy's size)
        csg.gemv_all_reduce(ws.h, ws.W_ptr(0), ws.x_ptr(), y_a, R, N, K, B, s)
        csg.gemv_all_reduce(ws.h, y_a, ws.x_ptr(), ws.y_ptr(), R, N, K, B, s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        return ws.read_y()
    finally:
        ws.close()


def test_weights_that_are_the_previous_output_are_not_read_early():
    assert np.array_equal(_weights_from_previous_output(1), _weights_from_previous_output(0))


def _rmsnorm_chain(chain: int, steps: int = 8):
    """R = 1, N = K: fused calls with the bias + RMSNorm epilogue, each
    reading the previous call's normalised output as x; the norm kernel lets
    the next fused call start early."""
    N = K = 2048
    B = 2
    W, x = synth.gemv_inputs(1, N, K, B, seed=29, w_std=1.0 / np.sqrt(K), x="normal")
    bias, gamma = synth.norm_vectors(N, 29)
    ws = GemvWorkspace(1, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        ws.load_W(W)
        ws.load_vectors(bias, gamma)
        vbytes = B * N * 2
        vstep = (vbytes + 255) // 256 * 256
        base = ws.W_ptr(1)
        ws.view(0, ws.w_off[1], vbytes).copy_(torch.from_numpy(np.ascontiguousarray(x[0])).view(torch.uint8).reshape(-1))
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for i in range(steps):
            csg.gemv_all_reduce_bias_rmsnorm(ws.h, ws.W_ptr(0), base + i * vstep, ws.base + ws.bias_off,
                                             ws.base + ws.gamma_off, base + (i + 1) * vstep, 1, N, K, B, 1e-6, s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        region = ws.view(0, ws.w_off[1], (steps + 1) * vstep).cpu().numpy()
        return np.stack([region[(i + 1) * vstep:(i + 1) * vstep + vbytes].view(np.uint16) for i in range(steps)])
    finally:
        ws.close()


def test_rmsnorm_chain_matches_plain_stream_order():
    assert np.array_equal(_rmsnorm_chain(1), _rmsnorm_chain(0))
