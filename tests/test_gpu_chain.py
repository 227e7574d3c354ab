"""Chained calls (SYMM_OPT_CHAIN = 1): the persistent kernel and the one-shot
all-reduce launched as programmatic dependents of the previous call may start
while that call drains; the fused call loads W early and everything else only
after the previous grid has finished, the all-reduce reads nothing before.
Checked on the GPU, through the C ABI: a chain whose every call reads the
previous call's output gives the same bits as the same chain in plain stream
order, back-to-back calls on one handle never trip the protocol, W written by
the previous call (a fused call's y, an all-reduce's output) is not read
early, and the first result matches the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import AllReduceWorkspace, GemvWorkspace, RmsNormWorkspace
from gpu_common import check_gemv, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dependent_chain(chain: int, steps: int, B: int, path=csg.GEMV_PATH_DYN):
    """R = 1, N = K: call i + 1 reads call i's y as its x, so a call that read
    x before its predecessor finished would see a stale vector.  The vectors
    v_0 = x, v_1, ..., v_steps live in the second W copy's region, so the calls
    follow one another on the stream with nothing in between.  Returns
    (W, x, every call's y as bf16 words (steps, 1, B, N))."""
    N = K = 2048
    W, x = synth.gemv_inputs(1, N, K, B, seed=17, w_std=1.0 / np.sqrt(K), x="normal")
    ws = GemvWorkspace(1, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
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
@pytest.mark.parametrize("path", ["dyn", "ffma"])
def test_dependent_chain_matches_plain_stream_order(B, path):
    p = {"dyn": csg.GEMV_PATH_DYN, "ffma": csg.GEMV_PATH_FFMA}[path]
    W, x, plain = _dependent_chain(0, 12, B, p)
    _, _, chained = _dependent_chain(1, 12, B, p)
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


def _allreduce_chain(chain: int, steps: int = 10, kernel=csg.AR_KERNEL_PER_THREAD):
    """In-place one-shot all-reduces, each reading what the previous one
    wrote: a chained launch that read its inputs before its predecessor had
    finished would see stale values."""
    R, n = 4, (1 << 18) + 24
    aw = AllReduceWorkspace(R, n, separate_out=False)
    try:
        csg.symm_set_option(aw.h, csg.SYMM_OPT_CHAIN, chain)
        csg.symm_set_option(aw.h, csg.SYMM_OPT_AR_KERNEL, kernel)
        inp = synth.allreduce_inputs(R, n, 31)   # grows by about R per call: 10 calls stay finite
        aw.load_in(inp)
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for _ in range(steps):
            aw.run(s, op="one_shot")
        return aw.read_out()
    finally:
        aw.close()


@pytest.mark.parametrize("kernel", [csg.AR_KERNEL_PER_THREAD, csg.AR_KERNEL_STAGED])
def test_chained_allreduce_chain_matches_plain_stream_order(kernel):
    plain = _allreduce_chain(0, kernel=kernel)
    chained = _allreduce_chain(1, kernel=kernel)
    assert np.array_equal(chained, plain)
    # one call against the oracle
    inp = synth.allreduce_inputs(4, (1 << 18) + 24, 31)
    one = _allreduce_chain(1, steps=1, kernel=kernel)
    _, want = oracle.one_shot_all_reduce(inp)
    assert np.array_equal(one[0], want[0])


def test_weights_written_by_an_allreduce_are_not_read_early():
    """An all-reduce writes the region the next fused call reads as W; the
    fused call must then launch in plain stream order (a chained launch
    would load W before the all-reduce had finished)."""
    R, N, K, B = 2, 256, 2 * 256, 2
    W, x = synth.gemv_inputs(R, N, K, B, seed=37, w_std=0.05, x="normal")
    ws = GemvWorkspace(R, N, K, B, copies=2)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        ws.load_W(W, copy=0)
        ws.load_W(W, copy=1)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        n = N * (K // R)
        ws.run(s, copy=0)                                       # an earlier fused call
        csg.one_shot_all_reduce(ws.h, ws.W_ptr(1), ws.W_ptr(1), R, n, s)   # W copy 1 <- sum over ranks
        ws.run(s, copy=1)                                       # reads the all-reduce's output as W
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        _, summed = oracle.one_shot_all_reduce(W.reshape(R, -1))
        check_gemv(summed.reshape(R, N, K // R), x, ws.read_y())
    finally:
        ws.close()


def _collective_chain(chain: int, rounds: int = 5):
    """Two-shot (in place), reduce-scatter (reading the two-shot's output),
    multi-root tile reduce (quadrants of the same tensor) and one-shot (in
    place), repeated: every call reads what an earlier one wrote."""
    R, side = 4, 256
    n = side * side
    aw = AllReduceWorkspace(R, n)
    try:
        csg.symm_set_option(aw.h, csg.SYMM_OPT_CHAIN, chain)
        aw.load_in(synth.allreduce_inputs(R, n, 41))
        s = torch.cuda.current_stream()
        inp, out = aw.base + aw.in_off, aw.base + aw.out_off
        h = side // 2
        quads = [inp + (a * side + b) * 2 for a in (0, h) for b in (0, h)]
        torch.cuda.synchronize()
        for _ in range(rounds):
            csg.two_shot_all_reduce(aw.h, inp, inp, R, n, s)
            csg.reduce_scatter(aw.h, inp, out, R, n, s)
            csg.multi_root_tile_reduce(aw.h, quads, out + (n // R) * 2, [3, 2, 1, 0], h, h, side, side, s)
            csg.one_shot_all_reduce(aw.h, inp, inp, R, n, s)
        torch.cuda.synchronize()
        return (np.stack([aw.view(r, aw.in_off, n * 2).cpu().numpy() for r in range(R)]),
                np.stack([aw.view(r, aw.out_off, n * 2).cpu().numpy() for r in range(R)]))
    finally:
        aw.close()


def test_chained_collectives_match_plain_stream_order():
    plain = _collective_chain(0)
    chained = _collective_chain(1)
    assert np.array_equal(chained[0], plain[0]) and np.array_equal(chained[1], plain[1])


def _rmsnorm_standalone_chain(chain: int, steps: int = 8):
    """all_reduce_bias_rmsnorm in place, each call reading the previous
    call's normalised output."""
    R, rows, H = 8, 2, 8192
    nw = RmsNormWorkspace(R, rows, H, in_place=True)
    try:
        csg.symm_set_option(nw.h, csg.SYMM_OPT_CHAIN, chain)
        nw.load(*synth.rmsnorm_inputs(R, rows, H, 43))
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for _ in range(steps):
            nw.run(s)
        return nw.read_out()
    finally:
        nw.close()


def test_chained_standalone_rmsnorm_matches_plain_stream_order():
    assert np.array_equal(_rmsnorm_standalone_chain(1), _rmsnorm_standalone_chain(0))


def _interleaved(chain: int):
    """Two handles on one stream, their fused calls alternating, and a
    PyTorch kernel rewriting one handle's x between its calls: chained
    launches must read x only after the kernel before them has finished."""
    R, N, K, B = 4, 1024, 4 * 1024, 2
    Wa, xa = synth.gemv_inputs(R, N, K, B, seed=51, w_std=0.03, x="normal")
    Wb, xb = synth.gemv_inputs(R, N, K, B, seed=52, w_std=0.03, x="normal")
    _, xa2 = synth.gemv_inputs(R, N, K, B, seed=53, w_std=0.03, x="normal")
    wa, wb = GemvWorkspace(R, N, K, B), GemvWorkspace(R, N, K, B)
    try:
        for ws, W, x in ((wa, Wa, xa), (wb, Wb, xb)):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
            csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
            ws.load_W(W)
            ws.load_x(x)
        x_new = [torch.from_numpy(np.ascontiguousarray(xa2[r])).view(torch.int16).reshape(-1).to(wa.device)
                 for r in range(R)]
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        ys = []
        for i in range(6):
            wa.run(s)
            wb.run(s)
            if i == 2:
                for r in range(R):   # a PyTorch kernel writes x of handle a right before its next call
                    torch.bitwise_xor(x_new[r], 0, out=wa.x_view(r).view(torch.int16))
            ys.append((wa.read_y(), wb.read_y()) if i in (2, 5) else None)
        assert csg.symm_status(wa.h, s)[0] == csg.SYMM_OK and csg.symm_status(wb.h, s)[0] == csg.SYMM_OK
        return [y for y in ys if y is not None], (Wa, xa, xa2, Wb, xb)
    finally:
        wa.close()
        wb.close()


def test_two_handles_and_foreign_writes_between_chained_calls():
    plain, (Wa, xa, xa2, Wb, xb) = _interleaved(0)
    chained, _ = _interleaved(1)
    for (ya_p, yb_p), (ya_c, yb_c) in zip(plain, chained):
        assert np.array_equal(ya_p, ya_c) and np.array_equal(yb_p, yb_c)
    check_gemv(Wa, xa, chained[0][0])
    check_gemv(Wa, xa2, chained[1][0])
    check_gemv(Wb, xb, chained[1][1])


def _rewritten_row_major_weights(chain: int):
    """Row-major W_r rewritten by a PyTorch kernel right before each fused
    call, with no synchronisation in between: a chained call must load a
    row-major W only after the kernel before it has finished (only packed
    weights, which symm_pack_w alone writes, are loaded early)."""
    R, N, K, B = 4, 2048, 4 * 2048, 2
    Ws = [synth.gemv_inputs(R, N, K, B, seed=80 + i, w_std=0.03, x="normal")[0] for i in range(4)]
    _, x = synth.gemv_inputs(R, N, K, B, seed=80, w_std=0.03, x="normal")
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        ws.load_W(Ws[0])
        ws.load_x(x)
        dev_w = [[torch.from_numpy(np.ascontiguousarray(W[r])).view(torch.int16).reshape(-1).to(ws.device)
                  for r in range(R)] for W in Ws]
        outs = [torch.empty((R, B * N), dtype=torch.int16, device=ws.device) for _ in Ws]
        s = torch.cuda.current_stream()
        torch.cuda.synchronize()
        for i in range(len(Ws)):
            if i > 0:
                for r in range(R):   # PyTorch kernels write the weights right before the call
                    torch.bitwise_xor(dev_w[i][r], 0, out=ws.w_view(r).view(torch.int16))
            ws.run(s)
            for r in range(R):
                outs[i][r].copy_(ws.y_view(r).view(torch.int16))
        torch.cuda.synchronize()
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        return [o.cpu().numpy().view(np.uint16).reshape(R, B, N) for o in outs], Ws, x
    finally:
        ws.close()


def test_row_major_weights_written_just_before_a_chained_call():
    plain, Ws, x = _rewritten_row_major_weights(0)
    chained, _, _ = _rewritten_row_major_weights(1)
    for i, (yp, yc) in enumerate(zip(plain, chained)):
        assert np.array_equal(yp, yc), f"call {i}: chained differs from plain stream order"
        check_gemv(Ws[i], x, yc)
