"""gemv_all_reduce_noalloc through the C ABI, against gemv_all_reduce.

The allocation-free entry point serves callers that cannot allocate device
memory (their memory belongs to another allocator, or allocation's implicit
synchronisation is not allowed where they run).  It computes in the library's
fixed working array instead of a handle's scratch and signal pad.  This file
is collected last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process and after the others.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import require_gpu
from helpers import f64_to_words_via_f32, tolerance_ratio, words_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CASES = [
    # (R, N, K, B): the decode shape, a ragged small batch, a wide batch
    (8, 8192, 28672, 1),
    (4, 777, 4 * 264, 3),
    (4, 2048, 4 * 1024, 16),
]


@pytest.mark.parametrize("R,N,K,B", CASES, ids=[f"R{c[0]}N{c[1]}K{c[2]}B{c[3]}" for c in CASES])
def test_noalloc_matches_gemv_all_reduce(R, N, K, B):
    """Two calls in a row of the allocation-free entry point against
    gemv_all_reduce on its CUDA-core kernel (the kernel the allocation-free
    one is a variant of) and against the fp64 oracle, within the parity
    tolerance."""
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + B, w_std=0.02, x="normal")
    y_oracle, _ = oracle.gemv_all_reduce(W, x)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_FFMA)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        ws.fill_y(0xFF)
        ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        y_existing = words_to_f64(ws.read_y()[0])
        outs = []
        for _ in range(2):   # two calls in a row share (and reuse) the fixed array
            ws.fill_y(0xFF)
            csg.gemv_all_reduce_noalloc(ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), ws.stride, R, N, K, B, s)
            y = ws.read_y()
            for r in range(1, R):
                assert np.array_equal(y[r], y[0]), f"replica {r} differs"
            got = words_to_f64(y[0])
            assert tolerance_ratio(got, y_existing) <= 1.0
            assert tolerance_ratio(got, y_oracle) <= 1.0
            outs.append(y)
        # the second call, on an array the first one left behind, gives the
        # first call's bits
        assert np.array_equal(outs[1], outs[0]), "the second call's bits differ from the first's"
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


INT_CASES = [(2, 256, 2 * 256, 1), (3, 77, 3 * 40, 5), (8, 300, 8 * 24, 16)]


@pytest.mark.parametrize("R,N,K,B", INT_CASES, ids=[f"R{c[0]}N{c[1]}K{c[2]}B{c[3]}" for c in INT_CASES])
def test_noalloc_small_integers_bit_exact(R, N, K, B):
    """Small-integer inputs make every product and partial sum an exact
    integer in fp32, so the allocation-free call must give the oracle's bf16
    words exactly, on two calls in a row (the second reuses the shared array
    the first one left behind), and the same words as gemv_all_reduce."""
    rng = np.random.default_rng(N + B)
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, K // R)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, K // R)).astype(np.float64))
    _, y_or = oracle.gemv_all_reduce(W, x)
    ws = GemvWorkspace(R, N, K, B)
    try:
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        ws.fill_y(0xFF)
        ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        y_existing = ws.read_y()
        outs = []
        for _ in range(2):
            ws.fill_y(0xFF)
            csg.gemv_all_reduce_noalloc(ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), ws.stride, R, N, K, B, s)
            y = ws.read_y()
            for r in range(R):
                assert np.array_equal(y[r], y_or[0]), f"rank {r}'s y differs from the oracle's words"
            outs.append(y)
        assert np.array_equal(outs[1], outs[0])
        assert np.array_equal(outs[0], y_existing), "differs from gemv_all_reduce"
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


def test_noalloc_rejects_what_does_not_fit():
    ws = GemvWorkspace(2, 64, 128, 2)
    try:
        s = torch.cuda.current_stream()
        with pytest.raises(csg.SymmError) as e:   # 64 * 16 * 8192 * 4 B of partials > 16 MiB
            csg.gemv_all_reduce_noalloc(ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), ws.stride, 64, 8192, 64 * 8, 16, s)
        assert e.value.code == csg.SYMM_ERANGE
        assert "no-alloc" in csg.symm_last_error()
        with pytest.raises(csg.SymmError) as e:   # y overlapping W
            csg.gemv_all_reduce_noalloc(ws.W_ptr(), ws.x_ptr(), ws.W_ptr(), ws.stride, 2, 64, 128, 2, s)
        assert e.value.code == csg.SYMM_EINVAL
        with pytest.raises(csg.SymmError) as e:   # misaligned stride
            csg.gemv_all_reduce_noalloc(ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), ws.stride + 8, 2, 64, 128, 2, s)
        assert e.value.code == csg.SYMM_EINVAL
    finally:
        ws.close()
