"""The unfused form of the fused layer (SYMM_OPT_UNFUSED): the persistent
GEMV storing every rank's fp32 partials, then a separate all-reduce kernel
over them.  It exists to measure what fusion buys, so it must compute exactly
what the fused call computes: the same bits, on every shape, split count and
weight layout, and the oracle's words on small-integer inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu
from helpers import f64_to_words_via_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(W, x, unfused, splits=0, packed=False, chain=1, repeat=2):
    R, N, Kr = W.shape
    B = x.shape[1]
    ws = GemvWorkspace(R, N, R * Kr, B, packed=packed)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, splits)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, chain)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, int(unfused))
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        outs = []
        for _ in range(repeat):
            ws.fill_y(0xFF)
            ws.run(s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            outs.append(ws.read_y())
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        return outs
    finally:
        ws.close()


SHAPES = [(8, 1000, 8 * 512, 1), (4, 8192 // 8, 4 * 1024, 8), (2, 130, 2 * 520, 3), (8, 300, 8 * 264, 16),
          (3, 257, 3 * 136, 2)]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("packed", [False, True], ids=["rowmajor", "packed"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"R{a}N{b}K{c}B{d}" for a, b, c, d in SHAPES])
def test_unfused_gives_the_fused_bits(splits, packed, shape):
    R, N, K, B = shape
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + B + splits, w_std=0.02, x="normal")
    fused = _run(W, x, False, splits, packed)
    unfused = _run(W, x, True, splits, packed)
    for y in fused + unfused:
        assert np.array_equal(y, fused[0])
    check_gemv(W, x, unfused[0])


@pytest.mark.parametrize("chain", [0, 1])
def test_unfused_small_integers_bit_exact(chain):
    rng = np.random.default_rng(5)
    R, N, Kr, B = 4, 300, 264, 5
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    (y, _) = _run(W, x, True, chain=chain)
    check_gemv(W, x, y, exact=True)


def test_unfused_and_fused_calls_alternate_on_one_handle():
    """The unfused launches keep the pad's protocol state consistent: fused
    and unfused calls alternate, chained, with no reset in between."""
    R, N, K, B = 8, 1024, 8 * 1024, 2
    W, x = synth.gemv_inputs(R, N, K, B, seed=9, w_std=0.02, x="normal")
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        for i in range(12):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, i % 2)
            ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


def test_unfused_rejections():
    R, N, K, B = 2, 64, 2 * 64, 2
    ws = GemvWorkspace(R, N, K, B)
    try:
        s = torch.cuda.current_stream()
        csg.symm_set_option(ws.h, csg.SYMM_OPT_UNFUSED, 1)
        for mode in ("reduce_scatter", "bias_rmsnorm"):
            with pytest.raises(csg.SymmError) as e:
                ws.run(s, mode=mode)
            assert e.value.code == csg.SYMM_EINVAL
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_FFMA)
        with pytest.raises(csg.SymmError) as e:
            ws.run(s)
        assert e.value.code == csg.SYMM_EINVAL
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_AUTO)
        with pytest.raises(csg.SymmError) as e:   # K = 0
            csg.gemv_all_reduce(ws.h, ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), R, N, 0, B, s)
        assert e.value.code == csg.SYMM_EINVAL
    finally:
        ws.close()
