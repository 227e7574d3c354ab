"""Shared pieces of the GPU tests: run a GEMV / all-reduce through the C ABI
and compare with the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
from collective_split_gemv_gb300.workspace import AllReduceWorkspace, GemvWorkspace
from helpers import tolerance_ratio, ulp_distance, words_to_f64


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from collective_split_gemv_gb300 import _build
    _build.build()
    csg.lib()


def run_gemv(W, x, path=csg.GEMV_PATH_AUTO, order=0, repeat=1, y_fill=0xFF, options=()):
    """Run the fused kernel `repeat` times; returns (list of y (R, B, N) words,
    workspace status triple of the last run).  `options`: further
    (option, value) pairs set on the handle."""
    R, N, Kr = W.shape
    B = x.shape[1]
    ws = GemvWorkspace(R, N, R * Kr, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_TILE_ORDER, order)
        for opt, val in options:
            csg.symm_set_option(ws.h, opt, val)
        ws.load_W(W)
        ws.load_x(x)
        stream = torch.cuda.current_stream()
        outs = []
        status = None
        for _ in range(repeat):
            ws.fill_y(y_fill)
            ws.run(stream)
            status = csg.symm_status(ws.h, stream)
            outs.append(ws.read_y())
        rc, bad_rank, band = csg.symm_check_guards(ws.h)
        assert rc == csg.SYMM_OK, f"guard band {band} of rank {bad_rank} overwritten"
        return outs, status
    finally:
        ws.close()


def check_gemv(W, x, y, y_ref=None, exact=False):
    """y (R, B, N) words against the oracle: tolerance, replicas identical.
    Returns (tolerance ratio, fraction bit-equal to the oracle's bf16, max ulp)."""
    if y_ref is None:
        y_ref, y_or = oracle.gemv_all_reduce(W, x)
    else:
        y_or = None
    R = y.shape[0]
    for s in range(1, R):
        assert np.array_equal(y[s], y[0]), f"replica {s} differs from replica 0"
    if exact:
        assert y_or is not None
        assert np.array_equal(y[0], y_or[0]), "exact case differs from the oracle"
    ratio = tolerance_ratio(words_to_f64(y[0]), y_ref)
    assert ratio <= 1.0, f"tolerance exceeded: ratio {ratio}"
    if y_or is not None:
        eq = float(np.mean(y[0] == y_or[0])) if y[0].size else 1.0
        ulp = int(ulp_distance(y[0], y_or[0]).max()) if y[0].size else 0
    else:
        eq, ulp = float("nan"), -1
    return ratio, eq, ulp


def run_allreduce(inp, in_place=False, kernel=csg.AR_KERNEL_AUTO):
    R, n = inp.shape
    aw = AllReduceWorkspace(R, n, separate_out=not in_place)
    try:
        csg.symm_set_option(aw.h, csg.SYMM_OPT_AR_KERNEL, kernel)
        aw.load_in(inp)
        aw.run(torch.cuda.current_stream())
        out = aw.read_out()
        rc, bad_rank, band = csg.symm_check_guards(aw.h)
        assert rc == csg.SYMM_OK, f"guard band {band} of rank {bad_rank} overwritten"
        return out
    finally:
        aw.close()
