"""Packed weights (symm_pack_w) on the GPU, through the C ABI.

The packed bytes are compared with the layout as the header defines it,
written out here in numpy; every fused form on a packed weight must give
bitwise the results of the same call on the row-major weight, and be within
the oracle's tolerance (small-integer inputs: equal to the oracle); the
registration rules (shape and path checks, release, overlap) hold."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _packed_layout(Wr: np.ndarray) -> np.ndarray:
    """One slot's packed bytes from its row-major (N, Kr) words: 128 x 64
    blocks, block-row-major; inside a block row i holds 8 chunks of 8
    elements, chunk c at position c XOR (i mod 8); zero padding; one zero
    block at the end."""
    N, Kr = Wr.shape
    T, J = -(-N // 128), -(-Kr // 64)
    full = np.zeros((T * 128, J * 64), dtype=np.uint16)
    full[:N, :Kr] = Wr
    out = np.zeros((T * J + 1, 128, 8, 8), dtype=np.uint16)     # block, row, chunk position, element
    rows = np.arange(128)[:, None]
    pos = np.arange(8)[None, :] ^ (rows & 7)
    for t in range(T):
        for j in range(J):
            blk = full[t * 128:(t + 1) * 128, j * 64:(j + 1) * 64].reshape(128, 8, 8)
            out[t * J + j][rows, pos] = blk
    return out.reshape(-1).view(np.uint8)


def _int_case(R, N, Kr, B, seed):
    rng = np.random.default_rng(seed)
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    return W, x


def _run(W, x, packed, options=(), mode="all_reduce", vectors=None, order=0):
    R, N, Kr = W.shape
    B = x.shape[1]
    ws = GemvWorkspace(R, N, R * Kr, B, packed=packed)
    try:
        for opt, val in options:
            csg.symm_set_option(ws.h, opt, val)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_TILE_ORDER, order)
        ws.load_W(W)
        ws.load_x(x)
        if vectors is not None:
            ws.load_vectors(*vectors)
        s = torch.cuda.current_stream()
        ws.fill_y(0xFF)
        ws.run(s, mode=mode)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        y = ws.read_y_rs() if mode == "reduce_scatter" else ws.read_y()
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        return y
    finally:
        ws.close()


@pytest.mark.parametrize("R,N,Kr", [(1, 1, 8), (2, 200, 200), (3, 128, 64), (2, 300, 1032), (4, 129, 136)])
def test_packed_bytes_follow_the_layout(R, N, Kr):
    W, _ = _int_case(R, N, Kr, 1, seed=N + Kr)
    ws = GemvWorkspace(R, N, R * Kr, 1, packed=True)
    try:
        ws.fill_y(0)
        for r in range(R):
            ws.view(r, ws.wp_off[0], ws.wp_bytes).fill_(0x5A)   # stale bytes the packer must overwrite
        ws.load_W(W)
        torch.cuda.synchronize()
        assert ws.wp_bytes == csg.symm_packed_w_bytes(R, N, R * Kr)
        for r in range(R):
            got = ws.view(r, ws.wp_off[0], ws.wp_bytes).cpu().numpy()
            assert np.array_equal(got, _packed_layout(W[r])), f"slot {r}"
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


PIPES = [(1, 1), (2, 1), (4, 1), (1, 2), (2, 2), (3, 2), (1, 3)]   # (slabs, CTAs per SM)
SHAPES = [(8, 300, 264, 2), (4, 1000, 2056, 3), (2, 17, 8, 1), (3, 513, 4096, 16), (2, 129, 72, 8)]


VARIANTS = [(s, c, sh) for s, c in PIPES for sh in SHAPES]


@pytest.mark.parametrize("slabs,cps,shape", VARIANTS,
                         ids=[f"slabs{s}-cps{c}-R{a}N{b}Kr{k}B{d}" for s, c, (a, b, k, d) in VARIANTS])
def test_packed_equals_row_major_on_every_pipeline(slabs, cps, shape):
    """Every ring shape, ragged rows and columns (K/R not a
    multiple of a stage): packed == row-major bitwise; the integer case
    equals the oracle."""
    R, N, Kr, B = shape
    opts = ((csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN), (csg.SYMM_OPT_SK_SLABS, slabs),
            (csg.SYMM_OPT_SK_CTAS_PER_SM, cps))
    for kind in ("int", "normal"):
        if kind == "int":
            W, x = _int_case(R, N, Kr, B, seed=N + slabs)
        else:
            W, x = synth.gemv_inputs(R, N, R * Kr, B, N + 7 * slabs, 0.02, "normal")
        y_pk = _run(W, x, True, opts)
        y_rm = _run(W, x, False, opts)
        assert np.array_equal(y_pk, y_rm)
        check_gemv(W, x, y_pk, exact=(kind == "int"))


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_packed_with_k_splits_and_reversed_order(splits):
    """K splits (more, smaller units) and reversed unit order on packed
    weights; the row-major call runs the same kernel and plan."""
    R, N, Kr, B = 4, 513, 1032, 2
    W, x = synth.gemv_inputs(R, N, R * Kr, B, 40 + splits, 0.02, "normal")
    opts = ((csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN), (csg.SYMM_OPT_DYN_SPLITS, splits))
    y_pk = _run(W, x, True, opts)
    assert np.array_equal(y_pk, _run(W, x, True, opts, order=1))
    assert np.array_equal(y_pk, _run(W, x, False, opts))
    check_gemv(W, x, y_pk)


def test_packed_reduce_scatter_and_bias_rmsnorm_forms():
    R, N, Kr, B = 4, 1024, 520, 8
    W, x = synth.gemv_inputs(R, N, R * Kr, B, 77, 0.02, "normal")
    rs_pk = _run(W, x, True, mode="reduce_scatter")
    assert np.array_equal(rs_pk, _run(W, x, False, mode="reduce_scatter"))
    y_ref, want = oracle.gemv_reduce_scatter(W, x)
    for s in range(R):
        assert tolerance_ratio(words_to_f64(rs_pk[s]), y_ref[s * (B // R):(s + 1) * (B // R)]) <= 1.0
    bias, gamma = synth.norm_vectors(N, 5)
    z_pk = _run(W, x, True, mode="bias_rmsnorm", vectors=(bias, gamma))
    assert np.array_equal(z_pk, _run(W, x, False, mode="bias_rmsnorm", vectors=(bias, gamma)))
    z_ref, z_or = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6)
    assert tolerance_ratio(words_to_f64(z_pk[0]), z_ref) <= 1.0


@pytest.mark.parametrize("name", ["attn_out_proj", "mlp_down_decode", "mlp_down_large"])
def test_packed_full_size_workload(name):
    """The benchmark's GEMV workloads with packed weights, every output
    against the fp64 oracle and bitwise equal to the row-major call."""
    W, x = synth.workload_inputs(name)
    y_pk = _run(W, x, True)
    y_ref, y_or = oracle.gemv_all_reduce(W, x)
    R = W.shape[0]
    for s in range(1, R):
        assert np.array_equal(y_pk[s], y_pk[0])
    assert tolerance_ratio(words_to_f64(y_pk[0]), y_ref) <= 1.0
    big = np.abs(y_ref) >= 0.1 * np.sqrt(np.mean(y_ref ** 2))
    assert float(np.mean(y_pk[0] == y_or[0])) >= 0.99
    assert int(ulp_distance(y_pk[0][big], y_or[0][big]).max()) <= 1
    assert np.array_equal(y_pk, _run(W, x, False))


def test_registration_rules():
    R, N, Kr, B = 2, 256, 128, 2
    K = R * Kr
    W, x = _int_case(R, N, Kr, B, seed=3)
    ws = GemvWorkspace(R, N, K, B, copies=2, packed=True)
    s = torch.cuda.current_stream()
    try:
        ws.load_W(W)
        ws.load_x(x)
        Wp = ws.W_ptr(0)
        for n_, k_ in ((N - 128, K), (N, K - 2 * 64)):   # another shape on the packed weight
            with pytest.raises(csg.SymmError) as e:
                csg.gemv_all_reduce(ws.h, Wp, ws.x_ptr(), ws.y_ptr(), R, n_, k_, B, s)
            assert e.value.code == csg.SYMM_EINVAL
        for path in (csg.GEMV_PATH_FFMA,):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
            with pytest.raises(csg.SymmError) as e:
                csg.gemv_all_reduce(ws.h, Wp, ws.x_ptr(), ws.y_ptr(), R, N, K, B, s)
            assert e.value.code == csg.SYMM_EINVAL
            csg.gemv_all_reduce(ws.h, ws.W_rowmajor_ptr(), ws.x_ptr(), ws.y_ptr(), R, N, K, B, s)   # row-major: fine
        for path in (csg.GEMV_PATH_DYN, csg.GEMV_PATH_AUTO):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
            ws.fill_y(0xFF)
            csg.gemv_all_reduce(ws.h, Wp, ws.x_ptr(), ws.y_ptr(), R, N, K, B, s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            check_gemv(W, x, ws.read_y(), exact=True)
        # packing a packed weight, or into an overlapping range, is rejected
        with pytest.raises(csg.SymmError) as e:
            csg.symm_pack_w(ws.h, Wp, ws.W_ptr(1), R, N, K, s)
        assert e.value.code == csg.SYMM_EINVAL
        with pytest.raises(csg.SymmError) as e:
            csg.symm_pack_w(ws.h, ws.W_rowmajor_ptr(), ws.W_rowmajor_ptr() + 256, R, N, K, s)
        assert e.value.code == csg.SYMM_EINVAL
        with pytest.raises(csg.SymmError) as e:   # Wp past the user region
            csg.symm_pack_w(ws.h, ws.W_rowmajor_ptr(), ws.base + ws.slot_bytes - 16, R, N, K, s)
        assert e.value.code == csg.SYMM_EINVAL
        # a pack over part of copy 0 ends copy 0's registration
        csg.symm_pack_w(ws.h, ws.W_rowmajor_ptr(), Wp + 16384, R, N, K, s)
        csg.gemv_all_reduce(ws.h, Wp, ws.x_ptr(), ws.y_ptr(), R, N - 128, K, B, s)   # read row-major now
        with pytest.raises(csg.SymmError):
            csg.symm_release_w(ws.h, Wp)
        csg.symm_release_w(ws.h, Wp + 16384)
        with pytest.raises(csg.SymmError) as e:
            csg.symm_release_w(ws.h, Wp + 16384)
        assert e.value.code == csg.SYMM_EINVAL
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


def test_repacking_new_weights_before_each_chained_call():
    """New weights packed into the same Wp right before each call (chaining
    on): each call reads the weights packed just before it."""
    R, N, Kr, B = 8, 512, 512, 1
    ws = GemvWorkspace(R, N, R * Kr, B, packed=True)
    s = torch.cuda.current_stream()
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_CHAIN, 1)
        x = None
        for i in range(4):
            W, x_i = _int_case(R, N, Kr, B, seed=100 + i)
            if x is None:
                x = x_i
                ws.load_x(x)
            ws.load_W(W)                       # staging copy + symm_pack_w on the stream
            ws.fill_y(0xFF)
            ws.run(s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            check_gemv(W, x, ws.read_y(), exact=True)
    finally:
        ws.close()


def test_packed_call_in_a_cuda_graph():
    R, N, Kr, B = 4, 1000, 1024, 3
    W, x = _int_case(R, N, Kr, B, seed=9)
    ws = GemvWorkspace(R, N, R * Kr, B, packed=True)
    try:
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        ws.run(s)                                  # eager first: plans and tensor maps exist
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ws.run(torch.cuda.current_stream())
        for _ in range(3):
            ws.fill_y(0xFF)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            check_gemv(W, x, ws.read_y(), exact=True)
        del g
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
    finally:
        ws.close()


def test_packed_k_zero_and_empty_shapes():
    R, N, B = 2, 100, 2
    ws = GemvWorkspace(R, N, 0, B, packed=True)
    s = torch.cuda.current_stream()
    try:
        ws.load_W(np.zeros((R, N, 0), dtype=np.uint16))   # only the zero block
        ws.fill_y(0xFF)
        csg.gemv_all_reduce(ws.h, ws.W_ptr(0), ws.x_ptr(), ws.y_ptr(), R, N, 0, B, s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        assert not ws.read_y().any()           # +0 everywhere
        csg.gemv_all_reduce(ws.h, ws.W_ptr(0), ws.x_ptr(), ws.y_ptr(), R, N, 0, 0, s)   # B = 0: no-op
    finally:
        ws.close()
