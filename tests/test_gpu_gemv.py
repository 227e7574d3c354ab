"""Fused GEMV + one-shot all-reduce on the GPU, through the C ABI, against the
CPU oracle: exact cases bit-for-bit, random cases within
|y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(y_ref), replicas bit-identical, runs and
CTA orders bit-identical, guard bands intact, bad arguments rejected without a
launch, protocol faults reported (never waited on)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300 import DeviceView
from collective_split_gemv_gb300.workspace import GemvWorkspace
from gpu_common import check_gemv, require_gpu, run_gemv
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu

PATHS = [csg.GEMV_PATH_AUTO, csg.GEMV_PATH_FFMA, csg.GEMV_PATH_DYN]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _int_case(R, N, Kr, B, seed):
    rng = np.random.default_rng(seed)
    W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
    x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    return W, x


def _normal_case(R, N, K, B, seed, w_std=0.02):
    return synth.gemv_inputs(R, N, K, B, seed, w_std, "normal")


# Small-integer inputs: every product and partial sum is an integer below
# 2^24, so fp32 accumulation is exact in any order and the GPU must equal the
# oracle bit for bit.  Shapes cover ragged row tiles, K/R not a multiple of a
# warp's 32 x 16-byte stride, every batch class and non-power-of-two R.
INT_CASES = [(1, 1, 8, 1), (2, 3, 16, 2), (4, 17, 24, 5), (2, 33, 8, 16), (8, 40, 64, 3),
             (3, 100, 256, 4), (4, 129, 520, 7), (2, 250, 1032, 1), (5, 31, 2056, 8),
             (8, 300, 264, 12), (2, 16, 4096, 16)]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", INT_CASES, ids=[f"R{c[0]}N{c[1]}Kr{c[2]}B{c[3]}" for c in INT_CASES])
def test_integer_inputs_bit_exact(path, case):
    R, N, Kr, B = case
    W, x = _int_case(R, N, Kr, B, seed=sum(case))
    (y,), status = run_gemv(W, x, path=path)
    assert status[0] == csg.SYMM_OK, status
    check_gemv(W, x, y, exact=True)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_workload(path):
    W, x = synth.workload_inputs("tiny")
    outs, status = run_gemv(W, x, path=path, repeat=2)
    assert status[0] == csg.SYMM_OK
    ratio, eq, ulp = check_gemv(W, x, outs[0])
    assert np.array_equal(outs[0], outs[1]), "second run differs"
    assert eq >= 0.99 and ulp <= 1, (eq, ulp)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("B", list(range(1, 17)))
def test_every_batch_width(path, B):
    # N = 77 rows: ragged last tile; K/R = 264: 33 16-byte chunks per row.
    W, x = _normal_case(4, 77, 4 * 264, B, seed=100 + B)
    (y,), status = run_gemv(W, x, path=path)
    assert status[0] == csg.SYMM_OK
    check_gemv(W, x, y)


def test_x_staged_in_several_passes():
    # B = 16 and K/R = 1600: x_r does not fit one shared-memory pass.
    W, x = _normal_case(2, 40, 3200, 16, seed=5)
    (y,), status = run_gemv(W, x, path=csg.GEMV_PATH_FFMA)
    assert status[0] == csg.SYMM_OK
    check_gemv(W, x, y)


@pytest.mark.parametrize("path", PATHS)
def test_cta_order_does_not_change_bits(path):
    W, x = _normal_case(8, 1000, 8 * 512, 3, seed=9)
    (y0,), _ = run_gemv(W, x, path=path, order=0)
    (y1,), st = run_gemv(W, x, path=path, order=1)
    assert st[0] == csg.SYMM_OK
    assert np.array_equal(y0, y1)
    check_gemv(W, x, y0)


def test_one_hot_passes_column_through():
    R, N, K = 4, 300, 4 * 128
    W = synth.normal(5, synth.TAG_W, N, K, std=0.5, shards=R)
    Wg = W.transpose(1, 0, 2).reshape(N, K)
    for k in (0, 129, 511):
        xg = np.zeros((1, K))
        xg[0, k] = 1.0
        x = synth.shard_columns(f64_to_words_via_f32(xg), R)
        (y,), _ = run_gemv(W, x)
        assert np.array_equal(words_to_f64(y[0, 0]), words_to_f64(Wg[:, k])), k


def test_power_of_two_scaling_is_exact():
    W, x = _normal_case(4, 200, 4 * 256, 2, seed=13)
    x4 = f64_to_words_via_f32(words_to_f64(x) * 4.0)
    (y,), _ = run_gemv(W, x)
    (y4,), _ = run_gemv(W, x4)
    assert np.array_equal(words_to_f64(y4), 4.0 * words_to_f64(y))


def test_k_zero_writes_positive_zero():
    W = np.zeros((2, 50, 0), dtype=np.uint16)
    x = np.zeros((2, 3, 0), dtype=np.uint16)
    (y,), status = run_gemv(W, x, y_fill=0xFF)
    assert status[0] == csg.SYMM_OK
    assert np.all(y == 0)


def test_empty_calls_are_no_ops():
    ws = GemvWorkspace(2, 64, 128, 2)
    try:
        ws.fill_y(0xAB)
        s = torch.cuda.current_stream()
        csg.gemv_all_reduce(ws.h, ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), 2, 0, 128, 2, s)
        csg.gemv_all_reduce(ws.h, ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), 2, 64, 128, 0, s)
        assert np.all(ws.read_y() == 0xABAB)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
    finally:
        ws.close()


@pytest.mark.parametrize("R,N,Kr,B", [(1, 513, 512, 1), (64, 40, 8, 2), (3, 65, 136, 5),
                                      (2, 100000, 8, 1), (8, 7, 8, 16)])
def test_rank_counts_and_shapes(R, N, Kr, B):
    W, x = _normal_case(R, N, R * Kr, B, seed=R * 1000 + N)
    (y,), status = run_gemv(W, x)
    assert status[0] == csg.SYMM_OK
    check_gemv(W, x, y)


@pytest.mark.parametrize("name", ["tiny", "attn_out_proj", "mlp_down_decode", "mlp_down_large"])
def test_full_size_workload(name):
    """The benchmark's workloads at full size, every output against the fp64
    oracle; second run and reversed CTA order bit-identical, and so is the
    persistent kernel's other ending (drawn units with the global-memory
    protocol where the plan takes the cluster epilogue), in reversed order."""
    W, x = synth.workload_inputs(name)
    y_ref, y_or = oracle.gemv_all_reduce(W, x)
    outs, status = run_gemv(W, x, repeat=2)
    assert status[0] == csg.SYMM_OK
    R = W.shape[0]
    for s in range(1, R):
        assert np.array_equal(outs[0][s], outs[0][0])
    assert np.array_equal(outs[0], outs[1])
    ratio = tolerance_ratio(words_to_f64(outs[0][0]), y_ref)
    eq = float(np.mean(outs[0][0] == y_or[0]))
    # Away from zero the fp32 sum is within half a bf16 step of the fp64 one,
    # so the rounded results differ by at most one step; near zero the fp32
    # rounding error of a long sum can exceed a (tiny) bf16 step there.
    big = np.abs(y_ref) >= 0.1 * np.sqrt(np.mean(y_ref ** 2))
    ulp_all = int(ulp_distance(outs[0][0], y_or[0]).max())
    ulp_big = int(ulp_distance(outs[0][0][big], y_or[0][big]).max())
    print(f"{name}: tolerance ratio {ratio:.3f}, bit-equal {eq:.5f}, max ulp {ulp_all} "
          f"({ulp_big} where |y| >= 0.1 rms)")
    assert ratio <= 1.0
    assert eq >= 0.99 and ulp_big <= 1
    (y_rev,), _ = run_gemv(W, x, order=1)
    assert np.array_equal(y_rev, outs[0])
    (y_drawn,), st = run_gemv(W, x, order=1, options=((csg.SYMM_OPT_DYN_CLUSTER, 0),))
    assert st[0] == csg.SYMM_OK
    assert np.array_equal(y_drawn, outs[0])


# --------------------------------------------------------------- arguments


def test_bad_arguments_are_rejected_without_launch():
    R, N, K, B = 2, 64, 128, 2
    ws = GemvWorkspace(R, N, K, B)
    try:
        ws.fill_y(0xAB)
        s = torch.cuda.current_stream()
        W, x, y = ws.W_ptr(), ws.x_ptr(), ws.y_ptr()
        bad = [
            ((W, x, y, 3, N, K, B), csg.SYMM_EINVAL),          # R mismatch
            ((W, x, y, R, N, 130, B), csg.SYMM_EINVAL),        # K % R
            ((W, x, y, R, N, 2 * 12, B), csg.SYMM_EINVAL),     # K/R % 8
            ((W, x, y, R, N, K, 17), csg.SYMM_EINVAL),         # B > 16
            ((W, x, y, R, -1, K, B), csg.SYMM_EINVAL),         # N < 0
            ((W + 2, x, y, R, N, K, B), csg.SYMM_EINVAL),      # misaligned W
            ((W, x + 8, y, R, N, K, B), csg.SYMM_EINVAL),      # misaligned x
            ((W, x, W, R, N, K, B), csg.SYMM_EINVAL),          # y overlaps W
            ((W, x, x, R, N, K, B), csg.SYMM_EINVAL),          # y overlaps x
            ((ws.slots[1], x, y, R, N, K, B), csg.SYMM_EINVAL),  # not a slot-0 address
            ((W + ws.slot_bytes, x, y, R, N, K, B), csg.SYMM_EINVAL),  # past the user region
            ((W, x, y, R, 4 * N, K, B), csg.SYMM_EINVAL),      # W/y extent past the region
        ]
        for args, code in bad:
            with pytest.raises(csg.SymmError) as e:
                csg.gemv_all_reduce(ws.h, *args, s)
            assert e.value.code == code, args
        assert np.all(ws.read_y() == 0xABAB)
        assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
    finally:
        ws.close()


def test_retired_kernels_and_engine_are_refused():
    """Paths 2 and 3 and the persistent kernel's CUDA-core engine were
    retired (none won on any shape measured): asking for them is an error,
    not a silent substitute."""
    ws = GemvWorkspace(2, 64, 128, 1)
    try:
        for opt, val in ((csg.SYMM_OPT_GEMV_PATH, 2), (csg.SYMM_OPT_GEMV_PATH, 3), (csg.SYMM_OPT_SK_ENGINE, 1)):
            with pytest.raises(csg.SymmError) as e:
                csg.symm_set_option(ws.h, opt, val)
            assert e.value.code == csg.SYMM_EINVAL and "retired" in str(e.value)
        for val in (-1, 0):
            csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_ENGINE, val)
    finally:
        ws.close()


def test_capacity_errors():
    # scratch too small for B*N fp32 partials
    h = csg.symm_alloc(2, 1 << 20, 256, 4096)
    try:
        base = csg.symm_rendezvous(h)[0][0]
        with pytest.raises(csg.SymmError) as e:
            csg.gemv_all_reduce(h, base, base + 65536, base + 131072, 2, 128, 16, 1)
        assert e.value.code == csg.SYMM_ERANGE
    finally:
        csg.symm_free(h)
    # more row tiles than the signal pad holds (scratch is ample here)
    h = csg.symm_alloc(2, 1 << 20, 1 << 20, 4096)
    try:
        base = csg.symm_rendezvous(h)[0][0]
        tiles = csg.symm_info(h)["max_tiles"]
        rows = csg.symm_gemv_plan(h, 16, 0, 1)["rows_per_tile"]   # K = 0: CUDA-core kernel
        N = (tiles + 1) * rows
        with pytest.raises(csg.SymmError) as e:
            csg.gemv_all_reduce(h, base, base + 65536, base + 131072, 2, N, 0, 1)
        assert e.value.code == csg.SYMM_ERANGE
        assert csg.symm_check_guards(h)[0] == csg.SYMM_OK
    finally:
        csg.symm_free(h)


# ---------------------------------------------------------------- protocol


def _counter_view(ws, tile):
    info = csg.symm_info(ws.h)
    counters_off = 128 + -(-4 * info["max_tiles"] // 128) * 128
    return torch.as_tensor(DeviceView(ws.pads[0] + counters_off + 4 * tile, (1,), "<i4"),
                           device=ws.device)


def test_corrupted_counter_is_reported_and_recovered():
    """A tile counter left in a wrong state (as an overlapping launch on
    another stream would leave it) is detected by the kernel and reported by
    symm_status; no CTA waits on it.  The handle then works again."""
    R, N, K, B = 4, 64, 4 * 64, 1
    W, x = _normal_case(R, N, K, B, seed=3)
    y_ref, y_or = oracle.gemv_all_reduce(W, x)
    ws = GemvWorkspace(R, N, K, B)
    try:
        # the per-tile kernel of the global-memory protocol (the automatic
        # choice for so small a layer is the cluster kernel, which keeps no
        # state in the pad)
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_FFMA)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        y1 = ws.read_y()
        cnt = _counter_view(ws, 0)
        assert int(cnt.item()) == 0               # tile 0's reducer put its counter back to zero
        cnt.fill_(R - 1)                          # pretend R-1 arrivals of launch 2 happened
        ws.fill_y(0xFF)
        ws.run(s)
        code, rank, tile = csg.symm_status(ws.h, s)
        assert code == csg.SYMM_EPROTO and tile == 0, (code, rank, tile)
        y = ws.read_y()
        rows = csg.symm_gemv_plan(ws.h, N, K, B)["rows_per_tile"]
        # Tile 0's first arriver holds the "last" ticket.  It stores nothing
        # if some peer's flag is still stale; if every peer had already
        # published (flags are set before tickets are taken) its sum is the
        # correct one.  Either way nothing else changes.
        t0 = y[:, :, :rows]
        assert np.all(t0 == 0xFFFF) or np.array_equal(t0, y1[:, :, :rows])
        assert np.array_equal(y[:, :, rows:], y1[:, :, rows:])  # other tiles unaffected
        ws.run(s)                                 # the handle recovered
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


@pytest.mark.parametrize("path", PATHS)
def test_shape_changes_on_one_handle(path):
    """One handle, calls of different N and B (hence different tile counts and
    K-splits) in a row: the signal pad's tickets stay consistent."""
    R, N, K, B = 4, 700, 4 * 256, 8
    W, x = _normal_case(R, N, K, B, seed=23)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        for n_rows, b in ((700, 8), (100, 8), (700, 3), (5, 16 if B >= 16 else 8), (700, 8)):
            ws.fill_y(0xFF)
            csg.gemv_all_reduce(ws.h, ws.W_ptr(), ws.x_ptr(), ws.y_ptr(), R, n_rows, K, b, s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK, (n_rows, b)
            y = ws.read_y().reshape(R, -1)[:, : b * n_rows].reshape(R, b, n_rows)
            # the sub-problem: first n_rows rows of W, x rows 0..b-1 laid out
            # with row stride K/R (x is [B][K/R], so rows 0..b-1 are a prefix)
            check_gemv(np.ascontiguousarray(W[:, :n_rows]), np.ascontiguousarray(x[:, :b]), y)
    finally:
        ws.close()


@pytest.mark.parametrize("path", [csg.GEMV_PATH_FFMA, csg.GEMV_PATH_DYN])
def test_many_launches_leave_the_pad_consistent(path):
    R, N, K, B = 8, 1000, 8 * 512, 2
    W, x = _normal_case(R, N, K, B, seed=17)
    ws = GemvWorkspace(R, N, K, B)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
        ws.load_W(W)
        ws.load_x(x)
        s = torch.cuda.current_stream()
        for _ in range(50):
            ws.run(s)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        # each launch's reducer puts the tile counters back to zero; the
        # launch epoch in slot 0's pad counts the launches
        tiles = csg.symm_gemv_plan(ws.h, N, K, B)["tiles"]
        assert all(int(_counter_view(ws, t).item()) == 0 for t in range(tiles))
        epoch = torch.as_tensor(DeviceView(ws.pads[0] + 96, (1,), "<i4"), device=ws.device)
        assert int(epoch.item()) == 50
        check_gemv(W, x, ws.read_y())
    finally:
        ws.close()


# ------------------------------------------- persistent-kernel variants

SK_PIPES = [(1, 1), (2, 1), (4, 1), (1, 2), (2, 2), (3, 2), (1, 3)]   # (slabs, CTAs per SM)
SK_VARIANTS = [(slabs, cps) for slabs, cps in SK_PIPES]
SK_SHAPES = [(8, 300, 8 * 264, 2), (4, 1000, 4 * 2056, 2), (2, 17, 2 * 8, 1), (3, 513, 3 * 4096, 2),
             (8, 2048, 8 * 512, 1)]


@pytest.mark.parametrize("path", [csg.GEMV_PATH_DYN], ids=["persistent"])
@pytest.mark.parametrize("slabs,cps", SK_VARIANTS, ids=[f"slabs{s}-cps{c}" for s, c in SK_VARIANTS])
@pytest.mark.parametrize("shape", SK_SHAPES, ids=[f"R{a}N{b}K{c}B{d}" for a, b, c, d in SK_SHAPES])
def test_tma_kernels_pipelines(path, slabs, cps, shape):
    """The persistent TMA kernel, every pipeline shape: integer inputs bit-exact, normal inputs within tolerance,
    replicas identical, reversed CTA / unit order identical."""
    R, N, K, B = shape
    for kind in ("int", "normal"):
        if kind == "int":
            W, x = _int_case(R, N, K // R, B, seed=N + slabs)
        else:
            W, x = _normal_case(R, N, K, B, seed=N + 7 * slabs)
        ws = GemvWorkspace(R, N, K, B)
        try:
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
            csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_SLABS, slabs)
            csg.symm_set_option(ws.h, csg.SYMM_OPT_SK_CTAS_PER_SM, cps)
            plan = csg.symm_gemv_plan(ws.h, N, K, B)
            assert plan["path"] == path and plan["engine"] == 0 and plan["slabs"] == slabs
            assert plan["ctas_per_sm"] == cps
            ws.load_W(W)
            ws.load_x(x)
            s = torch.cuda.current_stream()
            ws.fill_y(0xFF)
            ws.run(s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            y0 = ws.read_y()
            csg.symm_set_option(ws.h, csg.SYMM_OPT_TILE_ORDER, 1)
            ws.fill_y(0xFF)
            ws.run(s)
            assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            assert np.array_equal(ws.read_y(), y0), "reversed CTA order changed bits"
            assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        finally:
            ws.close()
        check_gemv(W, x, y0, exact=(kind == "int"))


@pytest.mark.parametrize("splits", [2, 3, 5])
@pytest.mark.parametrize("shape", [(8, 300, 8 * 1032, 2), (4, 513, 4 * 4096, 1), (2, 130, 2 * 520, 2)],
                         ids=["R8N300", "R4N513", "R2N130"])
def test_persistent_kernel_k_splits(splits, shape):
    """The persistent kernel with every (tile, rank) cut into K splits: more,
    smaller units for the work counter; integer inputs stay bit-exact."""
    R, N, K, B = shape
    for kind in ("int", "normal"):
        W, x = (_int_case(R, N, K // R, B, seed=splits + N) if kind == "int"
                else _normal_case(R, N, K, B, seed=3 * splits + N))
        ws = GemvWorkspace(R, N, K, B)
        try:
            csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
            csg.symm_set_option(ws.h, csg.SYMM_OPT_DYN_SPLITS, splits)
            plan = csg.symm_gemv_plan(ws.h, N, K, B)
            assert plan["splits"] > 1
            ws.load_W(W)
            ws.load_x(x)
            s = torch.cuda.current_stream()
            for _ in range(2):
                ws.fill_y(0xFF)
                ws.run(s)
                assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
            y = ws.read_y()
            assert csg.symm_check_guards(ws.h)[0] == csg.SYMM_OK
        finally:
            ws.close()
        check_gemv(W, x, y, exact=(kind == "int"))
