"""The further collectives on the GPU, through the C ABI, against the CPU
oracle: reduce-scatter, two-shot all-reduce, 2-D tile reduce to one or
several roots, all-reduce + bias + RMSNorm.  Integer inputs bit-exact;
random inputs within |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(y_ref); replicas
and repeated runs bit-identical; bad arguments rejected; guard bands intact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import AllReduceWorkspace, RmsNormWorkspace, TileWorkspace
from gpu_common import require_gpu
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _guards_ok(h):
    rc, bad_rank, band = csg.symm_check_guards(h)
    assert rc == csg.SYMM_OK, f"guard band {band} of rank {bad_rank} overwritten"


def _int_words(rng, shape, lo=-100, hi=100):
    return f64_to_words_via_f32(rng.integers(lo, hi + 1, size=shape).astype(np.float64))


def _run_ar(inp, op, in_place=False, fill=0xFFFF, repeat=1):
    R, n = inp.shape
    aw = AllReduceWorkspace(R, n, separate_out=not in_place)
    try:
        outs = []
        for _ in range(repeat):
            aw.load_in(inp)
            if not in_place:
                for r in range(R):
                    aw.out_view(r).fill_(fill & 0xFF)
            aw.run(torch.cuda.current_stream(), op=op)
            outs.append(aw.read_out(count=n // R if op == "reduce_scatter" else n))
        _guards_ok(aw.h)
        return outs if repeat > 1 else outs[0]
    finally:
        aw.close()


# ------------------------------------------------------------ reduce-scatter


@pytest.mark.parametrize("R,n", [(1, 8), (2, 16), (4, 36), (8, 64 * 1000), (3, 3 * 17), (8, 8 * 4099),
                                 (64, 64 * 8), (5, 5)])
def test_reduce_scatter_integers_bit_exact(R, n):
    inp = _int_words(np.random.default_rng(R * 31 + n), (R, n))
    _, want = oracle.reduce_scatter(inp)
    out = _run_ar(inp, "reduce_scatter")
    assert np.array_equal(out, want)


def test_reduce_scatter_full_size():
    inp = synth.workload_inputs("allreduce")
    ref, want = oracle.reduce_scatter(inp)
    outs = _run_ar(inp, "reduce_scatter", repeat=2)
    R, n = inp.shape
    got = outs[0].reshape(-1)
    assert tolerance_ratio(words_to_f64(got), ref) <= 1.0
    assert float(np.mean(got == want.reshape(-1))) >= 0.999
    assert int(ulp_distance(got, want.reshape(-1)).max()) <= 1
    assert np.array_equal(outs[0], outs[1])
    # the blocks are exactly the one-shot all-reduce's elements
    one = _run_ar(inp, "one_shot")
    assert np.array_equal(got, one[0])


def test_reduce_scatter_bad_arguments():
    aw = AllReduceWorkspace(4, 64)
    try:
        s = torch.cuda.current_stream()
        csg.reduce_scatter(aw.h, aw.base, aw.base + aw.out_off, 4, 0, s)          # no-op
        for args in ((aw.base, aw.base + aw.out_off, 4, 62),                     # n % R
                     (aw.base, aw.base + aw.out_off, 3, 63),                     # R mismatch
                     (aw.base, aw.base + 32, 4, 64),                             # out overlaps in
                     (aw.base + 2, aw.base + aw.out_off, 4, 32)):                # misaligned
            with pytest.raises(csg.SymmError) as e:
                csg.reduce_scatter(aw.h, *args, s)
            assert e.value.code == csg.SYMM_EINVAL, args
        _guards_ok(aw.h)
    finally:
        aw.close()


# ------------------------------------------------------------ two-shot


@pytest.mark.parametrize("R,n", [(1, 8), (2, 7), (3, 1003), (4, 1), (8, 5), (8, 100000), (16, 999), (64, 65)])
def test_two_shot_integers_bit_exact(R, n):
    inp = _int_words(np.random.default_rng(R * 17 + n), (R, n))
    _, want = oracle.one_shot_all_reduce(inp)
    assert np.array_equal(_run_ar(inp, "two_shot"), want)
    assert np.array_equal(_run_ar(inp, "two_shot", in_place=True), want)


def test_two_shot_full_size_matches_one_shot():
    inp = synth.workload_inputs("allreduce")
    ref, want = oracle.one_shot_all_reduce(inp)
    two = _run_ar(inp, "two_shot", repeat=2)
    one = _run_ar(inp, "one_shot")
    for s in range(1, inp.shape[0]):
        assert np.array_equal(two[0][s], two[0][0])
    assert np.array_equal(two[0], one), "two-shot differs from one-shot"
    assert np.array_equal(two[0], two[1])
    assert tolerance_ratio(words_to_f64(two[0][0]), ref) <= 1.0
    assert int(ulp_distance(two[0][0], want[0]).max()) <= 1
    inplace = _run_ar(inp, "two_shot", in_place=True)
    assert np.array_equal(inplace, one)


# ------------------------------------------------------------ tile reduce


def _tile_case(R, sr, sc, orows, ocols, tiles, roots, rows, cols, out_at, seed, integers=True):
    rng = np.random.default_rng(seed)
    if integers:
        full = _int_words(rng, (R, sr, sc), -60, 60)
    else:
        full = synth.tile_inputs(R, sr, sc, seed)
    before = rng.integers(0, 0x7F00, size=(R, orows, ocols)).astype(np.uint16)
    tw = TileWorkspace(R, sr, sc, orows, ocols)
    try:
        tw.load_in(full)
        tw.fill_out(before)
        tw.run(tiles, roots, rows, cols, out_at, torch.cuda.current_stream())
        got = tw.read_out()
        _guards_ok(tw.h)
    finally:
        tw.close()
    offs = [a * sc + b for a, b in tiles]
    oo = out_at[0] * ocols + out_at[1]
    ref, want = oracle.tile_reduce(full.reshape(R, -1), before.reshape(R, -1), offs, oo, roots, rows, cols, sc,
                                   ocols)
    return got.reshape(R, -1), want, ref, before.reshape(R, -1)


@pytest.mark.parametrize("case", [
    # R, slot rows x cols, out rows x cols, tiles, roots, tile rows x cols, out_at
    (4, 64, 64, 32, 32, [(0, 0), (0, 32), (32, 0), (32, 32)], [0, 1, 2, 3], 32, 32, (0, 0)),   # docs' quadrants
    (2, 9, 40, 9, 40, [(2, 8)], [1], 5, 24, (3, 16)),                                         # 16-byte rows
    (3, 9, 7, 6, 9, [(2, 3)], [2], 5, 4, (1, 2)),                                             # odd, scalar
    (8, 5, 48, 3, 20, [(1, 1), (0, 20), (3, 5)], [6, 0, 3], 2, 17, (1, 2)),                   # ragged cols
    (8, 300, 264, 130, 136, [(0, 0), (170, 128)], [7, 2], 130, 136, (0, 0)),                  # several CTAs
])
def test_tile_reduce_integers_bit_exact(case):
    R, sr, sc, orows, ocols, tiles, roots, rows, cols, out_at = case
    got, want, _, before = _tile_case(R, sr, sc, orows, ocols, tiles, roots, rows, cols, out_at, seed=sr * sc)
    assert np.array_equal(got, want)
    untouched = [r for r in range(R) if r not in roots]
    for r in untouched:
        assert np.array_equal(got[r], before[r]), f"rank {r} is no root but its output changed"


def test_multi_root_full_size():
    w = synth.WORKLOADS["multi_root_tile"]
    R, n = w["R"], w["rows"]
    h = n // 2
    tiles = [(0, 0), (0, h), (h, 0), (h, h)]
    got, want, ref, _ = _tile_case(R, n, n, h, h, tiles, [0, 1, 2, 3], h, h, (0, 0), seed=w["seed"], integers=False)
    for i, root in enumerate([0, 1, 2, 3]):
        assert tolerance_ratio(words_to_f64(got[root]), ref[i].reshape(-1)) <= 1.0
        assert int(ulp_distance(got[root], want[root]).max()) <= 1
        assert float(np.mean(got[root] == want[root])) >= 0.999


def test_tile_reduce_bad_arguments():
    tw = TileWorkspace(4, 16, 16, 8, 8)
    try:
        s = torch.cuda.current_stream()
        base_in = tw.base + tw.in_offs[0]
        out = tw.base + tw.out_offs[0]
        csg.tile_reduce(tw.h, base_in, out, 0, 0, 8, 16, 8, s)                      # rows = 0: no-op
        bad = [
            lambda: csg.multi_root_tile_reduce(tw.h, [base_in, base_in + 16], out, [1, 1], 4, 4, 16, 8, s),
            lambda: csg.tile_reduce(tw.h, base_in, out, 4, 4, 4, 16, 8, s),         # root out of range
            lambda: csg.tile_reduce(tw.h, base_in, out, 0, 4, 9, 16, 8, s),         # cols > ld_out
            lambda: csg.tile_reduce(tw.h, base_in, base_in + 64, 0, 4, 4, 16, 16, s),  # overlap
            lambda: csg.tile_reduce(tw.h, base_in + 1, out, 0, 4, 4, 16, 8, s),     # odd address
            lambda: csg.multi_root_tile_reduce(tw.h, [base_in] * 5, out, [0, 1, 2, 3, 4], 4, 4, 16, 8, s),
        ]
        for fn in bad:
            with pytest.raises(csg.SymmError) as e:
                fn()
            assert e.value.code == csg.SYMM_EINVAL
        _guards_ok(tw.h)
    finally:
        tw.close()


# -------------------------------------------------- all-reduce + bias + RMSNorm


def _run_norm(inp, bias, gamma, eps, in_place=False, repeat=1):
    R, rows, H = inp.shape
    nw = RmsNormWorkspace(R, rows, H, in_place=in_place)
    try:
        outs = []
        for _ in range(repeat):
            nw.load(inp, bias, gamma)
            nw.run(torch.cuda.current_stream(), eps=eps, bias=bias is not None, gamma=gamma is not None)
            outs.append(nw.read_out())
        _guards_ok(nw.h)
        return outs if repeat > 1 else outs[0]
    finally:
        nw.close()


def _check_norm(out, ref, want):
    R = out.shape[0]
    for s in range(1, R):
        assert np.array_equal(out[s], out[0]), f"replica {s} differs"
    ratio = tolerance_ratio(words_to_f64(out[0]), ref)
    assert ratio <= 1.0, ratio
    # at most one rounding step from the oracle's bf16 wherever the value is
    # not tiny next to the row's scale (near zero, fp32 sums of large, partly
    # cancelling terms legitimately differ from the fp64 sum by many steps)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    big = np.abs(ref) >= 0.1 * rms
    assert int(ulp_distance(out[0][big], want[0][big]).max(initial=0)) <= 1
    return float(np.mean(out[0] == want[0]))


@pytest.mark.parametrize("R,rows,H,eps,use_bias,use_gamma", [
    (8, 1, 8192, 1e-6, True, True),      # decode-sized message (16 KB per rank)
    (4, 16, 4096, 1e-5, True, True),
    (2, 3, 8, 0.0, False, False),
    (3, 5, 8 * 1001, 1e-3, True, False),  # ragged: the last CTA of the cluster gets fewer vectors
    (8, 2, 65536, 1e-6, False, True),    # largest H: eight vectors per thread
    (1, 1, 1024, 0.5, True, True),
    (64, 2, 256, 1e-6, True, True),
])
def test_all_reduce_bias_rmsnorm(R, rows, H, eps, use_bias, use_gamma):
    inp, bias, gamma = synth.rmsnorm_inputs(R, rows, H, seed=R + rows + H)
    bias = bias if use_bias else None
    gamma = gamma if use_gamma else None
    ref, want = oracle.all_reduce_bias_rmsnorm(inp, bias, gamma, eps)
    outs = _run_norm(inp, bias, gamma, eps, repeat=2)
    eq = _check_norm(outs[0], ref, want)
    assert eq >= 0.99
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(_run_norm(inp, bias, gamma, eps, in_place=True), outs[0])


def test_all_reduce_bias_rmsnorm_workload():
    w = synth.WORKLOADS["ar_bias_rmsnorm"]
    inp, bias, gamma = synth.workload_inputs("ar_bias_rmsnorm")
    ref, want = oracle.all_reduce_bias_rmsnorm(inp, bias, gamma, w["eps"])
    eq = _check_norm(_run_norm(inp, bias, gamma, w["eps"]), ref, want)
    print(f"ar_bias_rmsnorm: bit-equal {eq:.5f}")


def test_all_reduce_bias_rmsnorm_bad_arguments():
    nw = RmsNormWorkspace(2, 4, 64)
    try:
        s = torch.cuda.current_stream()
        i0, o0 = nw.base + nw.in_offs[0], nw.base + nw.out_offs[0]
        csg.all_reduce_bias_rmsnorm(nw.h, i0, None, None, o0, 2, 0, 64, 1e-6, s)     # rows = 0: no-op
        bad = [
            (i0, None, None, o0, 2, 4, 60, 1e-6),            # H % 8
            (i0, None, None, o0, 2, 4, 0, 1e-6),
            (i0, None, None, o0, 3, 4, 64, 1e-6),            # R mismatch
            (i0, None, None, o0, 2, 4, 64, -1.0),            # eps < 0
            (i0, None, None, o0, 2, 4, 64, float("nan")),
            (i0, None, None, i0 + 16, 2, 4, 64, 1e-6),       # partial overlap
            (i0, o0, None, o0, 2, 4, 64, 1e-6),              # bias overlaps out
            (i0, nw.base + nw.bias_off + 2, None, o0, 2, 4, 64, 1e-6),   # misaligned bias
            (i0, None, None, o0, 2, 4, 1 << 17, 1e-6),       # H too large
        ]
        for args in bad:
            with pytest.raises(csg.SymmError) as e:
                csg.all_reduce_bias_rmsnorm(nw.h, *args, s)
            assert e.value.code == csg.SYMM_EINVAL, args
        _guards_ok(nw.h)
    finally:
        nw.close()


# ------------------------------------- the fused layer's other two endings

PATHS = [csg.GEMV_PATH_AUTO, csg.GEMV_PATH_FFMA, csg.GEMV_PATH_DYN]


def _gemv_ws(W, x, path):
    from collective_split_gemv_gb300.workspace import GemvWorkspace
    R, N, Kr = W.shape
    ws = GemvWorkspace(R, N, R * Kr, x.shape[1])
    csg.symm_set_option(ws.h, csg.SYMM_OPT_GEMV_PATH, path)
    ws.load_W(W)
    ws.load_x(x)
    return ws


def _run_mode(W, x, path, mode, bias=None, gamma=None, eps=1e-6, pdl=1):
    ws = _gemv_ws(W, x, path)
    try:
        csg.symm_set_option(ws.h, csg.SYMM_OPT_NORM_PDL, pdl)
        ws.load_vectors(bias, gamma)
        ws.fill_y(0xFF)
        s = torch.cuda.current_stream()
        ws.run(s, mode=mode, eps=eps, bias=bias is not None, gamma=gamma is not None)
        assert csg.symm_status(ws.h, s)[0] == csg.SYMM_OK
        out = ws.read_y_rs() if mode == "reduce_scatter" else ws.read_y()
        # the all-reduce form on the same handle, for comparison
        ws.run(s, mode="all_reduce")
        full = ws.read_y()
        _guards_ok(ws.h)
        return out, full
    finally:
        ws.close()


def _int_gemv(R, N, Kr, B, seed):
    rng = np.random.default_rng(seed)
    return (f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64)),
            f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64)))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("R,N,Kr,B", [(2, 300, 64, 2), (4, 129, 128, 8), (8, 1000, 256, 16), (1, 64, 8, 3)])
def test_gemv_reduce_scatter_integers(path, R, N, Kr, B):
    W, x = _int_gemv(R, N, Kr, B, seed=R * N + B)
    _, want = oracle.gemv_reduce_scatter(W, x)
    out, full = _run_mode(W, x, path, "reduce_scatter")
    assert np.array_equal(out, want)
    Bs = B // R
    for s in range(R):
        assert np.array_equal(out[s], full[0][s * Bs:(s + 1) * Bs])


@pytest.mark.parametrize("name", ["attn_out_proj", "mlp_down_large_rs"])
def test_gemv_reduce_scatter_full_size(name):
    W, x = synth.workload_inputs(name)
    y_ref, want = oracle.gemv_reduce_scatter(W, x)
    out, full = _run_mode(W, x, csg.GEMV_PATH_AUTO, "reduce_scatter")
    R, B = W.shape[0], x.shape[1]
    Bs = B // R
    got = out.reshape(B, -1)
    assert tolerance_ratio(words_to_f64(got), y_ref) <= 1.0
    for s in range(R):
        assert np.array_equal(out[s], full[0][s * Bs:(s + 1) * Bs]), "rows differ from the all-reduce form"


def test_gemv_reduce_scatter_rejects_ragged_batch():
    W, x = _int_gemv(4, 64, 8, 6, 1)
    with pytest.raises(csg.SymmError) as e:
        _run_mode(W, x, csg.GEMV_PATH_AUTO, "reduce_scatter")
    assert e.value.code == csg.SYMM_EINVAL


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("R,N,K,B,use_bias,use_gamma", [
    (2, 256, 512, 1, True, True), (4, 1000, 2048, 3, True, False), (8, 8192, 8192, 2, False, True),
    (1, 64, 64, 16, True, True)])
def test_gemv_bias_rmsnorm(path, R, N, K, B, use_bias, use_gamma):
    W, x = synth.gemv_inputs(R, N, K, B, seed=N + B, w_std=0.05)
    bias, gamma = synth.norm_vectors(N, seed=N)
    bias = bias if use_bias else None
    gamma = gamma if use_gamma else None
    y_ref, want = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-5)
    out, _ = _run_mode(W, x, path, "bias_rmsnorm", bias, gamma, 1e-5)
    _check_norm(out, y_ref, want)


@pytest.mark.parametrize("pdl", [1, 0])
def test_gemv_bias_rmsnorm_decode_full_size(pdl):
    w = synth.WORKLOADS["mlp_down_decode_rmsnorm"]
    W, x, bias, gamma = synth.workload_inputs("mlp_down_decode_rmsnorm")
    y_ref, want = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, w["eps"])
    out, _ = _run_mode(W, x, csg.GEMV_PATH_AUTO, "bias_rmsnorm", bias, gamma, w["eps"], pdl=pdl)
    eq = _check_norm(out, y_ref, want)
    print(f"mlp_down_decode_rmsnorm pdl={pdl}: bit-equal {eq:.5f}")


def test_gemv_bias_rmsnorm_large_batch():
    W, x = synth.workload_inputs("mlp_down_large")
    bias, gamma = synth.norm_vectors(W.shape[1], 4)
    y_ref, want = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6)
    out, _ = _run_mode(W, x, csg.GEMV_PATH_AUTO, "bias_rmsnorm", bias, gamma, 1e-6)
    _check_norm(out, y_ref, want)


def test_gemv_bias_rmsnorm_rejects_ragged_n():
    W, x = _int_gemv(2, 60, 8, 1, 2)
    with pytest.raises(csg.SymmError) as e:
        _run_mode(W, x, csg.GEMV_PATH_AUTO, "bias_rmsnorm")
    assert e.value.code == csg.SYMM_EINVAL


# ------------------------------------------------------- staging copies


@pytest.mark.parametrize("engine", [0, 1])
def test_copy_to_and_from_slots_round_trip(engine):
    # engine 0: pinned host memory copied by the SMs (a kernel); 1: the copy engine
    R, n = 4, 1000
    aw = AllReduceWorkspace(R, n)
    try:
        csg.symm_set_option(aw.h, csg.SYMM_OPT_COPY_ENGINE, engine)
        s = torch.cuda.current_stream()
        host = torch.arange(R * n, dtype=torch.int16).view(torch.uint8).pin_memory()
        csg.symm_copy_to_slots(aw.h, aw.base + aw.in_offs[0], host.data_ptr(), n * 2, R, s)
        s.synchronize()
        for r in range(R):
            got = aw.in_view(r).cpu().view(torch.int16)
            assert torch.equal(got, torch.arange(r * n, (r + 1) * n, dtype=torch.int16)), r
        back = torch.zeros(R * n * 2, dtype=torch.uint8).pin_memory()
        csg.symm_copy_from_slots(aw.h, back.data_ptr(), aw.base + aw.in_offs[0], n * 2, R, s)
        s.synchronize()
        assert torch.equal(back, host)
        # the result of a call read back from slot 0 only
        aw.run(s)
        one = torch.zeros(n * 2, dtype=torch.uint8).pin_memory()
        csg.symm_copy_from_slots(aw.h, one.data_ptr(), aw.base + aw.out_offs[0], n * 2, 1, s)
        s.synchronize()
        assert torch.equal(one, aw.out_view(0).cpu())
        for args in ((aw.slots[1], host.data_ptr(), 16, 1),          # not a slot-0 pointer
                     (aw.base, host.data_ptr(), 16, R + 1),          # too many ranks
                     (aw.base, 0, 16, 1)):                           # NULL source
            with pytest.raises(csg.SymmError) as e:
                csg.symm_copy_to_slots(aw.h, *args, s)
            assert e.value.code == csg.SYMM_EINVAL
        _guards_ok(aw.h)
    finally:
        aw.close()


@pytest.mark.parametrize("kind", ["pinned", "pageable", "device", "ragged_pinned"])
@pytest.mark.parametrize("engine", [0, 1])
def test_copy_slots_sources(kind, engine):
    """Every kind of contiguous buffer, both engines: pinned host and device
    memory go through the SMs (engine 0), pageable host memory through the
    copy engine whatever the option; block sizes that are not multiples of
    16 bytes take the byte-wise kernel."""
    R = 3
    nbytes = 4093 if kind == "ragged_pinned" else 4096
    aw = AllReduceWorkspace(R, 4096)
    try:
        csg.symm_set_option(aw.h, csg.SYMM_OPT_COPY_ENGINE, engine)
        s = torch.cuda.current_stream()
        data = torch.randint(0, 256, (R * nbytes,), dtype=torch.uint8)
        if kind in ("pinned", "ragged_pinned"):
            src = data.pin_memory()
            dst = torch.zeros_like(data).pin_memory()
        elif kind == "device":
            src = data.to(aw.device)
            dst = torch.zeros_like(src)
        else:
            src = data.clone()
            dst = torch.zeros_like(data)
        sym = aw.base + aw.in_offs[0]
        csg.symm_copy_to_slots(aw.h, sym, src.data_ptr(), nbytes, R, s)
        csg.symm_copy_from_slots(aw.h, dst.data_ptr(), sym, nbytes, R, s)
        s.synchronize()
        assert torch.equal(dst.cpu(), data)
        for r in range(R):
            assert torch.equal(aw.view(r, aw.in_offs[0], nbytes).cpu(), data[r * nbytes:(r + 1) * nbytes])
        _guards_ok(aw.h)
    finally:
        aw.close()
