"""Pins of the oracle's further collectives to things other than the oracle
(CPU only): reduce-scatter (flat and along the fused layer's batch rows),
all-reduce + bias + RMSNorm (alone and as the fused layer's epilogue), and the
2-D tile reduce to one or several roots.

What each pin rests on:
  * exact brute force with Python integers / numpy slicing on small-integer
    inputs (every sum exact in fp64 and in bf16);
  * the hand-worked cases of tests/golden/collectives_worked.txt;
  * the already pinned one-shot all-reduce and GEMV definitions (the
    reduce-scatter blocks must be the all-reduce's elements, bit for bit);
  * RMSNorm closed forms and invariants worked in plain Python arithmetic
    (math.fsum, math.sqrt): unit mean square with eps = 0, exact invariance
    under power-of-two scaling, constant rows, the bias as an extra rank.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth
from helpers import f64_to_words_via_f32, load_golden, tolerance_ratio, words_to_f64

GOLD = "collectives_worked.txt"


def _int_words(rng, shape, lo=-8, hi=8):
    vals = rng.integers(lo, hi + 1, size=shape).astype(np.float64)
    return vals, f64_to_words_via_f32(vals)


def _words(a):
    return f64_to_words_via_f32(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------- reduce-scatter


def pin_rs_golden(orc):
    g = load_golden(GOLD)
    for name in ("reduce_scatter_R2_n4_ties", "reduce_scatter_R4_n8"):
        c = g[name]
        R, n = int(c["R"]), int(c["n"])
        ref, out = orc.reduce_scatter(_words(c["in"]).reshape(R, n))
        assert np.array_equal(ref, np.asarray(c["sum_exact"]).reshape(n)), name
        assert np.array_equal(out, _words(c["out_bf16"]).reshape(R, n // R)), name


def pin_rs_brute_force(orc):
    rng = np.random.default_rng(5)
    for R, n in ((1, 7), (2, 10), (4, 36), (8, 64), (3, 9)):
        vals, words = _int_words(rng, (R, n), -100, 100)
        ref, out = orc.reduce_scatter(words)
        exact = [sum(int(vals[r, i]) for r in range(R)) for i in range(n)]
        assert np.array_equal(ref, np.array(exact, dtype=np.float64))
        c = n // R
        for s in range(R):
            assert np.array_equal(out[s], _words(exact[s * c:(s + 1) * c])), (R, n, s)


def pin_rs_blocks_are_allreduce(orc):
    inp = synth.allreduce_inputs(8, 8 * 1000, 11)
    _, ar = orc.one_shot_all_reduce(inp)
    _, rs = orc.reduce_scatter(inp)
    assert np.array_equal(rs.reshape(-1), ar[0])


def pin_rs_rejects_ragged(orc):
    with pytest.raises(ValueError):
        orc.reduce_scatter(np.zeros((4, 10), dtype=np.uint16))


def pin_gemv_rs_brute_force(orc):
    rng = np.random.default_rng(6)
    for R, N, Kr, B in ((1, 3, 8, 1), (2, 5, 16, 2), (4, 9, 8, 8), (2, 17, 24, 16), (8, 3, 8, 16)):
        Wv, Ww = _int_words(rng, (R, N, Kr))
        xv, xw = _int_words(rng, (R, B, Kr))
        y_ref, out = orc.gemv_reduce_scatter(Ww, xw)
        exact = np.zeros((B, N), dtype=np.int64)
        for b in range(B):
            for n in range(N):
                exact[b, n] = sum(int(Wv[r, n, k]) * int(xv[r, b, k]) for r in range(R) for k in range(Kr))
        assert np.array_equal(y_ref, exact.astype(np.float64))
        Bs = B // R
        assert out.shape == (R, Bs, N)
        for s in range(R):
            assert np.array_equal(out[s], _words(exact[s * Bs:(s + 1) * Bs].astype(np.float64))), (R, B, s)


def pin_gemv_rs_golden(orc):
    c = load_golden("rowparallel_worked.txt")["rowparallel_R2_N3_K4_B2"]
    R, N, K, B = (int(c[k]) for k in ("R", "N", "K", "B"))
    Wg, xg = np.asarray(c["W"]), np.asarray(c["x"])
    Ww = _words(synth.shard_columns(Wg, R).reshape(R, N, K // R))
    xw = _words(synth.shard_columns(xg, R).reshape(R, B, K // R))
    _, out = orc.gemv_reduce_scatter(Ww, xw)
    y = np.asarray(c["y_bf16"])
    for s in range(R):
        assert np.array_equal(out[s], _words(y[s:s + 1]))


def pin_gemv_rs_rejects_ragged_batch(orc):
    with pytest.raises(ValueError):
        orc.gemv_reduce_scatter(np.zeros((4, 2, 8), dtype=np.uint16), np.zeros((4, 6, 8), dtype=np.uint16))


# ------------------------------------------------- all-reduce + bias + RMSNorm


def _opt(c, key):
    v = c[key]
    return None if v is None else _words(np.asarray(v).reshape(-1))


def pin_rmsnorm_golden(orc):
    g = load_golden(GOLD)
    for name in ("rmsnorm_R2_H4_bias_gamma", "rmsnorm_R3_H2_eps", "rmsnorm_R2_H2_irrational"):
        c = g[name]
        R, rows, H = int(c["R"]), int(c["rows"]), int(c["H"])
        inp = _words(c["in"]).reshape(R, rows, H)
        ref, out = orc.all_reduce_bias_rmsnorm(inp, _opt(c, "bias"), _opt(c, "gamma"), float(c["eps"]))
        want = np.asarray(c["y_exact"]).reshape(rows, H)
        assert np.allclose(ref, want, rtol=1e-11, atol=0), name
        wb = _words(np.asarray(c["y_bf16"]).reshape(rows, H))
        for s in range(R):
            assert np.array_equal(out[s], wb), name


def _py_rmsnorm(z, gamma, eps):
    ms = math.fsum(v * v for v in z) / len(z)
    d = math.sqrt(ms + eps)
    return [v / d * g for v, g in zip(z, gamma)]


def pin_rmsnorm_python_arithmetic(orc):
    R, rows, H = 4, 3, 256
    inp = synth.allreduce_inputs(R, rows * H, 21).reshape(R, rows, H)
    bias = synth.normal(21, 90, 1, H, std=0.5)[0, 0]
    gamma = synth.normal(21, 91, 1, H, std=1.0, mean=1.0)[0, 0]
    ref, _ = orc.all_reduce_bias_rmsnorm(inp, bias, gamma, 1e-5)
    iv, bv, gv = words_to_f64(inp), words_to_f64(bias), words_to_f64(gamma)
    for i in range(rows):
        z = [math.fsum(iv[:, i, h]) + bv[h] for h in range(H)]
        want = _py_rmsnorm(z, gv, 1e-5)
        assert np.allclose(ref[i], want, rtol=1e-12, atol=1e-14)


def pin_rmsnorm_unit_mean_square(orc):
    inp = synth.allreduce_inputs(8, 4 * 1000, 22).reshape(8, 4, 1000)
    ref, _ = orc.all_reduce_bias_rmsnorm(inp, None, None, 0.0)
    for i in range(4):
        assert abs(math.fsum(v * v for v in ref[i]) / 1000 - 1.0) < 1e-13


def pin_rmsnorm_power_of_two_invariance(orc):
    rng = np.random.default_rng(23)
    vals, words = _int_words(rng, (4, 2, 64), -50, 50)
    gamma = synth.normal(23, 92, 1, 64, std=1.0)[0, 0]
    ref, out = orc.all_reduce_bias_rmsnorm(words, None, gamma, 0.0)
    for j in (-3, 2, 5):
        ref2, out2 = orc.all_reduce_bias_rmsnorm(_words(vals * 2.0 ** j), None, gamma, 0.0)
        assert np.array_equal(ref2, ref) and np.array_equal(out2, out), j


def pin_rmsnorm_constant_row_eps(orc):
    # z = c everywhere: y = c / sqrt(c^2 + eps) * gamma
    for c, eps in ((3.0, 0.0), (-2.0, 5.0), (0.5, 0.75)):
        inp = _words(np.full((2, 1, 16), c / 2))
        gamma = _words(np.arange(-8, 8) * 0.25)
        ref, _ = orc.all_reduce_bias_rmsnorm(inp, None, gamma, eps)
        want = c / math.sqrt(c * c + eps) * words_to_f64(gamma)
        assert np.allclose(ref[0], want, rtol=1e-15, atol=0)


def pin_rmsnorm_bias_is_an_extra_rank(orc):
    rng = np.random.default_rng(24)
    vals, words = _int_words(rng, (3, 2, 40), -20, 20)
    bvals, bwords = _int_words(rng, (40,), -20, 20)
    ref, out = orc.all_reduce_bias_rmsnorm(words, bwords, None, 1e-3)
    extra = np.concatenate([vals, np.broadcast_to(bvals, (1, 2, 40))], axis=0)
    ref2, out2 = orc.all_reduce_bias_rmsnorm(_words(extra), None, None, 1e-3)
    assert np.array_equal(ref, ref2)
    assert np.array_equal(out[0], out2[0])


def pin_gemv_rmsnorm_composition(orc):
    W, x = synth.gemv_inputs(4, 96, 512, 3, 25, 0.05)
    bias = synth.normal(25, 93, 1, 96, std=0.3)[0, 0]
    gamma = synth.normal(25, 94, 1, 96, std=0.2, mean=1.0)[0, 0]
    y_ref, y = orc.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6)
    g_ref, _ = orc.gemv_all_reduce(W, x)
    bv, gv = words_to_f64(bias), words_to_f64(gamma)
    for b in range(3):
        want = _py_rmsnorm([g_ref[b, n] + bv[n] for n in range(96)], gv, 1e-6)
        assert np.allclose(y_ref[b], want, rtol=1e-12, atol=1e-14)
    for s in range(4):
        assert np.array_equal(y[s], y[0])
    assert tolerance_ratio(words_to_f64(y[0]), y_ref) <= 0.98


# -------------------------------------------------------------- tile reduce


def pin_tile_golden(orc):
    g = load_golden(GOLD)
    for name in ("tile_R2_3x4_root1", "multi_root_R2_4x4_quadrants"):
        c = g[name]
        R = int(c["R"])
        se = int(c["slot_rows"]) * int(c["slot_cols"])
        slots_in = _words(c["in"]).reshape(R, se)
        before = np.full((R, se), 0x7FC0, dtype=np.uint16)   # NaN marks "left as it was"
        offs = np.atleast_1d(np.asarray(c["in_offs"])).astype(int).reshape(-1)
        roots = np.atleast_1d(np.asarray(c["roots"])).astype(int).reshape(-1)
        rows, cols = int(c["rows"]), int(c["cols"])
        ref, out = orc.tile_reduce(slots_in, before, offs, int(c["out_off"]), roots, rows, cols,
                                   int(c["ld_in"]), int(c["ld_out"]))
        assert np.array_equal(ref.reshape(len(offs), -1), np.asarray(c["tile_exact"]).reshape(len(offs), -1))
        after = np.asarray(c["out_after"]).reshape(R, se)
        keep = np.isnan(after)
        assert np.array_equal(out[keep], before[keep]), name
        assert np.array_equal(out[~keep], _words(after[~keep])), name


def _np_tile(slots, off, rows, cols, ld):
    return np.stack([np.lib.stride_tricks.as_strided(s[off:], shape=(rows, cols), strides=(ld * s.itemsize, s.itemsize))
                     for s in slots])


def pin_tile_brute_force(orc):
    rng = np.random.default_rng(26)
    cases = [  # R, slot rows x cols (row-major, ld = cols), tiles (row0, col0), roots, rows, cols
        (4, 16, 24, [(0, 0), (0, 12), (8, 0), (8, 12)], [0, 1, 2, 3], 8, 12),
        (2, 9, 7, [(2, 3)], [1], 5, 4),
        (8, 5, 40, [(1, 1), (0, 20), (3, 5)], [6, 0, 3], 2, 17),
        (3, 4, 4, [(0, 0)], [2], 0, 3),
    ]
    for R, sr, sc, tiles, roots, rows, cols in cases:
        vals, words = _int_words(rng, (R, sr * sc), -60, 60)
        before = rng.integers(0, 0x7F00, size=(R, sr * sc)).astype(np.uint16)
        offs = [a * sc + b for a, b in tiles]
        # output tile: a rows x cols block of a (rows+1) x (cols+3) tensor at (1, 2)
        ldo = cols + 3
        oo = 1 * ldo + 2
        ref, out = orc.tile_reduce(words, before, offs, oo, roots, rows, cols, sc, ldo)
        want_out = before.copy()
        for i, (off, root) in enumerate(zip(offs, roots)):
            t = _np_tile(vals, off, rows, cols, sc).sum(axis=0)
            assert np.array_equal(ref[i], t), (R, i)
            for a in range(rows):
                want_out[root, oo + a * ldo: oo + a * ldo + cols] = _words(t[a])
        assert np.array_equal(out, want_out), (R, sr, sc)


def pin_tile_separate_output_tensor(orc):
    # the docs' quadrant example: a full n x n tensor per rank, the output a
    # separate (n/2) x (n/2) tensor; quadrant q summed into rank q's output
    rng = np.random.default_rng(27)
    R, n = 4, 12
    h = n // 2
    vals, words = _int_words(rng, (R, n * n), -30, 30)
    before = np.full((R, h * h), 0x7FC0, dtype=np.uint16)
    offs = [0, h, h * n, h * n + h]
    ref, out = orc.tile_reduce(words, before, offs, 0, [0, 1, 2, 3], h, h, n, h)
    full = vals.reshape(R, n, n).sum(axis=0)
    quads = [full[:h, :h], full[:h, h:], full[h:, :h], full[h:, h:]]
    for q in range(4):
        assert np.array_equal(ref[q], quads[q])
        assert np.array_equal(out[q], _words(quads[q].reshape(-1)))
    with pytest.raises(ValueError):    # the output tile must fit the output slot
        orc.tile_reduce(words, before, offs, 1, [0, 1, 2, 3], h, h, n, h)


def pin_tile_rejects_bad_roots_and_extents(orc):
    z = np.zeros((4, 64), dtype=np.uint16)
    for offs, roots, rows, cols, ld in (([0, 8], [1, 1], 2, 2, 8),     # root twice
                                        ([0], [4], 2, 2, 8),           # root out of range
                                        ([0], [-1], 2, 2, 8),
                                        ([60], [0], 2, 2, 8),          # tile leaves the slot
                                        ([0], [0], 2, 9, 8)):          # cols > leading dimension
        with pytest.raises(ValueError):
            orc.tile_reduce(z, z, offs, 0, roots, rows, cols, ld, ld)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load())
