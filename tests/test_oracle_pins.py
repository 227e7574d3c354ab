"""Pins of the CPU oracle to things other than itself (CPU only).

Each ``pin_*`` function takes an oracle instance and raises AssertionError on a
mismatch; ``test_oracle_mutants.py`` re-runs them against deliberately broken
copies of the oracle to show that every planted mistake trips at least one.

What each pin rests on:
  * bf16 decode: numpy's float32 decoding of the same bit pattern.
  * bf16 rounding: every bf16 value, every midpoint between neighbours (ties
    to even) and the fp64 numbers one step either side of each midpoint.
  * GEMV / all-reduce: exact brute force with Python integers on small-integer
    inputs; math.fsum with the standard summation error bound on random ones;
    closed forms (one-hot x, zero W, equal inputs); the hand-worked fixture in
    tests/golden/rowparallel_worked.txt; the row-parallel algebra (R = 1 is
    the unsharded product, any R gives the same fp64 sum up to associativity);
    exact power-of-two scaling; rank-order permutation within fp64 rounding.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import (f64_to_words_via_f32, load_golden, tolerance_ratio, words_to_f64)

U = 2.0 ** -53


def _int_words(rng, shape, lo=-8, hi=8):
    vals = rng.integers(lo, hi + 1, size=shape).astype(np.float64)
    return vals, f64_to_words_via_f32(vals)


# ------------------------------------------------------------------ bf16


def pin_bf16_decode(orc):
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_value(w)
    want = words_to_f64(w)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zero survives decoding
    assert math.copysign(1.0, orc.bf16_value(np.uint16(0x8000)).item()) == -1.0


def _finite_positive_words():
    return np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)


def pin_bf16_round_grid(orc):
    w = _finite_positive_words()
    v = words_to_f64(w)
    assert np.array_equal(orc.bf16_round(v), w)
    assert np.array_equal(orc.bf16_round(-v), w | np.uint16(0x8000))
    assert orc.bf16_round(np.inf).item() == 0x7F80
    assert orc.bf16_round(-np.inf).item() == 0xFF80


def pin_bf16_round_midpoints(orc):
    w = _finite_positive_words()
    lo = words_to_f64(w[:-1])
    hi = words_to_f64(w[1:])
    mid = (lo + hi) / 2.0                      # exact: 9 significant bits
    even = np.where(w[:-1] % 2 == 0, w[:-1], w[1:])
    assert np.array_equal(orc.bf16_round(mid), even)
    above = np.nextafter(mid, np.inf)
    below = np.nextafter(mid, 0.0)
    assert np.array_equal(orc.bf16_round(above), w[1:])
    assert np.array_equal(orc.bf16_round(below), w[:-1])
    # overflow: the midpoint between the largest finite bf16 and 2^128 ties to
    # even, and 0x7F80's "mantissa" is even, so it goes to infinity
    top = words_to_f64(np.uint16(0x7F7F)).item()
    assert orc.bf16_round(top + 2.0 ** 119).item() == 0x7F80
    assert orc.bf16_round(np.nextafter(top + 2.0 ** 119, 0.0)).item() == 0x7F7F
    # below half the smallest subnormal -> zero; just above -> smallest subnormal
    assert orc.bf16_round(2.0 ** -134).item() == 0x0000
    assert orc.bf16_round(np.nextafter(2.0 ** -134, 1.0)).item() == 0x0001


# ------------------------------------------------------------------ GEMV


def _brute_gemv(Wv, xv):
    """Exact y = sum_r W_r x_r with Python integers (inputs are integers)."""
    R, N, Kr = Wv.shape
    B = xv.shape[1]
    y = np.zeros((B, N), dtype=object)
    for b in range(B):
        for n in range(N):
            y[b, n] = sum(int(Wv[r, n, k]) * int(xv[r, b, k]) for r in range(R) for k in range(Kr))
    return y


def pin_gemv_brute_force(orc):
    rng = np.random.default_rng(1234)
    combos = [(1, 1, 8, 1), (2, 3, 16, 2), (4, 8, 24, 5), (2, 17, 8, 16), (4, 3, 16, 1),
              (1, 17, 24, 2), (2, 8, 24, 5), (4, 1, 8, 16)]
    for R, N, Kr, B in combos:
        Wv, Ww = _int_words(rng, (R, N, Kr))
        xv, xw = _int_words(rng, (R, B, Kr))
        exact = _brute_gemv(Wv, xv)
        y_ref, y = orc.gemv_all_reduce(Ww, xw)
        assert y.shape == (R, B, N)
        assert np.array_equal(y_ref, exact.astype(np.float64)), (R, N, Kr, B)
        # |y| <= 16 * 24 * 64 < 2^24, so fp32 holds it exactly
        want = f64_to_words_via_f32(exact.astype(np.float64))
        for s in range(R):
            assert np.array_equal(y[s], want), (R, N, Kr, B, s)


def pin_gemv_partials_brute_force(orc):
    rng = np.random.default_rng(99)
    R, N, Kr, B = 4, 5, 16, 3
    Wv, Ww = _int_words(rng, (R, N, Kr))
    xv, xw = _int_words(rng, (R, B, Kr))
    for b, n in [(0, 0), (2, 4), (1, 3)]:
        want = [sum(int(Wv[r, n, k]) * int(xv[r, b, k]) for k in range(Kr)) for r in range(R)]
        assert np.array_equal(orc.gemv_partials(Ww, xw, b, n), np.array(want, dtype=np.float64))


def pin_gemv_golden(orc):
    g = load_golden("rowparallel_worked.txt")
    for name in ("rowparallel_R2_N3_K4_B2", "rounding_ties_R2_N2_K2_B1"):
        c = g[name]
        R, N, K, B = int(c["R"]), int(c["N"]), int(c["K"]), int(c["B"])
        Wg = np.asarray(c["W"], dtype=np.float64).reshape(N, K)
        xg = np.asarray(c["x"], dtype=np.float64).reshape(B, K)
        Ww = synth.shard_columns(f64_to_words_via_f32(Wg), R)
        xw = synth.shard_columns(f64_to_words_via_f32(xg), R)
        y_ref, y = orc.gemv_all_reduce(Ww, xw)
        assert np.array_equal(y_ref, np.asarray(c["y_exact"]).reshape(B, N)), name
        want = f64_to_words_via_f32(np.asarray(c["y_bf16"]).reshape(B, N))
        for s in range(R):
            assert np.array_equal(y[s], want), name
        for r, key in enumerate(("P0", "P1")):
            P = np.asarray(c[key]).reshape(B, N)
            for b in range(B):
                for n in range(N):
                    assert orc.gemv_partials(Ww, xw, b, n)[r] == P[b, n], (name, key, b, n)


def pin_gemv_fsum_bound(orc):
    """Random bf16 inputs: y_ref is the sequentially summed fp64 value, so it
    lies within (K - 1) u sum|terms| of the exactly rounded sum (math.fsum);
    every product of two bf16 values is exact in fp64."""
    R, N, K, B = 4, 6, 256, 3
    W = synth.normal(7, synth.TAG_W, N, K, std=0.02, shards=R)
    x = synth.normal(7, synth.TAG_X, B, K, std=1.0, shards=R)
    Wf = words_to_f64(W)
    xf = words_to_f64(x)
    y_ref, _ = orc.gemv_all_reduce(W, x)
    for b in range(B):
        for n in range(N):
            terms = [Wf[r, n, k] * xf[r, b, k] for r in range(R) for k in range(K // R)]
            exact = math.fsum(terms)
            bound = (K - 1) * U * math.fsum(abs(t) for t in terms)
            assert abs(y_ref[b, n] - exact) <= bound, (b, n)


def pin_gemv_r1_is_unsharded(orc):
    """R = 1 is the plain (unsharded) GEMV: compare with a dot product summed
    in the same ascending order by Python floats (bit-identical)."""
    N, K, B = 5, 96, 2
    W = synth.normal(11, synth.TAG_W, N, K, std=0.02, shards=1)
    x = synth.normal(11, synth.TAG_X, B, K, std=1.0, shards=1)
    Wf, xf = words_to_f64(W[0]), words_to_f64(x[0])
    y_ref, _ = orc.gemv_all_reduce(W, x)
    for b in range(B):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Wf[n, k] * xf[b, k]
            assert y_ref[b, n] == acc


def pin_gemv_sharding_invariance(orc):
    """The same global W, x split over R = 1, 2, 4, 8 ranks: identical fp64
    sums up to associativity, and within the parity tolerance after rounding."""
    N, K, B = 7, 512, 2
    W = synth.normal(3, synth.TAG_W, N, K, std=0.02, shards=1)[0]
    x = synth.normal(3, synth.TAG_X, B, K, std=1.0, shards=1)[0]
    absum = np.abs(words_to_f64(W)) @ np.abs(words_to_f64(x)).T   # (N, B)
    base = None
    for R in (1, 2, 4, 8):
        y_ref, y = orc.gemv_all_reduce(synth.shard_columns(W, R), synth.shard_columns(x, R))
        if base is None:
            base = y_ref
            continue
        assert np.all(np.abs(y_ref - base) <= 2 * K * U * absum.T), R
        assert tolerance_ratio(words_to_f64(y[0]), base) <= 1.0


def pin_gemv_one_hot(orc):
    """x = e_k (value 1 at global column k): y = W[:, k] exactly."""
    R, N, K = 4, 9, 64
    W = synth.normal(5, synth.TAG_W, N, K, std=0.5, shards=1)[0]
    for k in (0, 17, 40, 63):
        xg = np.zeros((1, K))
        xg[0, k] = 1.0
        y_ref, y = orc.gemv_all_reduce(synth.shard_columns(W, R),
                                       synth.shard_columns(f64_to_words_via_f32(xg), R))
        assert np.array_equal(y_ref[0], words_to_f64(W[:, k])), k
        assert np.array_equal(words_to_f64(y[0, 0]), words_to_f64(W[:, k])), k


def pin_gemv_zero_weights(orc):
    R, N, K, B = 2, 4, 32, 3
    W = np.zeros((R, N, K // R), dtype=np.uint16)
    x = synth.normal(1, synth.TAG_X, B, K, shards=R)
    y_ref, y = orc.gemv_all_reduce(W, x)
    assert np.all(y_ref == 0.0)
    assert np.all(y == 0)                      # +0, not -0


def pin_gemv_power_of_two_scaling(orc):
    """y(2^j x) = 2^j y(x) bit-exactly (scaling by 2^j is exact everywhere)."""
    R, N, K, B = 4, 8, 128, 2
    W = synth.normal(9, synth.TAG_W, N, K, std=0.02, shards=R)
    x = synth.normal(9, synth.TAG_X, B, K, std=1.0, shards=R)
    y_ref, y = orc.gemv_all_reduce(W, x)
    for j in (1, 3, -2):
        xs = f64_to_words_via_f32(words_to_f64(x) * 2.0 ** j)
        y2_ref, y2 = orc.gemv_all_reduce(W, xs)
        assert np.array_equal(y2_ref, y_ref * 2.0 ** j), j
        assert np.array_equal(words_to_f64(y2), words_to_f64(y) * 2.0 ** j), j


def pin_gemv_additivity(orc):
    """y(x1 + x2) = y(x1) + y(x2) (x1 + x2 exact in bf16; fp64 rounding only)."""
    rng = np.random.default_rng(5)
    R, N, K, B = 2, 6, 64, 2
    W = synth.normal(4, synth.TAG_W, N, K, std=0.02, shards=R)
    x1 = rng.integers(-64, 64, size=(R, B, K // R)) / 16.0
    x2 = rng.integers(-64, 64, size=(R, B, K // R)) / 16.0
    ya, _ = orc.gemv_all_reduce(W, f64_to_words_via_f32(x1))
    yb, _ = orc.gemv_all_reduce(W, f64_to_words_via_f32(x2))
    ys, _ = orc.gemv_all_reduce(W, f64_to_words_via_f32(x1 + x2))
    scale = np.abs(words_to_f64(W)).sum(axis=(0, 2)).max() * 8.0
    assert np.all(np.abs(ys - (ya + yb)) <= 4 * K * U * scale)
    assert not np.allclose(ya, 0.0)


def pin_gemv_rank_order(orc):
    """Summing the rank partials in another order moves fp64 results only by
    rounding, and the bf16 result stays within tolerance."""
    R, N, K, B = 8, 16, 256, 2
    W = synth.normal(21, synth.TAG_W, N, K, std=0.02, shards=R)
    x = synth.normal(21, synth.TAG_X, B, K, std=1.0, shards=R)
    y_ref, y = orc.gemv_all_reduce(W, x)
    absum = np.abs(words_to_f64(W).transpose(1, 0, 2).reshape(N, K)) @ \
        np.abs(words_to_f64(x).transpose(1, 0, 2).reshape(B, K)).T
    for order in ([7, 6, 5, 4, 3, 2, 1, 0], [3, 0, 6, 1, 7, 2, 5, 4]):
        y2_ref, y2 = orc.gemv_all_reduce(W, x, order=order)
        assert np.all(np.abs(y2_ref - y_ref) <= 2 * K * U * absum.T)
        assert tolerance_ratio(words_to_f64(y2[0]), y_ref) <= 1.0
    # the order really is used: rank 0 first vs. last gives the same partials
    p = orc.gemv_partials(W, x, 1, 3)
    assert abs(sum(p) - y_ref[1, 3]) <= 2 * R * U * np.abs(p).sum()


def pin_summation_order_is_sequential(orc):
    """The definition sums each rank's terms in ascending k and the partials in
    rank order, sequentially.  Terms 2^60, 1, -2^60 expose the order exactly:
    (2^60 + 1) - 2^60 = 0 in fp64, while (2^60 - 2^60) + 1 = 1."""
    big = 2.0 ** 60
    # across ranks: R = 3, one term per rank
    W = f64_to_words_via_f32(np.array([[[big]], [[1.0]], [[-big]]]))
    x = f64_to_words_via_f32(np.ones((3, 1, 1)))
    assert orc.gemv_all_reduce(W, x)[0][0, 0] == 0.0
    assert orc.gemv_all_reduce(W, x, order=[0, 2, 1])[0][0, 0] == 1.0
    assert orc.gemv_all_reduce(W, x, order=[2, 0, 1])[0][0, 0] == 1.0
    assert orc.gemv_all_reduce(W, x, order=[1, 0, 2])[0][0, 0] == 0.0
    # within one rank: ascending k
    W1 = f64_to_words_via_f32(np.array([[[big, 1.0, -big]]]))
    x1 = f64_to_words_via_f32(np.ones((1, 1, 3)))
    assert orc.gemv_all_reduce(W1, x1)[0][0, 0] == 0.0
    W2 = f64_to_words_via_f32(np.array([[[big, -big, 1.0]]]))
    assert orc.gemv_all_reduce(W2, x1)[0][0, 0] == 1.0
    # all-reduce: same rule over ranks
    inp = f64_to_words_via_f32(np.array([[big], [1.0], [-big]]))
    assert orc.one_shot_all_reduce(inp)[0][0] == 0.0
    assert orc.one_shot_all_reduce(inp, order=[0, 2, 1])[0][0] == 1.0


def pin_gemv_element_matches_full(orc):
    R, N, K, B = 4, 10, 64, 3
    W = synth.normal(2, synth.TAG_W, N, K, std=0.02, shards=R)
    x = synth.normal(2, synth.TAG_X, B, K, shards=R)
    y_ref, _ = orc.gemv_all_reduce(W, x)
    for b, n in itertools.product(range(B), (0, 5, 9)):
        assert orc.gemv_element(W, x, b, n) == y_ref[b, n]


def pin_rounding_meets_tolerance(orc):
    """Sanity of the tolerance reading: correct RNE rounding of y_ref always
    passes |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms."""
    W, x = synth.gemv_inputs(2, 256, 512, 1, 0, 0.02, "normal")
    y_ref, y = orc.gemv_all_reduce(W, x)
    assert tolerance_ratio(words_to_f64(y[0]), y_ref) <= 0.98


# ------------------------------------------------------------ all-reduce


def pin_allreduce_brute_force(orc):
    rng = np.random.default_rng(77)
    for R, n in ((1, 5), (2, 33), (8, 100), (3, 1)):
        vals, words = _int_words(rng, (R, n), -100, 100)
        ref, out = orc.one_shot_all_reduce(words)
        exact = vals.sum(axis=0)                 # small integers: exact
        assert np.array_equal(ref, exact)
        for s in range(R):
            assert np.array_equal(out[s], f64_to_words_via_f32(exact))


def pin_allreduce_constant(orc):
    for R in (1, 2, 8):
        c = 0.375
        words = f64_to_words_via_f32(np.full((R, 17), c))
        ref, out = orc.one_shot_all_reduce(words)
        assert np.all(ref == R * c)
        assert np.all(words_to_f64(out) == R * c)


def pin_allreduce_golden(orc):
    g = load_golden("rowparallel_worked.txt")
    for name in ("allreduce_R3_n4", "allreduce_tie_R2_n2"):
        c = g[name]
        R, n = int(c["R"]), int(c["n"])
        words = f64_to_words_via_f32(np.asarray(c["in"]).reshape(R, n))
        ref, out = orc.one_shot_all_reduce(words)
        assert np.array_equal(ref, np.asarray(c["y_exact"]).reshape(n)), name
        want = f64_to_words_via_f32(np.asarray(c["y_bf16"]).reshape(n))
        for s in range(R):
            assert np.array_equal(out[s], want), name


def pin_allreduce_fsum_bound(orc):
    inp = synth.allreduce_inputs(8, 1000, 1)
    v = words_to_f64(inp)
    ref, _ = orc.one_shot_all_reduce(inp)
    for i in range(0, 1000, 7):
        exact = math.fsum(v[:, i])
        assert abs(ref[i] - exact) <= 7 * U * np.abs(v[:, i]).sum()


def pin_allreduce_order(orc):
    inp = synth.allreduce_inputs(8, 500, 3)
    ref, _ = orc.one_shot_all_reduce(inp)
    ref2, _ = orc.one_shot_all_reduce(inp, order=[7, 6, 5, 4, 3, 2, 1, 0])
    assert np.all(np.abs(ref2 - ref) <= 8 * U * np.abs(words_to_f64(inp)).sum(axis=0))


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load())
