"""The seeded input generator: determinism, layout, distributions (CPU only)."""
from __future__ import annotations

import numpy as np

import synth
from helpers import words_to_f64


def test_deterministic_and_thread_invariant(monkeypatch):
    a = synth.normal(3, synth.TAG_W, 37, 64, std=0.02, shards=4)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    b = synth.normal(3, synth.TAG_W, 37, 64, std=0.02, shards=4)
    monkeypatch.setattr(synth, "_threads", lambda: 7)
    c = synth.normal(3, synth.TAG_W, 37, 64, std=0.02, shards=4)
    assert np.array_equal(a, b) and np.array_equal(a, c)
    assert not np.array_equal(a, synth.normal(4, synth.TAG_W, 37, 64, std=0.02, shards=4))


def test_sharding_is_a_column_split():
    g = synth.normal(5, synth.TAG_X, 6, 48, shards=1)[0]
    s = synth.normal(5, synth.TAG_X, 6, 48, shards=4)
    for r in range(4):
        assert np.array_equal(s[r], g[:, r * 12:(r + 1) * 12])
    assert np.array_equal(synth.shard_columns(g, 4), s)


def test_normal_moments():
    v = words_to_f64(synth.normal(1, synth.TAG_W, 512, 1024, std=0.02))
    assert abs(v.mean()) < 2e-4
    assert abs(v.std() / 0.02 - 1.0) < 0.01


def test_uniform_range():
    v = words_to_f64(synth.allreduce_inputs(8, 10000, 1))
    assert v.min() >= -1.0 and v.max() <= 1.0
    assert abs(v.mean()) < 0.02


def test_workload_recipes_small():
    W, x = synth.gemv_inputs(2, 256, 512, 1, 0, 0.02, "normal")
    assert W.shape == (2, 256, 256) and x.shape == (2, 1, 256)
    W, x = synth.gemv_inputs(8, 16, 1024, 2, 3, 0.01, "silu_mul")
    xv = words_to_f64(x)
    assert x.shape == (8, 2, 128) and np.isfinite(xv).all()
    W, x = synth.gemv_inputs(8, 16, 1600, 3, 4, 0.006, "outliers")
    ch = synth.outlier_channels(1600, 4)
    assert len(ch) == 16 and len(set(ch.tolist())) == 16 and ch.min() >= 0 and ch.max() < 1600
    xg = words_to_f64(x).transpose(1, 0, 2).reshape(3, 1600)
    mask = np.zeros(1600, bool)
    mask[ch] = True
    assert np.abs(xg[:, mask]).mean() > 10 * np.abs(xg[:, ~mask]).mean()


def test_round_bf16_matches_fp32_route():
    rng = np.random.default_rng(0)
    f = rng.standard_normal(10000).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    want = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(synth.round_bf16(f.astype(np.float64)), want)
