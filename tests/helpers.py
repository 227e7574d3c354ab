"""Small test helpers: bf16 decoding by numpy, the parity tolerance, fixtures.

Nothing here computes the method; these are the yardsticks the tests hold the
oracle and the GPU path against.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Parity tolerance on every output: |y - y_ref| <= REL * |y_ref| + ABS * rms(y_ref),
# y_ref = the oracle's fp64 value before rounding, rms over all B*N outputs.
# A correctly rounded bf16 is within 2^-8 |y_ref| (< REL) of y_ref, and fp32
# accumulation error is far below ABS * rms for these sizes.
REL = 4e-3
ABS = 1e-3


def words_to_f64(words) -> np.ndarray:
    """bf16 words -> float64 through numpy's float32 decoding (bf16 is the top
    half of an fp32 word)."""
    w = np.asarray(words, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_words_via_f32(values) -> np.ndarray:
    """fp64 -> bf16 RNE for values exactly representable in fp32 (single
    rounding fp32 -> bf16 with the integer carry trick on the fp32 word)."""
    v = np.asarray(values, dtype=np.float64)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), v), "value not exact in fp32"
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def tolerance_ratio(y: np.ndarray, y_ref: np.ndarray, rms: float | None = None) -> float:
    """max over outputs of |y - y_ref| / (REL |y_ref| + ABS rms); <= 1 passes."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if y_ref.size == 0:
        return 0.0
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    bound = REL * np.abs(y_ref) + ABS * rms
    err = np.abs(y - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    return float(np.max(ratio))


def ulp_distance(a_words, b_words) -> np.ndarray:
    """Distance in bf16 steps between two arrays of finite bf16 words."""
    def ordered(w):
        w = np.asarray(w, dtype=np.uint16).astype(np.int64)
        return np.where(w & 0x8000, -(w & 0x7FFF), w)
    return np.abs(ordered(a_words) - ordered(b_words))


def load_golden(name: str) -> dict:
    """Parse a golden text fixture into {case: {key: value}}."""
    cases: dict = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                cur = cases.setdefault(line[5:].strip(), {})
                continue
            key, val = line.split(":", 1)
            if val.strip() == "none":
                cur[key.strip()] = None
                continue
            # "-" marks an entry the case leaves unspecified (NaN here)
            rows = [[float("nan") if t == "-" else float(t) for t in r.split()] for r in val.split(";")]
            cur[key.strip()] = rows[0][0] if len(rows) == 1 and len(rows[0]) == 1 else np.array(rows)
    return cases
