"""Seeded synthetic inputs for the GEMV + one-shot all-reduce workloads.

This module only produces input words (bf16 bit patterns as ``numpy.uint16``).
It holds none of the arithmetic of the method, so the CPU oracle and the GPU
path can both be fed from it without sharing any code with each other.

Generator: SplitMix64 in counter form plus Box-Muller for normals (see
``synth.c``).  Values are formed in fp64 and rounded once to bf16 (RNE).

Workloads (shapes, distributions and seeds of the five decode-time cases):

==================  =====================================================
name                recipe
==================  =====================================================
tiny                R=2 N=256 K=512 B=1; W~N(0,0.02) x~N(0,1); seed 0
allreduce           R=8 n=4,194,304; in_r~U[-1,1) for r=0..7; seed 1
attn_out_proj       R=4 N=8192 K=8192 B=8; W~N(0,0.02) x~N(0,1); seed 2
mlp_down_decode     R=8 N=8192 K=28672 B=1; W~N(0,0.01) x=SiLU(g)*u,
                    g,u~N(0,1); seed 3
mlp_down_large      R=8 N=16384 K=53248 B=16; W~N(0,0.006) x~N(0,1) with
                    floor(0.01 K) channels scaled x20; seed 4
ar_bias_rmsnorm     R=8 rows=1 H=8192; in_r~U[-1,1); bias~N(0,0.1),
                    gamma~N(1,0.1); eps 1e-6; seed 5
mlp_down_decode_rmsnorm
                    mlp_down_decode's W and x (seed 3) + bias~N(0,0.1),
                    gamma~N(1,0.1) over N; eps 1e-6
mlp_down_large_rs   mlp_down_large's W and x (seed 4), reduce-scatter of
                    the B=16 rows over R=8 ranks (2 rows each)
multi_root_tile     R=4, an 8192 x 8192 tensor per rank, in~U[-1,1);
                    its four 4096 x 4096 quadrants summed to roots 0..3;
                    seed 6
==================  =====================================================

"N(m, s)": s is the standard deviation.  W and x are generated as the global
row-major N x K and B x K tensors and then split by columns into the R rank
shards, so the same seed gives the same matrix for every R.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

TAG_W, TAG_X, TAG_G, TAG_U, TAG_OUTLIER, TAG_AR = 1, 2, 3, 4, 5, 6
TAG_BIAS, TAG_GAMMA, TAG_TILE = 7, 8, 9

WORKLOADS = {
    "tiny": dict(kind="gemv", R=2, N=256, K=512, B=1, seed=0, w_std=0.02, x="normal"),
    "allreduce": dict(kind="allreduce", R=8, n=4194304, seed=1),
    "attn_out_proj": dict(kind="gemv", R=4, N=8192, K=8192, B=8, seed=2, w_std=0.02, x="normal"),
    "mlp_down_decode": dict(kind="gemv", R=8, N=8192, K=28672, B=1, seed=3, w_std=0.01,
                            x="silu_mul"),
    "mlp_down_large": dict(kind="gemv", R=8, N=16384, K=53248, B=16, seed=4, w_std=0.006,
                           x="outliers"),
    "ar_bias_rmsnorm": dict(kind="ar_rmsnorm", R=8, rows=1, H=8192, seed=5, eps=1e-6),
    "mlp_down_decode_rmsnorm": dict(kind="gemv_rmsnorm", R=8, N=8192, K=28672, B=1, seed=3, w_std=0.01,
                                    x="silu_mul", eps=1e-6),
    "mlp_down_large_rs": dict(kind="gemv_rs", R=8, N=16384, K=53248, B=16, seed=4, w_std=0.006, x="outliers"),
    "multi_root_tile": dict(kind="tile", R=4, rows=8192, cols=8192, seed=6),
}


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, no GPU needed)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        for fn in (lib.synth_normal, lib.synth_uniform):
            fn.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double, ctypes.c_double,
                           ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, u16p, f64p, ctypes.c_int]
            fn.restype = ctypes.c_int
        lib.synth_choose.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.synth_choose.restype = ctypes.c_int
        lib.synth_round_array.argtypes = [f64p, ctypes.c_size_t, u16p]
        lib.synth_round_array.restype = None
        lib.synth_round_bf16.argtypes = [ctypes.c_double]
        lib.synth_round_bf16.restype = ctypes.c_uint16
        lib.synth_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_u64.restype = ctypes.c_uint64
        lib.synth_stream_base.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        lib.synth_stream_base.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray, ctype):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _gen(fn, seed, tag, p0, p1, rows, cols, shards, as_f64):
    lib = _load()
    if as_f64:
        out = np.empty((shards, rows, cols // shards), dtype=np.float64)
        rc = getattr(lib, fn)(seed, tag, p0, p1, rows, cols, shards, None, _ptr(out, ctypes.c_double),
                              _threads())
    else:
        out = np.empty((shards, rows, cols // shards), dtype=np.uint16)
        rc = getattr(lib, fn)(seed, tag, p0, p1, rows, cols, shards, _ptr(out, ctypes.c_uint16), None,
                              _threads())
    if rc != 0:
        raise ValueError(f"{fn}: bad arguments rows={rows} cols={cols} shards={shards}")
    return out


def normal(seed: int, tag: int, rows: int, cols: int, std: float = 1.0, mean: float = 0.0,
           shards: int = 1, as_f64: bool = False) -> np.ndarray:
    """N(mean, std) over a rows x cols tensor, split into ``shards`` column
    blocks: result shape (shards, rows, cols // shards)."""
    return _gen("synth_normal", seed, tag, mean, std, rows, cols, shards, as_f64)


def uniform(seed: int, tag: int, rows: int, cols: int, lo: float = -1.0, hi: float = 1.0,
            shards: int = 1, as_f64: bool = False) -> np.ndarray:
    """U[lo, hi) over a rows x cols tensor, shape (shards, rows, cols // shards)."""
    return _gen("synth_uniform", seed, tag, lo, hi, rows, cols, shards, as_f64)


def round_bf16(values: np.ndarray) -> np.ndarray:
    """fp64 values -> bf16 words (RNE), same shape."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().synth_round_array(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint16))
    return out


def choose(seed: int, tag: int, n: int, count: int) -> np.ndarray:
    """First ``count`` entries of a seeded Fisher-Yates shuffle of 0..n-1."""
    scratch = np.empty(max(n, 1), dtype=np.int32)
    out = np.empty(max(count, 1), dtype=np.int32)
    rc = _load().synth_choose(seed, tag, n, count, _ptr(scratch, ctypes.c_int), _ptr(out, ctypes.c_int))
    if rc != 0:
        raise ValueError("choose: bad arguments")
    return out[:count].copy()


def shard_columns(a: np.ndarray, R: int) -> np.ndarray:
    """(rows, K) -> (R, rows, K // R) column blocks."""
    rows, K = a.shape
    return np.ascontiguousarray(a.reshape(rows, R, K // R).transpose(1, 0, 2))


def gemv_inputs(R: int, N: int, K: int, B: int, seed: int, w_std: float, x: str = "normal"):
    """(W_shards [R, N, K/R], x_shards [R, B, K/R]) as bf16 words."""
    if K % R:
        raise ValueError("K must be a multiple of R")
    W = normal(seed, TAG_W, N, K, std=w_std, shards=R)
    if x == "normal":
        xs = normal(seed, TAG_X, B, K, std=1.0, shards=R)
    elif x == "silu_mul":
        g = normal(seed, TAG_G, B, K, as_f64=True)[0]
        u = normal(seed, TAG_U, B, K, as_f64=True)[0]
        xs = shard_columns(round_bf16(g / (1.0 + np.exp(-g)) * u), R)
    elif x == "outliers":
        xv = normal(seed, TAG_X, B, K, as_f64=True)[0]
        ch = choose(seed, TAG_OUTLIER, K, (K * 1) // 100)
        xv[:, ch] *= 20.0
        xs = shard_columns(round_bf16(xv), R)
    else:
        raise ValueError(f"unknown x recipe {x!r}")
    return W, xs


def outlier_channels(K: int, seed: int) -> np.ndarray:
    """The channels scaled x20 by the ``outliers`` x recipe."""
    return choose(seed, TAG_OUTLIER, K, (K * 1) // 100)


def allreduce_inputs(R: int, n: int, seed: int) -> np.ndarray:
    """in_r for r = 0..R-1 as one (R, n) array of bf16 words, U[-1, 1)."""
    return uniform(seed, TAG_AR, R, n, lo=-1.0, hi=1.0)[0]


def norm_vectors(n: int, seed: int):
    """(bias, gamma) for a bias + RMSNorm over n elements: bias ~ N(0, 0.1),
    gamma ~ N(1, 0.1), bf16 words of shape (n,)."""
    bias = normal(seed, TAG_BIAS, 1, n, std=0.1)[0, 0]
    gamma = normal(seed, TAG_GAMMA, 1, n, std=0.1, mean=1.0)[0, 0]
    return bias, gamma


def rmsnorm_inputs(R: int, rows: int, H: int, seed: int):
    """(in (R, rows, H), bias (H,), gamma (H,)) bf16 words; in_r ~ U[-1, 1)."""
    inp = uniform(seed, TAG_AR, R, rows * H, lo=-1.0, hi=1.0)[0].reshape(R, rows, H)
    bias, gamma = norm_vectors(H, seed)
    return inp, bias, gamma


def tile_inputs(R: int, rows: int, cols: int, seed: int) -> np.ndarray:
    """(R, rows, cols) bf16 words, U[-1, 1): each rank's full 2-D tensor."""
    return uniform(seed, TAG_TILE, R, rows * cols, lo=-1.0, hi=1.0)[0].reshape(R, rows, cols)


def workload_inputs(name: str):
    """Inputs of a named workload: (W, x) for GEMV cases (plus (bias, gamma)
    for the RMSNorm form), in_r for allreduce, (in, bias, gamma) for the
    all-reduce + bias + RMSNorm case, the full tensors for the tile case."""
    w = WORKLOADS[name]
    if w["kind"] == "allreduce":
        return allreduce_inputs(w["R"], w["n"], w["seed"])
    if w["kind"] == "ar_rmsnorm":
        return rmsnorm_inputs(w["R"], w["rows"], w["H"], w["seed"])
    if w["kind"] == "tile":
        return tile_inputs(w["R"], w["rows"], w["cols"], w["seed"])
    Wx = gemv_inputs(w["R"], w["N"], w["K"], w["B"], w["seed"], w["w_std"], w["x"])
    if w["kind"] == "gemv_rmsnorm":
        return Wx + norm_vectors(w["N"], w["seed"])
    return Wx
