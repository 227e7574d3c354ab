"""CPU oracle for the tensor-parallel GEMV + one-shot all-reduce (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may call it; the product package never imports it.
It shares no code with the CUDA path.

Every function follows the definitions stated in ``oracle.c``:

* ``gemv_all_reduce``: y[b][n] = sum_r sum_k W_r[n][k] x_r[b][k] in fp64 (per
  rank ascending k, ranks in order), rounded once fp64 -> bf16 (RNE) and
  written to every rank's slot.  Row-parallel linear layer ending in one
  all-reduce ("Bay.Area.AI: Tensor and 2D Parallelism", column-then-row
  sharding passage); fused GEMV + AllReduce ("Overlapping Collective
  Communication with Dependent Computation ...", Abstract).
* ``one_shot_all_reduce``: out[i] = sum_r in_r[i] in fp64, rank order, RNE to
  bf16 for every rank ("PyTorch Symmetric Memory" talk, one-shot segment;
  symmetric memory docs, ``one_shot_all_reduce``).
* ``reduce_scatter``: rank s keeps block s of the flat sum; ``gemv_reduce_scatter``:
  rank s keeps batch rows [s*B/R, (s+1)*B/R) of the fused layer's output
  ("Bay.Area.AI: Tensor and 2D Parallelism", sequence-parallel passage).  The
  two-shot all-reduce reaches the all-reduce definition, so its oracle is
  ``one_shot_all_reduce``.
* ``all_reduce_bias_rmsnorm`` / ``gemv_bias_rmsnorm``: all-reduce, plus bias, then
  RMS normalisation per row with gain gamma and eps inside the square root
  ("PyTorch Symmetric Memory" talk, fused-kernel segment).
* ``tile_reduce``: 2-D strided tiles summed over ranks into one root's output
  tile each (symmetric memory docs, ``tile_reduce`` / ``multi_root_tile_reduce``).
* ``bf16_value`` / ``bf16_round``: the bf16 encoding, decoded from its fields
  and rounded from fp64 bit fields.

Pins (tests/test_oracle_pins.py) check each of these against exact
brute force, closed forms, invariants and a hand-worked fixture.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile the oracle with gcc.  ``src``/``out`` let a test compile a
    deliberately broken copy elsewhere; the default is the real oracle."""
    src = src or _SRC
    out = out or _LIB_PATH
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = ctypes.c_double
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_gemv_all_reduce.argtypes = [ctypes.c_int] * 4 + [u16p, u16p, ip, f64p, u16p, ctypes.c_int]
    lib.oracle_gemv_all_reduce.restype = ctypes.c_int
    lib.oracle_gemv_element.argtypes = [ctypes.c_int] * 4 + [u16p, u16p, ctypes.c_int, ctypes.c_int]
    lib.oracle_gemv_element.restype = ctypes.c_double
    lib.oracle_gemv_partials.argtypes = [ctypes.c_int] * 4 + [u16p, u16p, ctypes.c_int, ctypes.c_int,
                                                              f64p]
    lib.oracle_gemv_partials.restype = ctypes.c_int
    lib.oracle_one_shot_all_reduce.argtypes = [ctypes.c_int, ctypes.c_size_t, u16p, ip, f64p, u16p,
                                               ctypes.c_int]
    lib.oracle_one_shot_all_reduce.restype = ctypes.c_int
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.oracle_reduce_scatter.argtypes = [ctypes.c_int, ctypes.c_size_t, u16p, f64p, u16p]
    lib.oracle_reduce_scatter.restype = ctypes.c_int
    lib.oracle_gemv_reduce_scatter.argtypes = [ctypes.c_int] * 4 + [u16p, u16p, f64p, u16p, ctypes.c_int]
    lib.oracle_gemv_reduce_scatter.restype = ctypes.c_int
    lib.oracle_all_reduce_bias_rmsnorm.argtypes = [ctypes.c_int] * 3 + [u16p, u16p, u16p, ctypes.c_double,
                                                                        f64p, u16p]
    lib.oracle_all_reduce_bias_rmsnorm.restype = ctypes.c_int
    lib.oracle_gemv_bias_rmsnorm.argtypes = [ctypes.c_int] * 4 + [u16p, u16p, u16p, u16p, ctypes.c_double,
                                                                  f64p, u16p, ctypes.c_int]
    lib.oracle_gemv_bias_rmsnorm.restype = ctypes.c_int
    lib.oracle_tile_reduce.argtypes = [ctypes.c_int, ctypes.c_size_t, u16p, ctypes.c_size_t, u16p, ctypes.c_int, szp,
                                       ctypes.c_size_t, ip, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                       ctypes.c_size_t, f64p]
    lib.oracle_tile_reduce.restype = ctypes.c_int
    return lib


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.lib = _bind(ctypes.CDLL(path))

    # -------------------------------------------------------------- bf16
    def bf16_value(self, words) -> np.ndarray:
        w = np.asarray(words, dtype=np.uint16)
        f = np.vectorize(self.lib.oracle_bf16_value, otypes=[np.float64])
        return f(w) if w.size else w.astype(np.float64)

    def bf16_round(self, values) -> np.ndarray:
        v = np.asarray(values, dtype=np.float64)
        f = np.vectorize(self.lib.oracle_bf16_round, otypes=[np.uint16])
        return f(v) if v.size else v.astype(np.uint16)

    # -------------------------------------------------------------- GEMV
    def gemv_all_reduce(self, W: np.ndarray, x: np.ndarray, order=None, threads: int | None = None):
        """W: (R, N, K_r) bf16 words, x: (R, B, K_r).  Returns (y_ref fp64
        (B, N), y bf16 words (R, B, N) -- one identical replica per rank)."""
        W = np.ascontiguousarray(W, dtype=np.uint16)
        x = np.ascontiguousarray(x, dtype=np.uint16)
        R, N, Kr = W.shape
        B = x.shape[1]
        assert x.shape == (R, B, Kr)
        y_ref = np.empty((B, N), dtype=np.float64)
        y = np.empty((R, B, N), dtype=np.uint16)
        ordp = None
        if order is not None:
            o = np.ascontiguousarray(order, dtype=np.int32)
            ordp = o.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
        rc = self.lib.oracle_gemv_all_reduce(
            R, N, R * Kr, B, _u16(W), _u16(x), ordp, _f64(y_ref), _u16(y), threads or _threads())
        if rc != 0:
            raise ValueError(f"oracle_gemv_all_reduce returned {rc}")
        return y_ref, y

    def gemv_element(self, W: np.ndarray, x: np.ndarray, b: int, n: int) -> float:
        W = np.ascontiguousarray(W, dtype=np.uint16)
        x = np.ascontiguousarray(x, dtype=np.uint16)
        R, N, Kr = W.shape
        B = x.shape[1]
        return self.lib.oracle_gemv_element(R, N, R * Kr, B, _u16(W), _u16(x), b, n)

    def gemv_partials(self, W: np.ndarray, x: np.ndarray, b: int, n: int) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint16)
        x = np.ascontiguousarray(x, dtype=np.uint16)
        R, N, Kr = W.shape
        B = x.shape[1]
        out = np.empty(R, dtype=np.float64)
        rc = self.lib.oracle_gemv_partials(R, N, R * Kr, B, _u16(W), _u16(x), b, n, _f64(out))
        if rc != 0:
            raise ValueError("oracle_gemv_partials: bad arguments")
        return out

    # -------------------------------------------------------- all-reduce
    def one_shot_all_reduce(self, inp: np.ndarray, order=None, threads: int | None = None):
        """inp: (R, n) bf16 words.  Returns (ref fp64 (n,), out bf16 (R, n))."""
        inp = np.ascontiguousarray(inp, dtype=np.uint16)
        R, n = inp.shape
        ref = np.empty(n, dtype=np.float64)
        out = np.empty((R, n), dtype=np.uint16)
        ordp = None
        if order is not None:
            o = np.ascontiguousarray(order, dtype=np.int32)
            ordp = o.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
        rc = self.lib.oracle_one_shot_all_reduce(R, n, _u16(inp), ordp, _f64(ref), _u16(out),
                                                 threads or _threads())
        if rc != 0:
            raise ValueError(f"oracle_one_shot_all_reduce returned {rc}")
        return ref, out

    def reduce_scatter(self, inp: np.ndarray):
        """inp: (R, n) bf16 words, n % R == 0.  Returns (ref fp64 (n,), out
        bf16 (R, n // R) -- rank s holds block s of the sum)."""
        inp = np.ascontiguousarray(inp, dtype=np.uint16)
        R, n = inp.shape
        ref = np.empty(n, dtype=np.float64)
        out = np.empty((R, n // R if R else 0), dtype=np.uint16)
        rc = self.lib.oracle_reduce_scatter(R, n, _u16(inp), _f64(ref), _u16(out))
        if rc != 0:
            raise ValueError(f"oracle_reduce_scatter returned {rc}")
        return ref, out

    def gemv_reduce_scatter(self, W: np.ndarray, x: np.ndarray, threads: int | None = None):
        """W (R, N, K_r), x (R, B, K_r), B % R == 0.  Returns (y_ref fp64
        (B, N), out bf16 (R, B // R, N) -- rank s holds rows s*B/R ...)."""
        W = np.ascontiguousarray(W, dtype=np.uint16)
        x = np.ascontiguousarray(x, dtype=np.uint16)
        R, N, Kr = W.shape
        B = x.shape[1]
        y_ref = np.empty((B, N), dtype=np.float64)
        out = np.empty((R, B // R, N), dtype=np.uint16)
        rc = self.lib.oracle_gemv_reduce_scatter(R, N, R * Kr, B, _u16(W), _u16(x), _f64(y_ref), _u16(out),
                                                 threads or _threads())
        if rc != 0:
            raise ValueError(f"oracle_gemv_reduce_scatter returned {rc}")
        return y_ref, out

    def all_reduce_bias_rmsnorm(self, inp: np.ndarray, bias=None, gamma=None, eps: float = 1e-6):
        """inp (R, rows, H) bf16 words; bias, gamma (H,) words or None.
        Returns (ref fp64 (rows, H), out bf16 (R, rows, H))."""
        inp = np.ascontiguousarray(inp, dtype=np.uint16)
        R, rows, H = inp.shape
        bp, gp = _opt_u16(bias, H), _opt_u16(gamma, H)
        ref = np.empty((rows, H), dtype=np.float64)
        out = np.empty((R, rows, H), dtype=np.uint16)
        rc = self.lib.oracle_all_reduce_bias_rmsnorm(R, rows, H, _u16(inp), bp[1], gp[1], eps, _f64(ref),
                                                     _u16(out))
        if rc != 0:
            raise ValueError(f"oracle_all_reduce_bias_rmsnorm returned {rc}")
        return ref, out

    def gemv_bias_rmsnorm(self, W: np.ndarray, x: np.ndarray, bias=None, gamma=None, eps: float = 1e-6,
                          threads: int | None = None):
        """The fused layer followed by bias + RMSNorm over each batch row's N
        outputs.  Returns (y_ref fp64 (B, N), y bf16 (R, B, N))."""
        W = np.ascontiguousarray(W, dtype=np.uint16)
        x = np.ascontiguousarray(x, dtype=np.uint16)
        R, N, Kr = W.shape
        B = x.shape[1]
        bp, gp = _opt_u16(bias, N), _opt_u16(gamma, N)
        y_ref = np.empty((B, N), dtype=np.float64)
        y = np.empty((R, B, N), dtype=np.uint16)
        rc = self.lib.oracle_gemv_bias_rmsnorm(R, N, R * Kr, B, _u16(W), _u16(x), bp[1], gp[1], eps,
                                               _f64(y_ref), _u16(y), threads or _threads())
        if rc != 0:
            raise ValueError(f"oracle_gemv_bias_rmsnorm returned {rc}")
        return y_ref, y

    def tile_reduce(self, slots_in: np.ndarray, slots_out: np.ndarray, in_offs, out_off: int, roots,
                    rows: int, cols: int, ld_in: int, ld_out: int):
        """slots_in (R, in_slot), slots_out (R, out_slot): bf16 words; tile i
        starts at element in_offs[i] of every input slot and is summed into
        slot roots[i]'s output tile at out_off.  Returns (ref fp64 (ntiles,
        rows, cols), the updated copy of slots_out)."""
        slots_in = np.ascontiguousarray(slots_in, dtype=np.uint16)
        out = np.array(slots_out, dtype=np.uint16, copy=True, order="C")
        R, in_slot = slots_in.shape
        if out.ndim != 2 or out.shape[0] != R:
            raise ValueError(f"slots_out must be ({R}, out_slot), got {out.shape}")
        offs = np.ascontiguousarray(in_offs, dtype=np.uint64)
        rts = np.ascontiguousarray(roots, dtype=np.int32)
        nt = len(offs)
        ref = np.empty((nt, rows, cols), dtype=np.float64)
        rc = self.lib.oracle_tile_reduce(R, in_slot, _u16(slots_in), out.shape[1], _u16(out), nt,
                                         offs.ctypes.data_as(ctypes.POINTER(ctypes.c_size_t)), out_off,
                                         rts.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), rows, cols, ld_in,
                                         ld_out, _f64(ref))
        if rc != 0:
            raise ValueError(f"oracle_tile_reduce returned {rc}")
        return ref, out


def _u16(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _opt_u16(a, n):
    """(array kept alive, pointer) for an optional bf16 vector of length n."""
    if a is None:
        return None, None
    v = np.ascontiguousarray(a, dtype=np.uint16)
    if v.shape != (n,):
        raise ValueError(f"expected a vector of {n} bf16 words, got shape {v.shape}")
    return v, _u16(v)


def _f64(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def load() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def gemv_all_reduce(W, x, order=None, threads=None):
    return load().gemv_all_reduce(W, x, order, threads)


def gemv_element(W, x, b, n):
    return load().gemv_element(W, x, b, n)


def gemv_partials(W, x, b, n):
    return load().gemv_partials(W, x, b, n)


def one_shot_all_reduce(inp, order=None, threads=None):
    return load().one_shot_all_reduce(inp, order, threads)


def bf16_value(words):
    return load().bf16_value(words)


def bf16_round(values):
    return load().bf16_round(values)


def reduce_scatter(inp):
    return load().reduce_scatter(inp)


def gemv_reduce_scatter(W, x, threads=None):
    return load().gemv_reduce_scatter(W, x, threads)


def all_reduce_bias_rmsnorm(inp, bias=None, gamma=None, eps=1e-6):
    return load().all_reduce_bias_rmsnorm(inp, bias, gamma, eps)


def gemv_bias_rmsnorm(W, x, bias=None, gamma=None, eps=1e-6, threads=None):
    return load().gemv_bias_rmsnorm(W, x, bias, gamma, eps, threads)


def tile_reduce(slots_in, slots_out, in_offs, out_off, roots, rows, cols, ld_in, ld_out):
    return load().tile_reduce(slots_in, slots_out, in_offs, out_off, roots, rows, cols, ld_in, ld_out)

