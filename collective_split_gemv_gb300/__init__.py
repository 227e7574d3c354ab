"""Python binding of the symmetric-slot GEMV + one-shot all-reduce C ABI.

The functions below carry the names of ``include/symm_gemv.h`` and only
marshal arguments into ``libsymm_gemv.so``; every step of the computation runs
in that library's CUDA kernels.  Non-zero return codes raise ``SymmError``
(its ``code`` is the SYMM_E* value, its message the library's last error).

Pointers are device addresses as Python ints (for example
``tensor.data_ptr()``); streams are CUDA stream handles as ints, objects with a
``cuda_stream`` attribute (``torch.cuda.Stream``), or None for the legacy
default stream.

There is no fallback: if the library has not been built, importing works but
the first call raises.  Build it with ``__graft_entry__.build()``.

``SYMM_GEMV_VARIANT=timeline`` in the environment loads the timeline build of
the same library instead (kernels with %globaltimer phase stamps, see
``symm_set_timeline``); it is built by ``_build.build(variant="timeline")``.
"""
from __future__ import annotations

import ctypes
import os

from ._build import lib_path as _lib_path

SYMM_OK = 0
SYMM_EINVAL = -1
SYMM_ENOMEM = -2
SYMM_ECUDA = -3
SYMM_ERANGE = -4
SYMM_EPROTO = -5
SYMM_ECORRUPT = -6

SYMM_MAX_RANKS = 64
SYMM_MAX_BATCH = 16

SYMM_OPT_GEMV_PATH = 1
SYMM_OPT_TILE_ORDER = 2
SYMM_OPT_SK_SLABS = 3
SYMM_OPT_SK_ENGINE = 4
SYMM_OPT_SK_CTAS_PER_SM = 5
SYMM_OPT_SK_GRID = 6
SYMM_OPT_DYN_SPLITS = 7
SYMM_OPT_NORM_PDL = 8
SYMM_OPT_CHAIN = 9
SYMM_OPT_AR_CTAS_PER_SM = 10
SYMM_OPT_AR_KERNEL = 11
SYMM_OPT_COPY_ENGINE = 12
SYMM_OPT_UNFUSED = 13
SYMM_OPT_DYN_CLUSTER = 14
AR_KERNEL_AUTO, AR_KERNEL_PER_THREAD, AR_KERNEL_STAGED = 0, 1, 2   # auto is the per-thread kernel

GEMV_PATH_AUTO, GEMV_PATH_FFMA, GEMV_PATH_DYN, GEMV_PATH_CLUSTER = 0, 1, 4, 5   # paths 2 and 3 were retired
TIMELINE_SLOTS = 16   # 64-bit words per CTA row of a timeline buffer

EXPORTED = ("symm_layout", "symm_alloc", "symm_mp_alloc", "symm_mp_import", "symm_rendezvous", "one_shot_all_reduce",
            "gemv_all_reduce", "symm_status", "symm_check_guards", "symm_set_option",
            "symm_info", "symm_gemv_plan", "gemv_all_reduce_noalloc", "gemv_reduce_scatter",
            "gemv_all_reduce_bias_rmsnorm", "reduce_scatter", "two_shot_all_reduce",
            "all_reduce_bias_rmsnorm", "tile_reduce", "multi_root_tile_reduce", "symm_copy_to_slots",
            "symm_copy_from_slots", "symm_packed_w_bytes", "symm_pack_w", "symm_release_w", "symm_set_timeline",
            "symm_free", "symm_last_error")

_lib = None


class SymmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class SymmInfo(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("device", ctypes.c_int), ("stride", ctypes.c_size_t),
                ("slot_bytes", ctypes.c_size_t), ("scratch_bytes", ctypes.c_size_t),
                ("signal_pad_bytes", ctypes.c_size_t), ("max_tiles", ctypes.c_int)]


class GemvPlan(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int) for k in ("path", "engine", "slabs", "rows_per_tile", "tiles", "splits",
                                            "grid", "parts_max", "kblocks", "ctas_per_sm", "cluster")]


def library_variant() -> str:
    """'' for the product library, 'timeline' for the stamped build."""
    v = os.environ.get("SYMM_GEMV_VARIANT", "")
    return "timeline" if v == "timeline" else ""


def library_path() -> str:
    return _lib_path(library_variant())


def lib() -> ctypes.CDLL:
    """The loaded ``libsymm_gemv.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: the CUDA library has not been built "
                               "(run __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.symm_layout.argtypes = [i, sz, sz, sz, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.symm_alloc.argtypes = [i, sz, sz, sz, vp, sz, ctypes.POINTER(vp)]
        L.symm_mp_alloc.argtypes = [i, i, sz, sz, sz, ctypes.POINTER(vp), ctypes.POINTER(i)]
        L.symm_mp_import.argtypes = [vp, i, i]
        L.symm_rendezvous.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(sz)]
        L.one_shot_all_reduce.argtypes = [vp, vp, vp, i, sz, vp]
        L.gemv_all_reduce.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.symm_status.argtypes = [vp, vp, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i)]
        L.symm_check_guards.argtypes = [vp, ctypes.POINTER(i), ctypes.POINTER(i)]
        L.symm_set_option.argtypes = [vp, i, i]
        L.symm_info.argtypes = [vp, ctypes.POINTER(SymmInfo)]
        L.symm_gemv_plan.argtypes = [vp, i, i, i, ctypes.POINTER(GemvPlan)]
        L.gemv_all_reduce_noalloc.argtypes = [vp, vp, vp, sz, i, i, i, i, vp]
        ll = ctypes.c_longlong
        f32 = ctypes.c_float
        L.gemv_reduce_scatter.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.gemv_all_reduce_bias_rmsnorm.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f32, vp]
        L.reduce_scatter.argtypes = [vp, vp, vp, i, sz, vp]
        L.two_shot_all_reduce.argtypes = [vp, vp, vp, i, sz, vp]
        L.all_reduce_bias_rmsnorm.argtypes = [vp, vp, vp, vp, vp, i, i, i, f32, vp]
        L.tile_reduce.argtypes = [vp, vp, vp, i, i, i, ll, ll, vp]
        L.multi_root_tile_reduce.argtypes = [vp, ctypes.POINTER(vp), vp, ctypes.POINTER(i), i, i, i, ll, ll, vp]
        L.symm_copy_to_slots.argtypes = [vp, vp, vp, sz, i, vp]
        L.symm_copy_from_slots.argtypes = [vp, vp, vp, sz, i, vp]
        L.symm_packed_w_bytes.argtypes = [i, i, i, ctypes.POINTER(sz)]
        L.symm_pack_w.argtypes = [vp, vp, vp, i, i, i, vp]
        L.symm_release_w.argtypes = [vp, vp]
        L.symm_set_timeline.argtypes = [vp, vp, sz]
        L.symm_free.argtypes = [vp]
        L.symm_last_error.argtypes = []
        L.symm_last_error.restype = ctypes.c_char_p
        for name in EXPORTED[:-1]:
            getattr(L, name).restype = i
        _lib = L
    return _lib


def symm_last_error() -> str:
    return lib().symm_last_error().decode(errors="replace")


def _check(rc: int) -> int:
    if rc != SYMM_OK:
        raise SymmError(rc, symm_last_error())
    return rc


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(0)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(int(stream.cuda_stream))
    return ctypes.c_void_p(int(stream))


def _vp(p) -> ctypes.c_void_p:
    return ctypes.c_void_p(int(p) if p is not None else 0)


def symm_layout(R: int, slot_bytes: int, scratch_bytes: int, signal_pad_bytes: int):
    """-> (stride, total_bytes)"""
    stride, total = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().symm_layout(R, slot_bytes, scratch_bytes, signal_pad_bytes,
                             ctypes.byref(stride), ctypes.byref(total)))
    return stride.value, total.value


def symm_alloc(R: int, slot_bytes: int, scratch_bytes: int, signal_pad_bytes: int,
               backing: int | None = None, backing_bytes: int = 0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().symm_alloc(R, slot_bytes, scratch_bytes, signal_pad_bytes, _vp(backing),
                            backing_bytes, ctypes.byref(h)))
    return h


def symm_mp_alloc(R: int, rank: int, slot_bytes: int, scratch_bytes: int, signal_pad_bytes: int):
    """This process's rank of a multi-process handle: its slot allocated and
    mapped, the others not yet.  -> (handle, fd): fd is the POSIX descriptor
    of the slot's allocation, to be sent to every other rank's process (see
    ``multiproc.exchange_fds``) and closed by this process once they have it."""
    h = ctypes.c_void_p()
    fd = ctypes.c_int(-1)
    _check(lib().symm_mp_alloc(R, rank, slot_bytes, scratch_bytes, signal_pad_bytes, ctypes.byref(h),
                               ctypes.byref(fd)))
    return h, fd.value


def symm_mp_import(h, peer: int, fd: int) -> None:
    """Maps rank `peer`'s slot (its process's descriptor, received by this one)."""
    _check(lib().symm_mp_import(h, peer, fd))


def symm_rendezvous(h):
    """-> (slot_ptrs[R], signal_pad_ptrs[R], stride)"""
    info = symm_info(h)
    R = info["R"]
    slots = (ctypes.c_void_p * R)()
    pads = (ctypes.c_void_p * R)()
    stride = ctypes.c_size_t()
    _check(lib().symm_rendezvous(h, slots, pads, ctypes.byref(stride)))
    return [int(p or 0) for p in slots], [int(p or 0) for p in pads], stride.value


def one_shot_all_reduce(h, inp: int, out: int, R: int, n: int, stream=None) -> None:
    _check(lib().one_shot_all_reduce(h, _vp(inp), _vp(out), R, n, _stream(stream)))


def gemv_all_reduce(h, W_r: int, x_r: int, y: int, R: int, N: int, K: int, B: int, stream=None) -> None:
    _check(lib().gemv_all_reduce(h, _vp(W_r), _vp(x_r), _vp(y), R, N, K, B, _stream(stream)))


def gemv_reduce_scatter(h, W_r: int, x_r: int, y: int, R: int, N: int, K: int, B: int, stream=None) -> None:
    _check(lib().gemv_reduce_scatter(h, _vp(W_r), _vp(x_r), _vp(y), R, N, K, B, _stream(stream)))


def gemv_all_reduce_bias_rmsnorm(h, W_r: int, x_r: int, bias, gamma, y: int, R: int, N: int, K: int, B: int,
                                 eps: float, stream=None) -> None:
    _check(lib().gemv_all_reduce_bias_rmsnorm(h, _vp(W_r), _vp(x_r), _vp(bias), _vp(gamma), _vp(y), R, N, K, B,
                                              float(eps), _stream(stream)))


def reduce_scatter(h, inp: int, out: int, R: int, n: int, stream=None) -> None:
    _check(lib().reduce_scatter(h, _vp(inp), _vp(out), R, n, _stream(stream)))


def two_shot_all_reduce(h, inp: int, out: int, R: int, n: int, stream=None) -> None:
    _check(lib().two_shot_all_reduce(h, _vp(inp), _vp(out), R, n, _stream(stream)))


def all_reduce_bias_rmsnorm(h, inp: int, bias, gamma, out: int, R: int, rows: int, H: int, eps: float,
                            stream=None) -> None:
    _check(lib().all_reduce_bias_rmsnorm(h, _vp(inp), _vp(bias), _vp(gamma), _vp(out), R, rows, H, float(eps),
                                         _stream(stream)))


def tile_reduce(h, in_tile: int, out_tile: int, root: int, rows: int, cols: int, ld_in: int, ld_out: int,
                stream=None) -> None:
    _check(lib().tile_reduce(h, _vp(in_tile), _vp(out_tile), root, rows, cols, ld_in, ld_out, _stream(stream)))


def multi_root_tile_reduce(h, in_tiles, out_tile: int, roots, rows: int, cols: int, ld_in: int, ld_out: int,
                           stream=None) -> None:
    nt = len(in_tiles)
    if len(roots) != nt:
        raise ValueError("in_tiles and roots differ in length")
    tiles = (ctypes.c_void_p * max(nt, 1))(*[int(p) for p in in_tiles])
    rts = (ctypes.c_int * max(nt, 1))(*[int(r) for r in roots])
    _check(lib().multi_root_tile_reduce(h, tiles, _vp(out_tile), rts, nt, rows, cols, ld_in, ld_out,
                                        _stream(stream)))


def symm_copy_to_slots(h, dst: int, src: int, bytes_per_rank: int, nranks: int, stream=None) -> None:
    """Block r of the contiguous buffer at `src` -> dst + r * stride (one strided copy)."""
    _check(lib().symm_copy_to_slots(h, _vp(dst), _vp(src), bytes_per_rank, nranks, _stream(stream)))


def symm_copy_from_slots(h, dst: int, src: int, bytes_per_rank: int, nranks: int, stream=None) -> None:
    """src + r * stride -> block r of the contiguous buffer at `dst` (one strided copy)."""
    _check(lib().symm_copy_from_slots(h, _vp(dst), _vp(src), bytes_per_rank, nranks, _stream(stream)))


def symm_packed_w_bytes(R: int, N: int, K: int) -> int:
    """Bytes per slot of the packed form of an N x (K/R) W_r."""
    out = ctypes.c_size_t()
    _check(lib().symm_packed_w_bytes(R, N, K, ctypes.byref(out)))
    return out.value


def symm_pack_w(h, W_r: int, Wp: int, R: int, N: int, K: int, stream=None) -> None:
    """Packs every slot's row-major W_r into Wp and registers Wp with the handle."""
    _check(lib().symm_pack_w(h, _vp(W_r), _vp(Wp), R, N, K, _stream(stream)))


def symm_release_w(h, Wp: int) -> None:
    _check(lib().symm_release_w(h, _vp(Wp)))


def symm_set_timeline(h, buf, nbytes: int) -> None:
    """Diagnostics: per-CTA phase stamps of later calls into `buf` (device
    pointer, rows of TIMELINE_SLOTS uint64); the timeline build only.  None
    switches it off."""
    _check(lib().symm_set_timeline(h, _vp(buf) if buf else None, nbytes if buf else 0))


def symm_status(h, stream=None):
    """-> (code, rank, tile); code is SYMM_OK or SYMM_EPROTO."""
    code, rank, tile = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().symm_status(h, _stream(stream), ctypes.byref(code), ctypes.byref(rank),
                             ctypes.byref(tile)))
    return code.value, rank.value, tile.value


def symm_check_guards(h):
    """-> (rc, bad_rank, bad_band); rc is SYMM_OK or SYMM_ECORRUPT."""
    rank, band = ctypes.c_int(), ctypes.c_int()
    rc = lib().symm_check_guards(h, ctypes.byref(rank), ctypes.byref(band))
    if rc not in (SYMM_OK, SYMM_ECORRUPT):
        _check(rc)
    return rc, rank.value, band.value


def symm_set_option(h, option: int, value: int) -> None:
    _check(lib().symm_set_option(h, option, value))


def symm_info(h) -> dict:
    info = SymmInfo()
    _check(lib().symm_info(h, ctypes.byref(info)))
    return {k: getattr(info, k) for k, _ in SymmInfo._fields_}


def symm_gemv_plan(h, N: int, K: int, B: int) -> dict:
    """Kernel and launch geometry gemv_all_reduce would use (no launch)."""
    plan = GemvPlan()
    _check(lib().symm_gemv_plan(h, N, K, B, ctypes.byref(plan)))
    return {k: getattr(plan, k) for k, _ in GemvPlan._fields_}


def gemv_all_reduce_noalloc(W_r: int, x_r: int, y: int, stride: int, R: int, N: int, K: int, B: int,
                            stream=None) -> None:
    """The fused call for callers that cannot allocate device memory: works on
    caller-owned tensors (rank r at ptr + r * stride) with the library's fixed
    16 MiB working array instead of a handle."""
    _check(lib().gemv_all_reduce_noalloc(_vp(W_r), _vp(x_r), _vp(y), stride, R, N, K, B, _stream(stream)))


def symm_free(h) -> None:
    _check(lib().symm_free(h))


class DeviceView:
    """A raw device range exposed through ``__cuda_array_interface__`` so that
    ``torch.as_tensor(view, device='cuda')`` aliases slot memory."""

    def __init__(self, ptr: int, shape, typestr: str = "|u1"):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}
