"""The C-ABI library loads and exports every declared entry point; host-only
validation works without a GPU (no compute calls here)."""
from __future__ import annotations

import os
import re

import pytest

import collective_split_gemv_gb300 as csg
from collective_split_gemv_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "symm_gemv.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return csg.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("symm_alloc", "symm_rendezvous", "one_shot_all_reduce", "gemv_all_reduce",
                     "symm_status", "symm_free", "symm_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in csg.EXPORTED, f"{name} has no Python binding"


def _header_enum(prefix):
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(" + prefix + r"\w*)\s*=\s*(-?\d+)", src)}


def test_option_and_status_codes_match_the_binding():
    """The binding's option numbers and status codes are the header's."""
    for prefix in ("SYMM_OPT_", "SYMM_E", "SYMM_OK"):
        declared = _header_enum(prefix)
        assert declared, prefix
        for name, value in declared.items():
            assert getattr(csg, name) == value, name
    opts = _header_enum("SYMM_OPT_")
    assert len(set(opts.values())) == len(opts)   # no two options share a number


def test_layout_arithmetic(lib):
    stride, total = csg.symm_layout(8, 1000, 4096, 4096)
    assert stride % (2 << 20) == 0 and stride >= 1000 + 4096 + 4096 + 3 * 4096
    assert total == 8 * stride
    stride2, _ = csg.symm_layout(1, 5 << 20, 0, 65536)
    assert stride2 == 6 << 20


@pytest.mark.parametrize("args,code", [
    ((0, 1024, 0, 4096), csg.SYMM_EINVAL),
    ((65, 1024, 0, 4096), csg.SYMM_EINVAL),
    ((2, 0, 0, 4096), csg.SYMM_EINVAL),
    ((2, 1024, 0, 100), csg.SYMM_EINVAL),
])
def test_layout_rejects(lib, args, code):
    with pytest.raises(csg.SymmError) as e:
        csg.symm_layout(*args)
    assert e.value.code == code
    assert csg.symm_last_error()


def test_null_handle_is_rejected(lib):
    for call in (lambda: csg.gemv_all_reduce(None, 0, 0, 0, 2, 8, 16, 1),
                 lambda: csg.one_shot_all_reduce(None, 0, 0, 2, 8),
                 lambda: csg.symm_status(None),
                 lambda: csg.symm_set_option(None, 1, 0),
                 lambda: csg.gemv_reduce_scatter(None, 0, 0, 0, 2, 8, 16, 2),
                 lambda: csg.gemv_all_reduce_bias_rmsnorm(None, 0, 0, None, None, 0, 2, 8, 16, 1, 1e-6),
                 lambda: csg.reduce_scatter(None, 0, 0, 2, 8),
                 lambda: csg.two_shot_all_reduce(None, 0, 0, 2, 8),
                 lambda: csg.all_reduce_bias_rmsnorm(None, 0, None, None, 0, 2, 1, 8, 1e-6),
                 lambda: csg.tile_reduce(None, 0, 0, 0, 4, 4, 4, 4),
                 lambda: csg.multi_root_tile_reduce(None, [0], 0, [0], 4, 4, 4, 4),
                 lambda: csg.symm_copy_to_slots(None, 0, 0, 16, 1),
                 lambda: csg.symm_copy_from_slots(None, 0, 0, 16, 1),
                 lambda: csg.symm_pack_w(None, 0, 0, 2, 8, 16),
                 lambda: csg.symm_release_w(None, 0)):
        with pytest.raises(csg.SymmError) as e:
            call()
        assert e.value.code == csg.SYMM_EINVAL
    csg.symm_free(None)   # freeing NULL is a no-op


@pytest.mark.parametrize("R,N,K", [(1, 1, 8), (2, 128, 128), (2, 129, 144), (8, 8192, 28672), (4, 0, 64),
                                   (3, 7, 0), (8, 16384, 53248)])
def test_packed_weight_size(lib, R, N, K):
    # one 16 KB block per 128 rows x 64 columns of W_r, rounded up, plus the zero block
    Kr = K // R
    blocks = ((N + 127) // 128) * ((Kr + 63) // 64) + 1
    assert csg.symm_packed_w_bytes(R, N, K) == blocks * 16384


@pytest.mark.parametrize("args", [(0, 8, 8), (65, 8, 8), (2, -1, 16), (2, 8, -2), (2, 8, 9), (2, 8, 12)])
def test_packed_weight_size_rejects(lib, args):
    with pytest.raises(csg.SymmError) as e:
        csg.symm_packed_w_bytes(*args)
    assert e.value.code == csg.SYMM_EINVAL


def test_alloc_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(csg.SymmError) as e:
        csg.symm_alloc(2, 1024, 1024, 4096)
    assert e.value.code in (csg.SYMM_ECUDA, csg.SYMM_ENOMEM)


def test_library_is_sm103a_only():
    assert any("compute_103a,code=sm_103a" in f for f in _build.NVCC_FLAGS)
    assert not any("sm_90" in f or "sm_100" in f for f in _build.NVCC_FLAGS)


def test_timeline_variant_builds_with_the_same_boundary():
    """The timeline build (per-CTA phase stamps, -DSYMM_TIMELINE) compiles and
    exports every entry point the product library does."""
    import ctypes

    tl = ctypes.CDLL(_build.build(variant="timeline"))
    for name in _declared_functions():
        assert hasattr(tl, name), name
