"""Build of the in-tree CUDA library ``libsymm_gemv.so`` (sm_103a only).

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file.  The CUDA runtime is linked dynamically so
that the process shares one runtime (and one primary context) with PyTorch.

Variant ``timeline`` (``build(variant="timeline")``) is the same library with
the kernels' %globaltimer phase stamps compiled in (``-DSYMM_TIMELINE``), as
``libsymm_gemv_timeline.so``; the binding loads it instead of the product
library when ``SYMM_GEMV_VARIANT=timeline`` is set.  It serves per-phase
launch timelines (``python -m collective_split_gemv_gb300.timeline``).
"""
from __future__ import annotations

import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libsymm_gemv.so")
VARIANTS = {
    "": (BUILD_DIR, LIB_PATH, ()),
    "timeline": (os.path.join(HERE, "_build_timeline"), os.path.join(HERE, "libsymm_gemv_timeline.so"),
                 ("-DSYMM_TIMELINE=1",)),
}


def lib_path(variant: str = "") -> str:
    return VARIANTS[variant][1]

SOURCES = ["symm_runtime.cu", "allreduce.cu", "gemv_ffma.cu", "gemv_dyn.cu", "gemv_noalloc.cu", "partials_ar.cu", "gemv_cluster.cu",
           "tile_reduce.cu", "rmsnorm.cu", "copy_slots.cu", "pack_w.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xptxas", "-warn-spills", "-I", INCLUDE]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "symm_gemv.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(variant: str = "") -> bool:
    path = lib_path(variant)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    build_dir, out_path, variant_flags = VARIANTS[variant]
    if not force and not extra_flags and up_to_date(variant):
        return out_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *variant_flags, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
