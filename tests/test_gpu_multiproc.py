"""Multi-process handles on the GPU: R processes, one rank each, their slots
mapped into one another (symm_mp_alloc / symm_mp_import), each launching its
own rank's share of the call.  The ranks' outputs must be bit-identical to
one another and agree with the oracle (small-integer inputs bit-exact); a rank
that leaves between calls makes the others' next call report SYMM_EPROTO,
and nothing hangs.  The processes share the one GPU: no kernel waits on
another process's kernel (the last arriver of a tile reduces it)."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

import collective_split_gemv_gb300 as csg
import oracle
import synth
from gpu_common import require_gpu
from helpers import tolerance_ratio, words_to_f64

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
N, KR, B, N_AR = 1000, 512, 4, 3 * 4096 + 24


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(scenario, world, tmp_path, timeout=300):
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    procs = [subprocess.Popen([sys.executable, os.path.join(HERE, "mp_worker.py"), scenario, str(r), str(world),
                               str(tmp_path)], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
             for r in range(world)]
    res = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise AssertionError(f"{scenario}: a rank did not finish in {timeout} s")
        res.append((p.returncode, out, err))
    for r, (rc, out, err) in enumerate(res):
        assert rc == 0, (scenario, r, rc, err[-3000:])
    return [dict(np.load(os.path.join(tmp_path, f"out{r}.npz"))) for r in range(world)]


@pytest.mark.parametrize("world", [2, 4, 8])
def test_multiprocess_gemv_all_reduce(world, tmp_path):
    outs = _run("gemv", world, tmp_path)
    R = world
    rng = np.random.default_rng(7)
    Wi = rng.integers(-8, 9, size=(R, N, KR)).astype(np.float32)
    xi = rng.integers(-8, 9, size=(R, B, KR)).astype(np.float32)
    cases = {"int": (synth.round_bf16(Wi.astype(np.float64)), synth.round_bf16(xi.astype(np.float64))),
             "normal": synth.gemv_inputs(R, N, R * KR, B, seed=11, w_std=0.02, x="normal")}
    for kind, (W, x) in cases.items():
        y_ref, y_or = oracle.gemv_all_reduce(W, x)
        # every rank's copy and every repeat of a kernel: the same bits (the
        # packed weight's call runs the persistent kernel on the same values);
        # the two kernels sum in different orders, so only exact inputs give
        # both the same bits
        groups = [[f"{kind}_p1_{i}" for i in range(3)], [f"{kind}_p4_{i}" for i in range(3)] + [kind + "_packed"]]
        for keys in groups:
            first = outs[0][keys[0]]
            for k in keys:
                for r in range(R):
                    assert np.array_equal(outs[r][k], first), (kind, k, r)
            got = first.reshape(B, N)
            if kind == "int":
                assert np.array_equal(got, y_or[0])
            assert tolerance_ratio(words_to_f64(got), y_ref) <= 1.0
        got = outs[0][kind + "_p1_0"].reshape(B, N)   # the reduce-scatter call ran on the CUDA-core kernel
        if B % R == 0:
            y_ref_rs, y_or_rs = oracle.gemv_reduce_scatter(W, x)
            for r in range(R):
                rows = slice(r * (B // R), (r + 1) * (B // R))
                got_rs = outs[r][kind + "_rs"].reshape(B // R, N)
                assert np.array_equal(got_rs, got[rows]), (kind, r)
    for r in range(R):
        assert int(outs[r]["status"][0]) == csg.SYMM_OK, outs[r]["status"]
        assert int(outs[r]["guards"][0]) == csg.SYMM_OK


@pytest.mark.parametrize("world", [2, 4, 8])
def test_multiprocess_one_shot_all_reduce(world, tmp_path):
    outs = _run("oneshot", world, tmp_path)
    for i in range(2):
        inp = synth.allreduce_inputs(world, N_AR, 20 + i)
        ref, want = oracle.one_shot_all_reduce(inp)
        for r in range(world):
            got = outs[r][f"ar_{i}"]
            assert np.array_equal(got, outs[0][f"ar_{i}"]), (i, r)
            assert tolerance_ratio(words_to_f64(got), ref) <= 1.0
    for r in range(world):
        assert int(outs[r]["status"][0]) == csg.SYMM_OK


@pytest.mark.parametrize("world,leaver", [(3, 2), (5, 4), (3, 0)])
def test_rank_leaving_between_calls_is_reported(world, leaver, tmp_path):
    """A rank leaves after the first call (the last one, or rank 0, whose pad
    holds the tile counters every rank shares); the others make one more
    call, which finishes (no kernel waits for the missing contributions), and
    after their barrier each reports SYMM_EPROTO naming the rank that left,
    whose launch count fell behind theirs.  They report one after another,
    so every report after the first reads the pads of survivors that have
    already reset theirs: a reset must keep a rank's launch count."""
    assert leaver in (0, world - 1)
    outs = _run("leave0" if leaver == 0 else "leave", world, tmp_path, timeout=180)
    W, x = synth.gemv_inputs(world, N, world * KR, B, seed=12, w_std=0.02, x="normal")
    y_ref, _ = oracle.gemv_all_reduce(W, x)
    for r in range(world):
        assert int(outs[r]["first_status"][0]) == csg.SYMM_OK
        assert tolerance_ratio(words_to_f64(outs[r]["first"].reshape(B, N)), y_ref) <= 1.0
    assert int(outs[leaver]["role"][0]) == 1
    for r in range(world):
        if r == leaver:
            continue
        assert int(outs[r]["role"][0]) == 0
        assert int(outs[r]["status"][0]) == csg.SYMM_EPROTO, outs[r]["status"]
        assert int(outs[r]["status"][1]) == leaver, outs[r]["status"]
