"""Seeded random sequences of fused calls on long-lived handles, every result
checked against the oracle.

Each handle (one per rank count) runs a sequence of random cases with no
reset in between: GEMV path, form (all-reduce, reduce-scatter, bias +
RMSNorm), shape (ragged tiles, every batch width), chained or plain launch,
natural or reversed CTA order, the persistent kernel's unit ending (drawn
units or the cluster epilogue), row-major or packed weights (packed anew over
the previous packed weight), eager call or a captured CUDA graph replayed.
This exercises what the signal pad carries from one launch to the next (the
launch epoch, the flags of earlier geometries, the counters put back to zero
by each launch) far beyond the hand-picked cases.  Small-integer inputs make
the all-reduce and reduce-scatter forms bit-exact; normal inputs and the
RMSNorm form are held to the tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300 import DeviceView
from collective_split_gemv_gb300.workspace import pad_bytes_for
from gpu_common import check_gemv, require_gpu
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu

N_MAX, KR_MAX, B_MAX = 1024, 2048, 16
PATHS = [csg.GEMV_PATH_AUTO, csg.GEMV_PATH_FFMA, csg.GEMV_PATH_DYN, csg.GEMV_PATH_CLUSTER]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


class Slots:
    """One handle with fixed regions for W, x, y, bias, gamma and a packed W."""

    def __init__(self, R):
        self.R = R
        self.w_off, self.x_off = 0, N_MAX * KR_MAX * 2
        self.y_off = self.x_off + B_MAX * KR_MAX * 2
        self.bias_off = self.y_off + B_MAX * N_MAX * 2
        self.gamma_off = self.bias_off + N_MAX * 2
        self.wp_off = self.gamma_off + N_MAX * 2
        wp_max = csg.symm_packed_w_bytes(R, N_MAX, R * KR_MAX)
        self.h = csg.symm_alloc(R, self.wp_off + wp_max, 9 * 4 * B_MAX * N_MAX, pad_bytes_for(N_MAX))
        self.slots, self.pads, self.stride = csg.symm_rendezvous(self.h)
        self.dev = torch.device("cuda", torch.cuda.current_device())

    def view(self, r, off, nbytes):
        return torch.as_tensor(DeviceView(self.slots[r] + off, (nbytes,)), device=self.dev)

    def put(self, off, words):   # words (R, ...) bf16: block r into slot r
        for r in range(self.R):
            self.view(r, off, words[r].nbytes).copy_(
                torch.from_numpy(np.ascontiguousarray(words[r]).view(np.uint8).reshape(-1)))

    def get(self, off, shape):   # (R, *shape) bf16 words
        torch.cuda.synchronize()
        n = int(np.prod(shape)) * 2
        return np.stack([self.view(r, off, n).cpu().numpy().view(np.uint16).reshape(shape) for r in range(self.R)])

    def ptr(self, off):
        return self.slots[0] + off

    def close(self):
        csg.symm_free(self.h)


def _case(rng, R):
    path = PATHS[rng.integers(len(PATHS))]
    packed = bool(rng.random() < 0.4)
    if packed and rng.random() < 0.8:   # mostly a path that reads packed weights; else the rejection
        path = [csg.GEMV_PATH_AUTO, csg.GEMV_PATH_DYN][rng.integers(2)]
    B = int(rng.integers(1, B_MAX + 1))
    forms = ["all_reduce"]
    if B % R == 0:
        forms.append("reduce_scatter")
    N = int(rng.integers(1, N_MAX + 1))
    if rng.random() < 0.3:
        N = int(rng.integers(1, N_MAX // 8 + 1)) * 8
    if N % 8 == 0:
        forms.append("bias_rmsnorm")
    return dict(path=path, B=B, N=N, Kr=int(rng.integers(1, KR_MAX // 8 + 1)) * 8, form=forms[rng.integers(len(forms))],
                ints=bool(rng.random() < 0.5), chain=int(rng.integers(2)), order=int(rng.integers(2)),
                graph=bool(rng.random() < 0.2), packed=packed, engine=int(rng.integers(-1, 1)),
                dyn_cluster=int(rng.integers(-1, 2)), seed=int(rng.integers(1 << 30)))


def _inputs(c, R):
    rng = np.random.default_rng(c["seed"])
    N, Kr, B = c["N"], c["Kr"], c["B"]
    if c["ints"]:
        W = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, N, Kr)).astype(np.float64))
        x = f64_to_words_via_f32(rng.integers(-8, 9, size=(R, B, Kr)).astype(np.float64))
    else:
        W = synth.round_bf16(rng.standard_normal((R, N, Kr)) * (1.0 / np.sqrt(R * Kr)))
        x = synth.round_bf16(rng.standard_normal((R, B, Kr)))
    bias = synth.round_bf16(rng.standard_normal(N) * 0.1)
    gamma = synth.round_bf16(1.0 + rng.standard_normal(N) * 0.1)
    return W, x, bias, gamma


def _call(sl, c, s):
    R, N, K, B = sl.R, c["N"], c["Kr"] * sl.R, c["B"]
    W, x, y = sl.ptr(sl.wp_off if c["packed"] else sl.w_off), sl.ptr(sl.x_off), sl.ptr(sl.y_off)
    if c["form"] == "all_reduce":
        csg.gemv_all_reduce(sl.h, W, x, y, R, N, K, B, s)
    elif c["form"] == "reduce_scatter":
        csg.gemv_reduce_scatter(sl.h, W, x, y, R, N, K, B, s)
    else:
        csg.gemv_all_reduce_bias_rmsnorm(sl.h, W, x, sl.ptr(sl.bias_off), sl.ptr(sl.gamma_off), y, R, N, K, B,
                                         1e-6, s)


def _check(sl, c, W, x, bias, gamma):
    R, N, B = sl.R, c["N"], c["B"]
    if c["form"] == "reduce_scatter":
        got = sl.get(sl.y_off, (B // R, N))
        y_ref, want = oracle.gemv_reduce_scatter(W, x)
        if c["ints"]:
            assert np.array_equal(got, want), c
        else:
            for s_ in range(R):
                rows = slice(s_ * (B // R), (s_ + 1) * (B // R))
                assert tolerance_ratio(words_to_f64(got[s_]), y_ref[rows]) <= 1.0, c
        return
    got = sl.get(sl.y_off, (B, N))
    if c["form"] == "all_reduce":
        check_gemv(W, x, got, exact=c["ints"])
        return
    y_ref, want = oracle.gemv_bias_rmsnorm(W, x, bias, gamma, 1e-6)
    for s_ in range(1, R):
        assert np.array_equal(got[s_], got[0]), c
    assert tolerance_ratio(words_to_f64(got[0]), y_ref) <= 1.0, c
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    big = np.abs(y_ref) >= 0.1 * rms
    assert int(ulp_distance(got[0][big], want[0][big]).max(initial=0)) <= 1, c


@pytest.mark.parametrize("R,cases,seed", [(1, 40, 5), (2, 60, 1), (3, 50, 2), (4, 60, 3), (5, 40, 6), (8, 60, 4)])
def test_random_call_sequences_on_one_handle(R, cases, seed):
    rng = np.random.default_rng(seed)
    sl = Slots(R)
    try:
        s = torch.cuda.current_stream()
        ran = 0
        for i in range(cases):
            c = _case(rng, R)
            W, x, bias, gamma = _inputs(c, R)
            sl.put(sl.w_off, W)
            sl.put(sl.x_off, x)
            sl.put(sl.bias_off, bias[None].repeat(R, 0))
            sl.put(sl.gamma_off, gamma[None].repeat(R, 0))
            sl.put(sl.y_off, np.full((R, B_MAX * N_MAX), 0xFFFF, dtype=np.uint16))
            csg.symm_set_option(sl.h, csg.SYMM_OPT_GEMV_PATH, c["path"])
            csg.symm_set_option(sl.h, csg.SYMM_OPT_CHAIN, c["chain"])
            csg.symm_set_option(sl.h, csg.SYMM_OPT_TILE_ORDER, c["order"])
            csg.symm_set_option(sl.h, csg.SYMM_OPT_SK_ENGINE, c["engine"])
            csg.symm_set_option(sl.h, csg.SYMM_OPT_DYN_CLUSTER, c["dyn_cluster"])
            if c["packed"]:   # new weights packed over the last packed ones (their registration ends)
                csg.symm_pack_w(sl.h, sl.ptr(sl.w_off), sl.ptr(sl.wp_off), R, c["N"], c["Kr"] * R, s)
            torch.cuda.synchronize()
            try:
                _call(sl, c, s)                     # eager (for a graph case: set-up before the capture)
            except csg.SymmError as e:
                # a shape the chosen path cannot plan (its partials or flags do not fit), a packed
                # weight with a path other than the persistent kernel forced, or the cluster kernel
                # forced beyond its ranks or batch: not a fault
                forced = c["path"] not in (csg.GEMV_PATH_AUTO, csg.GEMV_PATH_DYN)
                cluster_out = c["path"] == csg.GEMV_PATH_CLUSTER and (R > 8 or c["B"] > 4)
                assert e.code == csg.SYMM_ERANGE or ((c["packed"] and forced or cluster_out)
                                                     and e.code == csg.SYMM_EINVAL), (c, e)
                continue
            ran += 1
            if c["graph"]:
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    _call(sl, c, torch.cuda.current_stream())
                sl.put(sl.y_off, np.full((R, B_MAX * N_MAX), 0xFFFF, dtype=np.uint16))
                torch.cuda.synchronize()
                g.replay()
                g.replay()
                torch.cuda.synchronize()
                del g
            else:
                _call(sl, c, s)                     # a second, chained to the first when chaining is on
            code, rank, tile = csg.symm_status(sl.h, s)
            assert code == csg.SYMM_OK, (i, c, rank, tile)
            _check(sl, c, W, x, bias, gamma)
        assert ran >= cases // 2, (ran, cases)
        assert csg.symm_check_guards(sl.h)[0] == csg.SYMM_OK
    finally:
        sl.close()
