"""One rank of a multi-process handle, run as its own process by the
multi-process tests (TEST INFRASTRUCTURE).

    python tests/mp_worker.py <scenario> <rank> <world> <tmpdir>

Every rank generates the same seeded global inputs (synth), writes its own
rank's share into its own slot, and runs the scenario's calls, separated by
stream synchronisation and process-group barriers (gloo, through a file
store in tmpdir).  What each rank reads back from its own slot goes to
tmpdir/out<rank>.npz; the test process compares the ranks with each other and
with the oracle.  Scenarios:
  gemv     gemv_all_reduce on the CUDA-core (1) and persistent (4) kernels,
           three calls each, small-integer and normal inputs, row-major and
           packed weights; gemv_reduce_scatter;
  oneshot  one_shot_all_reduce, two calls;
  leave    rank world-1 leaves after the first call (its kernels finished);
           the others make one more call and report symm_status one after
           another;
  leave0   the same with rank 0 leaving, whose pad holds the tile counters
           every rank shares.
"""
from __future__ import annotations

import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import collective_split_gemv_gb300 as csg  # noqa: E402
import synth  # noqa: E402
from collective_split_gemv_gb300 import DeviceView  # noqa: E402
from collective_split_gemv_gb300.multiproc import mp_alloc  # noqa: E402
from collective_split_gemv_gb300.workspace import pad_bytes_for  # noqa: E402

N, KR, B = 1000, 512, 4          # gemv shape per rank (K = R * KR)
N_AR = 3 * 4096 + 24             # one-shot elements per rank


def _up(v, a=256):
    return (v + a - 1) // a * a


class Rank:
    def __init__(self, rank, world, tmpdir):
        self.rank, self.world = rank, world
        self.dev = torch.device("cuda", 0)
        wbytes, xbytes, ybytes = N * KR * 2, B * KR * 2, B * N * 2
        self.wp_bytes = csg.symm_packed_w_bytes(world, N, world * KR)
        self.w_off = 0
        self.wp_off = _up(wbytes)
        self.x_off = self.wp_off + _up(self.wp_bytes)
        self.y_off = self.x_off + _up(xbytes)
        self.in_off = self.y_off + _up(ybytes)
        self.out_off = self.in_off + _up(N_AR * 2)
        slot_bytes = self.out_off + _up(N_AR * 2)
        barrier = lambda: dist.barrier()   # noqa: E731
        self.h, self.slots, self.pads, self.stride = mp_alloc(world, rank, slot_bytes, 9 * 4 * B * N,
                                                              pad_bytes_for(N), tmpdir, barrier)

    def view(self, r, off, nbytes):
        return torch.as_tensor(DeviceView(self.slots[r] + off, (nbytes,)), device=self.dev)

    def put_own(self, off, words):
        a = np.ascontiguousarray(words)
        self.view(self.rank, off, a.nbytes).copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))

    def get_own(self, off, count):
        torch.cuda.synchronize()
        return self.view(self.rank, off, count * 2).cpu().numpy().view(np.uint16).copy()

    def ptr(self, off):
        return self.slots[0] + off


def step_barrier():
    torch.cuda.synchronize()
    dist.barrier()


def gemv(rk: Rank, out):
    R = rk.world
    s = torch.cuda.current_stream()
    rng = np.random.default_rng(7)
    Wi = rng.integers(-8, 9, size=(R, N, KR)).astype(np.float32)
    xi = rng.integers(-8, 9, size=(R, B, KR)).astype(np.float32)
    cases = {"int": (synth.round_bf16(Wi.astype(np.float64)), synth.round_bf16(xi.astype(np.float64))),
             "normal": synth.gemv_inputs(R, N, R * KR, B, seed=11, w_std=0.02, x="normal")}
    for kind, (W, x) in cases.items():
        rk.put_own(rk.w_off, W[rk.rank])
        rk.put_own(rk.x_off, x[rk.rank])
        step_barrier()
        for path in (csg.GEMV_PATH_FFMA, csg.GEMV_PATH_DYN):
            csg.symm_set_option(rk.h, csg.SYMM_OPT_GEMV_PATH, path)
            for i in range(3):
                rk.put_own(rk.y_off, np.full(B * N, 0xFFFF, dtype=np.uint16))
                step_barrier()
                csg.gemv_all_reduce(rk.h, rk.ptr(rk.w_off), rk.ptr(rk.x_off), rk.ptr(rk.y_off), R, N, R * KR, B, s)
                step_barrier()
                out[f"{kind}_p{path}_{i}"] = rk.get_own(rk.y_off, B * N)
        # packed weights (each rank packs its own), persistent kernel
        csg.symm_set_option(rk.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_AUTO)
        csg.symm_pack_w(rk.h, rk.ptr(rk.w_off), rk.ptr(rk.wp_off), R, N, R * KR, s)
        step_barrier()
        rk.put_own(rk.y_off, np.full(B * N, 0xFFFF, dtype=np.uint16))
        step_barrier()
        csg.gemv_all_reduce(rk.h, rk.ptr(rk.wp_off), rk.ptr(rk.x_off), rk.ptr(rk.y_off), R, N, R * KR, B, s)
        step_barrier()
        out[f"{kind}_packed"] = rk.get_own(rk.y_off, B * N)
        # the reduce-scatter form: rank s keeps batch rows [s*B/R, (s+1)*B/R)
        if B % R == 0:
            rk.put_own(rk.y_off, np.full(B * N, 0xFFFF, dtype=np.uint16))
            step_barrier()
            csg.gemv_reduce_scatter(rk.h, rk.ptr(rk.w_off), rk.ptr(rk.x_off), rk.ptr(rk.y_off), R, N, R * KR, B, s)
            step_barrier()
            out[f"{kind}_rs"] = rk.get_own(rk.y_off, (B // R) * N)
    code, rank, tile = csg.symm_status(rk.h, s)
    out["status"] = np.array([code, rank, tile])
    out["guards"] = np.array([csg.symm_check_guards(rk.h)[0]])


def oneshot(rk: Rank, out):
    R = rk.world
    s = torch.cuda.current_stream()
    for i in range(2):
        inp = synth.allreduce_inputs(R, N_AR, 20 + i)
        rk.put_own(rk.in_off, inp[rk.rank])
        rk.put_own(rk.out_off, np.full(N_AR, 0xFFFF, dtype=np.uint16))
        step_barrier()
        csg.one_shot_all_reduce(rk.h, rk.ptr(rk.in_off), rk.ptr(rk.out_off), R, N_AR, s)
        step_barrier()
        out[f"ar_{i}"] = rk.get_own(rk.out_off, N_AR)
    out["status"] = np.array(csg.symm_status(rk.h, s))


def leave(rk: Rank, out, survivors, leaver):
    R = rk.world
    s = torch.cuda.current_stream()
    W, x = synth.gemv_inputs(R, N, R * KR, B, seed=12, w_std=0.02, x="normal")
    rk.put_own(rk.w_off, W[rk.rank])
    rk.put_own(rk.x_off, x[rk.rank])
    csg.symm_set_option(rk.h, csg.SYMM_OPT_GEMV_PATH, csg.GEMV_PATH_DYN)
    step_barrier()
    csg.gemv_all_reduce(rk.h, rk.ptr(rk.w_off), rk.ptr(rk.x_off), rk.ptr(rk.y_off), R, N, R * KR, B, s)
    step_barrier()
    out["first"] = rk.get_own(rk.y_off, B * N)
    out["first_status"] = np.array(csg.symm_status(rk.h, s))
    # every rank has read its status before a survivor launches its next call
    # (the status compares the ranks' launch counts)
    step_barrier()
    if rk.rank == leaver:
        return "left"   # between calls, nothing of this rank in flight
    # the others go on without it: their next call finishes (nothing waits
    # for the missing rank) and symm_status, after their barrier, reports it
    csg.gemv_all_reduce(rk.h, rk.ptr(rk.w_off), rk.ptr(rk.x_off), rk.ptr(rk.y_off), R, N, R * KR, B, s)
    torch.cuda.synchronize()
    dist.barrier(group=survivors)
    # the survivors report one after another, in rank order: each report
    # resets that rank's pad (its launch count kept), and the later reports
    # read the pads of the ranks that have already reset
    for turn in [r for r in range(R) if r != leaver]:
        if turn == rk.rank:
            out["status"] = np.array(csg.symm_status(rk.h, s))
        dist.barrier(group=survivors)
    return "stayed"


def main():
    scenario, rank, world, tmpdir = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), sys.argv[4]
    torch.cuda.set_device(0)
    # a short timeout: a rank that fails makes the others' barriers raise
    # (after their kernels have finished) instead of blocking
    dist.init_process_group("gloo", init_method=f"file://{tmpdir}/pg", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=60))
    leaver = 0 if scenario == "leave0" else world - 1
    survivors = dist.new_group([r for r in range(world) if r != leaver]) if world > 1 else None
    rk = Rank(rank, world, tmpdir)
    out = {}
    try:
        if scenario == "gemv":
            gemv(rk, out)
        elif scenario == "oneshot":
            oneshot(rk, out)
        elif scenario in ("leave", "leave0"):
            out["role"] = np.array([1 if leave(rk, out, survivors, leaver) == "left" else 0])
        else:
            raise SystemExit(f"unknown scenario {scenario}")
        np.savez(os.path.join(tmpdir, f"out{rank}.npz"), **out)
    finally:
        torch.cuda.synchronize()
        if scenario not in ("leave", "leave0"):
            dist.barrier()
        csg.symm_free(rk.h)
    os._exit(0)   # no process-group teardown: a rank may have left


if __name__ == "__main__":
    main()
