"""The publish / last-arriver protocol played by host threads (CPU only).

R threads stand for the R ranks' CTAs of one tile set: arrival order is
randomised, a rank can be made to give up before a tile or publish a stale
flag, two launches can be made to overlap, the tile count can change from one
launch to the next, and the multi-GPU design's bounded flag wait can be made
to run out -- none of which can be staged on a shared GPU without risking a
hang.  The emulation (tests/hostsim/protocol_sim.cpp) follows the same rules
as the kernels: the epoch read from the pad, release flag, acq_rel ticket that
restarts at zero every launch, last ticket reduces in rank order, the last
tile's reducer advances the epoch, nothing ever waits."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hostsim", "protocol_sim.cpp")


@pytest.fixture(scope="module")
def sim(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("sim") / "libprotocol_sim.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", SRC, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    f64p = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.sim_init.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.sim_launch.argtypes = [ctypes.c_int, f64p, ctypes.c_uint, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, f64p, ip]
    lib.sim_overlap.argtypes = [f64p, ctypes.c_uint]
    lib.sim_epoch.restype = ctypes.c_uint32
    lib.sim_wait_flags.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_int]
    yield lib
    lib.sim_free()


def _launch(sim, values, seed, skip=(-1, -1), stale=(-1, -1), sleep_us=20, tiles=None):
    T = values.shape[1]
    y = np.empty(T, dtype=np.float64)
    bad = ctypes.c_int(-1)
    v = np.ascontiguousarray(values, dtype=np.float64)
    rc = sim.sim_launch(T if tiles is None else tiles, v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), seed,
                        skip[0], skip[1],
                        stale[0], stale[1], sleep_us, y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                        ctypes.byref(bad))
    return rc, y, bad.value


def _values(R, T, seed):
    # values whose sum depends on the order of addition, so any reordering shows
    rng = np.random.default_rng(seed)
    return rng.standard_normal((R, T)) * np.exp2(rng.integers(-30, 30, size=(R, T)))


def _rank_order_sum(values):
    acc = np.zeros(values.shape[1])
    for r in range(values.shape[0]):
        acc = acc + values[r]
    return acc


@pytest.mark.parametrize("R,T", [(2, 7), (8, 64), (5, 33)])
def test_arrival_order_does_not_change_the_bits(sim, R, T):
    assert sim.sim_init(R, T) == 0
    vals = _values(R, T, R * T)
    want = _rank_order_sum(vals)
    for launch, seed in enumerate((1, 2, 3, 4), start=1):
        rc, y, _ = _launch(sim, vals, seed)
        assert rc == 0
        assert np.array_equal(y, want), f"launch {launch}"
        assert sim.sim_epoch() == launch


def test_counters_restart_every_launch(sim):
    R, T = 4, 16
    assert sim.sim_init(R, T) == 0
    for launch in range(1, 40):
        vals = _values(R, T, launch)
        rc, y, _ = _launch(sim, vals, launch, sleep_us=0)
        assert rc == 0 and np.array_equal(y, _rank_order_sum(vals))
        assert sim.sim_epoch() == launch and sim.sim_counters_clear() == 1


def test_tile_count_may_change_between_launches(sim):
    """No reset between launches of different geometries (as a replayed CUDA
    graph interleaved with other calls would issue them)."""
    R, T = 4, 32
    assert sim.sim_init(R, T) == 0
    for launch, tiles in enumerate((32, 5, 17, 1, 32, 9), start=1):
        vals = _values(R, T, 100 + launch)
        rc, y, _ = _launch(sim, vals, launch, tiles=tiles)
        assert rc == 0
        assert np.array_equal(y[:tiles], _rank_order_sum(vals)[:tiles]), f"launch {launch}"
        assert np.isnan(y[tiles:]).all()
        assert sim.sim_epoch() == launch and sim.sim_counters_clear() == 1


def test_rank_that_gives_up_never_hangs_and_is_reported(sim):
    R, T = 4, 8
    assert sim.sim_init(R, T) == 0
    vals = _values(R, T, 5)
    rc, y, bad = _launch(sim, vals, 5, skip=(2, 3))
    assert rc == 3 and bad == 3                      # nobody waits: the launch ends, the give-up is latched
    assert np.isnan(y[3])                            # the tile without its rank-2 partial is not written
    ok = [t for t in range(T) if t != 3]
    assert np.array_equal(y[ok], _rank_order_sum(vals)[ok])
    assert sim.sim_epoch() == 0                      # the launch did not finish: the epoch stays
    sim.sim_reset()                                  # the host's reset after the reported error
    rc, y, _ = _launch(sim, vals, 7)
    assert rc == 0 and np.array_equal(y, _rank_order_sum(vals))
    assert sim.sim_epoch() == 1


def test_stale_flag_is_detected_not_summed(sim):
    R, T = 8, 16
    assert sim.sim_init(R, T) == 0
    vals = _values(R, T, 9)
    rc, y, _ = _launch(sim, vals, 9)
    assert rc == 0
    rc, y, bad = _launch(sim, vals, 10, stale=(5, 11))
    assert rc == 1 and bad == 11
    assert np.isnan(y[11])


def test_overlapping_launches_are_reported(sim):
    R, T = 4, 32
    assert sim.sim_init(R, T) == 0
    vals = _values(R, T, 11)
    seen = set()
    for trial in range(20):
        sim.sim_reset()
        seen.add(sim.sim_overlap(vals.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), trial))
        if seen - {0}:
            break
    assert seen - {0}, "two interleaved launches on one set of counters went unnoticed"


def test_bounded_flag_wait_times_out(sim):
    R, T = 4, 4
    assert sim.sim_init(R, T) == 0
    vals = _values(R, T, 13)
    rc, _, _ = _launch(sim, vals, 13, skip=(1, 2), sleep_us=0)
    assert rc == 3
    assert sim.sim_wait_flags(0, 1, 1000) == 0       # complete tile: returns at once
    assert sim.sim_wait_flags(2, 1, 20000) == -1     # rank 1 never published tile 2: gives up
