"""One-shot all-reduce on the GPU through the C ABI against the CPU oracle,
for both kernels: per-thread loads and stores, and the one staged through
shared memory by bulk (TMA) copies."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import collective_split_gemv_gb300 as csg
import oracle
import synth
from collective_split_gemv_gb300.workspace import AllReduceWorkspace
from gpu_common import require_gpu, run_allreduce
from helpers import f64_to_words_via_f32, tolerance_ratio, ulp_distance, words_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _check(inp, out, exact=False):
    ref, want = oracle.one_shot_all_reduce(inp)
    R = inp.shape[0]
    for s in range(1, R):
        assert np.array_equal(out[s], out[0]), f"replica {s} differs"
    if exact:
        assert np.array_equal(out[0], want[0])
    assert tolerance_ratio(words_to_f64(out[0]), ref) <= 1.0
    return float(np.mean(out[0] == want[0])) if out.size else 1.0, \
        int(ulp_distance(out[0], want[0]).max()) if out.size else 0


KERNELS = {"per_thread": csg.AR_KERNEL_PER_THREAD, "staged": csg.AR_KERNEL_STAGED}


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_full_size_workload(kernel):
    inp = synth.workload_inputs("allreduce")
    out = run_allreduce(inp, kernel=KERNELS[kernel])
    eq, ulp = _check(inp, out)
    print(f"allreduce ({kernel}): bit-equal {eq:.6f}, max ulp {ulp}")
    assert eq >= 0.999 and ulp <= 1
    out2 = run_allreduce(inp, kernel=KERNELS[kernel])
    assert np.array_equal(out, out2)


def test_kernels_and_auto_choice_agree_bit_for_bit():
    # the same sum order (fp32, rank 0..R-1, one rounding) in both kernels;
    # small and large sizes, ragged
    for R, n in ((8, 4096 * 64 + 5), (8, (1 << 19) + 3), (3, (1 << 20) + 11)):
        inp = synth.allreduce_inputs(R, n, R + n)
        outs = [run_allreduce(inp, kernel=k) for k in (csg.AR_KERNEL_AUTO, csg.AR_KERNEL_PER_THREAD,
                                                        csg.AR_KERNEL_STAGED)]
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2]), (R, n)
        _check(inp, outs[0])


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("R,n", [(1, 8), (2, 7), (3, 1003), (4, 1), (5, 4096 + 3), (8, 100000),
                                 (16, 999), (64, 65), (64, 64 * 1024 + 1), (2, 3 * 1024 * 1024 + 8)])
def test_integer_inputs_bit_exact(R, n, kernel):
    rng = np.random.default_rng(R * 7 + n)
    inp = f64_to_words_via_f32(rng.integers(-100, 101, size=(R, n)).astype(np.float64))
    out = run_allreduce(inp, kernel=KERNELS[kernel])
    _check(inp, out, exact=True)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("R,n", [(2, 12345), (8, 1 << 16), (3, 17), (8, (1 << 20) + 7)])
def test_in_place(R, n, kernel):
    inp = synth.allreduce_inputs(R, n, 9)
    out = run_allreduce(inp, in_place=True, kernel=KERNELS[kernel])
    _check(inp, out)


def test_zero_elements_and_bad_arguments():
    aw = AllReduceWorkspace(2, 64)
    try:
        s = torch.cuda.current_stream()
        csg.one_shot_all_reduce(aw.h, aw.base, aw.base + aw.out_off, 2, 0, s)   # no-op
        bad = [
            ((aw.base, aw.base + aw.out_off, 3, 64), csg.SYMM_EINVAL),        # R mismatch
            ((aw.base + 2, aw.base + aw.out_off, 2, 64), csg.SYMM_EINVAL),    # misaligned
            ((aw.base, aw.base + 16, 2, 64), csg.SYMM_EINVAL),                # partial overlap
            ((aw.base, aw.base + aw.out_off, 2, 10 ** 9), csg.SYMM_EINVAL),   # past the region
            ((aw.slots[1], aw.base + aw.out_off, 2, 64), csg.SYMM_EINVAL),    # not slot 0
        ]
        for args, code in bad:
            with pytest.raises(csg.SymmError) as e:
                csg.one_shot_all_reduce(aw.h, *args, s)
            assert e.value.code == code, args
        assert csg.symm_check_guards(aw.h)[0] == csg.SYMM_OK
    finally:
        aw.close()
