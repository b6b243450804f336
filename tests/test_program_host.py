"""Recorded programs (nq_program_* of include/nq.h), host side: recording runs every argument
check of the recorded call without a CUDA call and stores nothing for a call that fails them
or is empty. Fake device addresses are fine here: recording never dereferences them. No GPU."""
import ctypes

import pytest

from weight_only_groupwise_gb300 import nq as nqmod

NULL, SHAPE, ALIGN, ALIAS = -1, -2, -3, -4
A = 1 << 40          # fake, 16-byte aligned device addresses far apart
MB = 1 << 20


@pytest.fixture(scope="module")
def L():
    from weight_only_groupwise_gb300 import build
    build.build()
    return nqmod.lib()


@pytest.fixture
def prog(L):
    h = ctypes.c_void_p()
    assert L.nq_program_create(ctypes.byref(h)) == 0 and h.value
    yield h
    L.nq_program_destroy(h)


def info(L, h):
    out = (ctypes.c_int64 * 4)()
    assert L.nq_program_info(h, ctypes.cast(out, ctypes.c_void_p)) == 0
    return dict(zip(nqmod.PROGRAM_KEYS, list(out)))


def P(x):
    return ctypes.c_void_p(x)


def test_new_program_is_empty(L, prog):
    assert info(L, prog) == {"calls": 0, "kernels": 0, "builds": 0, "failed_call": -1}


def test_null_program_and_outputs(L):
    assert L.nq_program_create(None) == NULL
    assert L.nq_program_gemm(None, 4, P(A), P(2 * A), P(3 * A), P(4 * A), 1, 64, 16) == NULL
    assert L.nq_program_build(None) == NULL
    assert L.nq_program_launch(None, None) == NULL
    out = (ctypes.c_int64 * 4)()
    assert L.nq_program_info(None, ctypes.cast(out, ctypes.c_void_p)) == NULL
    L.nq_program_destroy(None)  # ignored


def test_recording_checks_match_the_calls(L, prog):
    g = L.nq_program_gemm
    assert g(prog, 3, P(A), P(2 * A), P(3 * A), P(4 * A), 1, 64, 16) == SHAPE      # bits
    assert g(prog, 4, P(A), P(2 * A), P(3 * A), P(4 * A), 65, 64, 16) == SHAPE     # T > 64
    assert g(prog, 4, P(A), P(2 * A), P(3 * A), P(4 * A), 1, 100, 16) == SHAPE     # K % 64
    assert g(prog, 5, P(A), P(2 * A), P(3 * A), P(4 * A), 1, 64, 24) == SHAPE      # N % 16
    assert g(prog, 4, None, P(2 * A), P(3 * A), P(4 * A), 1, 64, 16) == NULL
    assert g(prog, 4, P(A), P(2 * A), None, P(4 * A), 1, 64, 16) == NULL
    assert g(prog, 4, P(A + 8), P(2 * A), P(3 * A), P(4 * A), 1, 64, 16) == ALIGN
    assert g(prog, 4, P(A), P(2 * A), P(3 * A), P(A + 64), 2, 64, 16) == ALIAS     # Y inside X
    assert g(prog, 5, P(A), P(2 * A), P(3 * A), P(2 * A + 16), 1, 64, 16) == ALIAS  # Y inside Wq
    s = L.nq_program_swiglu
    assert s(prog, 6, P(A), P(2 * A), P(3 * A), P(4 * A), P(5 * A), P(6 * A), 1, 64, 16) == SHAPE
    assert s(prog, 4, P(A), P(2 * A), P(3 * A), None, P(5 * A), P(6 * A), 1, 64, 16) == NULL
    assert s(prog, 4, P(A), P(2 * A), P(3 * A), P(4 * A), P(5 * A), P(4 * A + 32), 1, 64, 16) == ALIAS
    f = L.nq_program_gemm_fp4
    assert f(prog, P(A), P(2 * A), P(3 * A), ctypes.c_float(1.0), P(4 * A + 4), 1, 64, 16) == ALIGN
    sf = L.nq_program_swiglu_fp4
    one = ctypes.c_float(1.0)
    assert sf(prog, P(A), P(2 * A), P(3 * A), one, P(4 * A), P(5 * A), one, P(6 * A), 1, 96, 16) == SHAPE
    assert sf(prog, P(A), P(2 * A), None, one, P(4 * A), P(5 * A), one, P(6 * A), 1, 64, 16) == NULL
    assert sf(prog, P(A), P(2 * A), P(3 * A), one, P(4 * A), P(5 * A), one, P(5 * A + 16), 1, 64, 16) == ALIAS
    assert info(L, prog)["calls"] == 0


def test_empty_calls_record_nothing(L, prog):
    assert L.nq_program_gemm(prog, 4, None, None, None, None, 0, 64, 16) == 0
    assert L.nq_program_gemm(prog, 5, None, None, None, None, 3, 64, 0) == 0
    assert L.nq_program_swiglu(prog, 4, None, None, None, None, None, None, 0, 64, 16) == 0
    assert info(L, prog)["calls"] == 0


def test_valid_calls_are_recorded_in_order(L, prog):
    assert L.nq_program_swiglu(prog, 4, P(A), P(2 * A), P(3 * A), P(4 * A), P(5 * A), P(6 * A), 8, 640, 1088) == 0
    assert L.nq_program_gemm(prog, 4, P(6 * A), P(7 * A), P(8 * A), P(9 * A), 8, 1088, 640) == 0
    assert L.nq_program_gemm_fp4(prog, P(A), P(10 * A), P(11 * A), ctypes.c_float(0.5), P(12 * A), 40, 640,
                                 272) == 0
    groups = (nqmod.NqGroup * 2)(nqmod.NqGroup(13 * A, 14 * A, 15 * A, 384), nqmod.NqGroup(16 * A, 17 * A, 18 * A, 64))
    assert L.nq_program_grouped(prog, 5, P(A), ctypes.cast(groups, ctypes.c_void_p), 2, 8, 640) == 0
    # K == 0 with outputs present is a call (it writes zeros), not an empty problem
    assert L.nq_program_gemm(prog, 5, P(A), P(2 * A), P(3 * A), P(19 * A), 4, 0, 32) == 0
    assert L.nq_program_swiglu_fp4(prog, P(A), P(20 * A), P(21 * A), ctypes.c_float(0.5), P(22 * A), P(23 * A),
                                   ctypes.c_float(0.25), P(24 * A), 8, 640, 1088) == 0
    i = info(L, prog)
    assert i["calls"] == 6 and i["kernels"] == 0 and i["builds"] == 0


def test_grouped_recording_checks(L, prog):
    gr = L.nq_program_grouped
    one = (nqmod.NqGroup * 1)(nqmod.NqGroup(2 * A, 3 * A, 4 * A, 48))
    arr = ctypes.cast(one, ctypes.c_void_p)
    assert gr(prog, 4, P(A), None, 1, 8, 640) == NULL
    assert gr(prog, 4, P(A), arr, 0, 8, 640) == SHAPE
    assert gr(prog, 14, P(A), arr, 1, 8, 640) == SHAPE        # no grouped NVFP4 call
    assert gr(prog, 4, P(A), arr, 1, 8, 96) == SHAPE          # K % 64
    overlapping = (nqmod.NqGroup * 2)(nqmod.NqGroup(2 * A, 3 * A, 4 * A, 48),
                                      nqmod.NqGroup(5 * A, 6 * A, 4 * A + 64, 16))
    assert gr(prog, 4, P(A), ctypes.cast(overlapping, ctypes.c_void_p), 2, 8, 640) == ALIAS
    assert gr(prog, 4, P(A), arr, 1, 0, 640) == 0             # empty: nothing recorded
    assert info(L, prog)["calls"] == 0


def test_build_without_a_gpu_reports_an_error(L, prog):
    """Without a CUDA device, building or launching a recorded program returns an error status
    (the runtime's device query fails) instead of crashing; the records stay."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert L.nq_program_gemm(prog, 4, P(A), P(2 * A), P(3 * A), P(4 * A), 1, 64, 16) == 0
    assert L.nq_program_build(prog) < 0
    assert L.nq_program_launch(prog, None) < 0
    i = info(L, prog)
    assert i["calls"] == 1 and i["builds"] == 0 and i["kernels"] == 0
