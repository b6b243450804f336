"""Bounded device-side waits. With the wait bound set far below a kernel's run time (1 ns),
the projection kernels abort instead of waiting: nq_device_error then reports
NQ_ERR_TIMEOUT once and clears the flag and the split-K tickets, and the next call with the
default bound is correct. The wait runs out because of the bound alone: nothing faults, traps
or spins without limit, and every aborted block still waits, on its own fixed bound, for the
copies it has issued before it exits."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from weight_only_groupwise_gb300 import build
    build.build()
    from weight_only_groupwise_gb300 import nq
    return nq


# decode (one slab, whole row pairs, fp16 operands) and a three-slab split-K shape (bf16
# operands, every run a partial: an abort leaves tickets part-counted)
@pytest.mark.parametrize("T,K,N,seed", [(1, 5120, 17408, 1), (8, 17408, 512, 3)])
def test_timeout_is_reported_and_next_call_is_correct(nq, T, K, N, seed):
    base = nq.wait_limit(0)
    assert base >= 1_000_000
    p = si.q4_problem(T, K, N, seed)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    gu.expect_timeout(nq, lambda: nq.gemm_q4(x, *w, N, out=y))
    assert nq.wait_limit(0) == base
    y = gu.host_f64(nq.gemm_q4(x, *w, N))
    nq.device_error()
    assert gu.rel_err(y, oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)) <= gu.TOL


def test_timeout_in_fused_swiglu(nq):
    T, K, N = 4, 2048, 2048
    p = si.swiglu_problem(T, K, N, 17)
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    x = gu.dev_bf16(p["x"])
    gu.expect_timeout(nq, lambda: nq.swiglu_q4(x, *wg, *wu, N))
    h = gu.host_f64(nq.swiglu_q4(x, *wg, *wu, N))
    nq.device_error()
    g, u, _ = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL


# the tensor-core kernel (8 < T <= 64): one K piece per row block, and a K split in three
# (tickets part-counted when a block aborts)
@pytest.mark.parametrize("bits,T,K,N,seed", [(4, 16, 640, 17408, 21), (5, 20, 5120, 6144, 22)])
def test_timeout_in_tensor_core_kernel(nq, bits, T, K, N, seed):
    assert nq.tensor_core_batches(1) == 1
    if bits == 4:
        p = si.q4_problem(T, K, N, seed)
        w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
        fn = nq.gemm_q4
        ref = lambda: oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    else:
        p = si.q5_problem(T, K, N, seed)
        w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
        fn = nq.gemm_q5
        ref = lambda: oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)
    x = gu.dev_bf16(p["x"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    gu.expect_timeout(nq, lambda: fn(x, *w, N, out=y))
    y = gu.host_f64(fn(x, *w, N))
    nq.device_error()
    assert gu.rel_err(y, ref()) <= gu.TOL


def test_timeout_in_tensor_core_swiglu(nq):
    """A SwiGLU block with 8 < T <= 64 is two tensor-core launches (gate, then up); both abort
    under the 1 ns bound, and the next call is correct."""
    assert nq.tensor_core_batches(1) == 1
    T, K, N = 24, 5120, 1024
    p = si.swiglu_problem(T, K, N, 23)
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    x = gu.dev_bf16(p["x"])
    gu.expect_timeout(nq, lambda: nq.swiglu_q4(x, *wg, *wu, N))
    h = gu.host_f64(nq.swiglu_q4(x, *wg, *wu, N))
    nq.device_error()
    g, u, _ = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    ref = g / (1.0 + np.exp(-g)) * u
    for t in range(T):
        assert gu.rel_err(h[t], ref[t]) <= gu.TOL


@pytest.mark.parametrize("T", [4, 24])
def test_timeout_in_nvfp4_swiglu(nq, T):
    """The NVFP4 SwiGLU block on the 8-token kernel (T = 4) and as two tensor-core launches
    (T = 24): both abort under the 1 ns bound, and the next call is correct."""
    K, N = 5120, 4096
    p = si.swiglu_fp4_problem(T, K, N, 27)
    wg = nq.pack_fp4(gu.dev_u32(p["cg"]), torch.from_numpy(np.ascontiguousarray(p["sfg"])).cuda(), K, N)
    wu = nq.pack_fp4(gu.dev_u32(p["cu"]), torch.from_numpy(np.ascontiguousarray(p["sfu"])).cuda(), K, N)
    x = gu.dev_bf16(p["x"])
    gu.expect_timeout(nq, lambda: nq.swiglu_fp4(x, *wg, p["gg"], *wu, p["gu"], N))
    h = gu.host_f64(nq.swiglu_fp4(x, *wg, p["gg"], *wu, p["gu"], N))
    nq.device_error()
    g, u, _ = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL


def test_timeout_in_a_recorded_program(nq):
    """A program built while the wait bound is 1 ns keeps that bound (settings are baked in at
    build time): its replay aborts and nq_device_error reports it; built again under the
    default bound, the replay is correct."""
    from weight_only_groupwise_gb300.nq import NqError
    T, K, N = 8, 5120, 6144
    p = si.q5_problem(T, K, N, 29)
    w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    prog = nq.Program()
    y = prog.gemm_q5(x, *w, N)
    timed_out = False
    for _ in range(5):
        prev = nq.wait_limit(1)
        try:
            prog.build()
        finally:
            nq.wait_limit(prev)
        prog.launch()
        try:
            nq.device_error()
        except NqError as e:
            assert e.status == -7, e
            nq.device_error()
            timed_out = True
            break
    assert timed_out, "no bounded wait ran out in the replay with a 1 ns bound"
    prog.build()
    prog.launch()
    torch.cuda.synchronize()
    nq.device_error()
    assert gu.rel_err(gu.host_f64(y), oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)) <= gu.TOL
    prog.close()
