"""nq_gemm_q4_noalloc: the Q4 projection for callers that cannot allocate device memory.

Plug-ins whose host framework owns all device memory, and processes that must keep within a
fixed memory budget once serving has started, cannot let the library cudaMalloc its split-K
scratch on first use. nq_gemm_q4_noalloc keeps that scratch in a fixed device array instead.
These tests call it through the C ABI twice in a row and check both results against
nq_gemm_q4 on the same inputs, within the parity tolerance; check that a problem too large
for the array is refused before anything runs; and check that a bounded wait that runs out
inside it is reported by nq_device_error. The file is collected last (file name) and must
pass both alone in a fresh process and after the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

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


# decode shape (one K slab, split-K runs at block edges) and the T=8 down projection shape
# (three K slabs: every run is a split-K partial, so the scratch is really used)
@pytest.mark.parametrize("T,K,N,seed", [(1, 5120, 17408, 1), (8, 17408, 5120, 3), (3, 640, 48, 9), (20, 1024, 272, 11)])
def test_noalloc_matches_allocating_call_twice(nq, T, K, N, seed):
    p = si.q4_problem(T, K, N, seed)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y_ref = gu.host_f64(nq.gemm_q4(x, *w, N))
    L = nq.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = L.nq_gemm_q4_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w[0].data_ptr()),
                                  ctypes.c_void_p(w[1].data_ptr()), ctypes.c_void_p(y.data_ptr()), T, K, N,
                                  stream)
        assert rc == 0, nq.status_string(rc)
        assert gu.rel_err(gu.host_f64(y), y_ref) <= gu.TOL
    nq.device_error()


def test_noalloc_rejects_problems_beyond_its_scratch(nq):
    # N = 2^20 needs 32768 row-pair tickets, far past the fixed array: refused before launch
    K, N = 64, 1 << 20
    L = nq.lib()
    x = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(nq.packed_bytes_q4(K, N), dtype=torch.uint8, device="cuda")
    s = torch.zeros(nq.scale_bytes(K, N), dtype=torch.uint8, device="cuda")
    y = torch.full((1, N), 2.0, dtype=torch.bfloat16, device="cuda")
    rc = L.nq_gemm_q4_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                              ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(y.data_ptr()), 1, K, N, None)
    assert rc == -8, nq.status_string(rc)
    torch.cuda.synchronize()
    assert bool((y.float() == 2.0).all())          # nothing was launched


def test_noalloc_timeout_is_reported(nq):
    """A 1 ns wait bound makes the kernel abort; the fixed array's error word is reported by
    nq_device_error (not cleared by the next call), and the next call is correct again."""
    T, K, N = 1, 5120, 17408
    p = si.q4_problem(T, K, N, 21)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y_ref = gu.host_f64(nq.gemm_q4(x, *w, N))
    gu.expect_timeout(nq, lambda: nq.gemm_q4_noalloc(x, *w, N))
    y = gu.host_f64(nq.gemm_q4_noalloc(x, *w, N))
    nq.device_error()
    assert gu.rel_err(y, y_ref) <= gu.TOL
