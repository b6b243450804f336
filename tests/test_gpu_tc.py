"""GPU parity of the large-batch tensor-core kernel (8 < T <= 64: tcgen05.mma with the decoded
weights in TMEM) against the fp64 CPU oracle, per token row within 5e-3, and against the
8-token-slice path. Shapes cover partial 128-row blocks, a K split across blocks (fp32 partials
added in fixed order), a single K group, every padded token count (16, 32, 64) and both code
widths."""
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
    assert nq.tensor_core_batches(-1) == 1
    return nq


TC_SHAPES = [
    # T, K, N, seed
    (9, 64, 16, 0), (16, 256, 128, 1), (17, 640, 272, 2), (32, 1024, 48, 3), (33, 5120, 384, 4),
    (48, 1536, 1040, 5), (64, 512, 144, 6), (64, 17408, 96, 7), (24, 6208, 2064, 8), (12, 192, 4096, 9),
    # 16 padded tokens with K split in five pieces of 14 and 15 groups: stages of 6, 6 and 2 or 3
    # groups, so full pairs, a pair and a lone group at a stage's end
    (16, 4544, 2064, 10),
]


def _problem(bits, T, K, N, seed):
    if bits == 4:
        p = si.q4_problem(T, K, N, seed)
        return p, lambda nq: gu.pack_q4(nq, p["wq"], p["s"], K, N), \
            lambda: oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    p = si.q5_problem(T, K, N, seed)
    return p, lambda nq: gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N), \
        lambda: oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("T,K,N,seed", TC_SHAPES)
def test_tc_parity(nq, bits, T, K, N, seed):
    p, pack, ref = _problem(bits, T, K, N, 800 + seed + 50 * bits)
    w = pack(nq)
    fn = nq.gemm_q4 if bits == 4 else nq.gemm_q5
    y = gu.host_f64(fn(gu.dev_bf16(p["x"]), *w, N))
    y_ref = ref()
    for t in range(T):
        assert np.all(np.isfinite(y[t]))
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t
    nq.device_error()


def test_tc_matches_slices_and_is_deterministic(nq):
    T, K, N = 40, 2048, 1152
    p = si.q4_problem(T, K, N, 880)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y1 = nq.gemm_q4(x, *w, N)
    y2 = nq.gemm_q4(x, *w, N)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    prev = nq.tensor_core_batches(0)
    try:
        ys = nq.gemm_q4(x, *w, N)
    finally:
        nq.tensor_core_batches(prev)
    y_ref = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    for y in (y1, ys):
        yh = gu.host_f64(y)
        for t in range(T):
            assert gu.rel_err(yh[t], y_ref[t]) <= gu.TOL
    nq.device_error()


def test_tc_zero_point_codes_give_exact_zero(nq):
    """Codes equal to z decode to exact bf16 zeros, so every product and sum is exactly 0."""
    T, K, N = 24, 1024, 272
    p = si.q4_problem(T, K, N, 881)
    x = gu.dev_bf16(p["x"])
    z4 = gu.pack_q4(nq, np.full((N, K // 8), 0x88888888, np.uint32), p["s"], K, N)
    assert torch.count_nonzero(nq.gemm_q4(x, *z4, N).float()) == 0
    z5 = gu.pack_q5(nq, np.zeros((N, K // 8), np.uint32), np.full((N, K // 32), 0xFFFFFFFF, np.uint32), p["s"], K, N)
    assert torch.count_nonzero(nq.gemm_q5(x, *z5, N).float()) == 0


@pytest.mark.parametrize("T", [16, 32, 64])
@pytest.mark.parametrize("bits,K,N", [(4, 5120, 17408), (5, 5120, 6144), (4, 17408, 5120)])
def test_tc_full_size_sampled(nq, T, bits, K, N):
    """The decode (Q4), verify (Q5) and down-projection (Q4, K split across blocks) weight
    shapes at every padded token count the bench times: full-size launch, sampled rows."""
    p, pack, _ = _problem(bits, T, K, N, 890 + bits + T)
    w = pack(nq)
    fn = nq.gemm_q4 if bits == 4 else nq.gemm_q5
    y = gu.host_f64(fn(gu.dev_bf16(p["x"]), *w, N))
    rows = gu.sample_rows(N, 128, 11)
    if bits == 4:
        y_ref = oracle.gemm_q4_rows(p["x"], p["wq"], p["s"], T, K, rows).T
    else:
        y_ref = oracle.gemm_q5_rows(p["x"], p["wn"], p["wh"], p["s"], T, K, rows).T
    for t in range(T):
        assert gu.rel_err(y[t, rows], y_ref[t]) <= gu.TOL, t


def test_tc_activation_outliers(nq):
    T, K, N = 20, 1280, 160
    p = si.q5_problem(T, K, N, 895)
    g = np.random.default_rng(896)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, 5] = 3.0e38
    x[1, :] *= 1.0e6
    x[3, :] *= 1.0e-30
    x[17, 700] = -2.0e37
    xb = si.bf16_bits(x)
    w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(xb), *w, N))
    y_ref = oracle.gemm_q5(xb, p["wn"], p["wh"], p["s"], T, K, N)
    for t in range(T):
        assert np.all(np.isfinite(y[t]))
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


_RESERVE_SCRIPT = r"""
import sys
import torch
from weight_only_groupwise_gb300 import nq
import oracle
import seeded_inputs as si
from tests import gpu_util as gu
# a small eager call at the same padded token count (64) prepares the kernel instantiation;
# its plan needs no partial sums, so it leaves a small workspace behind
small = si.q5_problem(40, 640, 256, 40)
ws = gu.pack_q5(nq, small["wn"], small["wh"], small["s"], 640, 256)
nq.gemm_q5(gu.dev_bf16(small["x"]), *ws, 256)
torch.cuda.synchronize()
T, K, N = 40, 5120, 6144                      # three K pieces per row block: fp32 partials
p = si.q5_problem(T, K, N, 41)
w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
x = gu.dev_bf16(p["x"])
y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
assert nq.plan_tc_info(5, T, K, N, torch.cuda.get_device_properties(0).multi_processor_count)["k_pieces"] > 1
nq.reserve(64, K, N)
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph):                 # an allocation here would fail the call
    nq.gemm_q5(x, *w, N, out=y)
graph.replay()
torch.cuda.synchronize()
nq.device_error()
err = gu.rel_err(gu.host_f64(y), oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N))
assert err <= gu.TOL, err
print("reserve-ok")
"""


def test_reserve_covers_tensor_core_partials(nq):
    """nq_reserve(64, K, N) allocates the tensor-core kernel's partial sums too: a later
    split-K call of that size, in a fresh process, runs inside CUDA graph capture (where the
    library could not allocate) and matches the oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _RESERVE_SCRIPT], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "reserve-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


# ---------------------------------------------------------------- SwiGLU blocks, 8 < T <= 64
# Two tensor-core launches: the gate projection writes fp32 G, the up projection's epilogue
# writes H = bf16(silu(G) * U).

TC_SWIGLU_SHAPES = [(9, 640, 272, 0), (20, 1024, 1040, 1), (33, 5120, 384, 2), (64, 512, 144, 3),
                    (48, 17408, 96, 4)]


def _swiglu_problem(bits, T, K, N, seed):
    return si.swiglu_problem(T, K, N, seed) if bits == 4 else si.swiglu_q5_problem(T, K, N, seed)


def _swiglu_dev(nq, bits, p, K, N):
    if bits == 4:
        wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
        wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
        return nq.swiglu_q4(gu.dev_bf16(p["x"]), *wg, *wu, N)
    wg = gu.pack_q5(nq, p["wgn"], p["wgh"], p["sg"], K, N)
    wu = gu.pack_q5(nq, p["wun"], p["wuh"], p["su"], K, N)
    return nq.swiglu_q5(gu.dev_bf16(p["x"]), *wg, *wu, N)


def _swiglu_ref(bits, p, T, K, N):
    if bits == 4:
        g, u, _ = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    else:
        g, u, _ = oracle.swiglu_q5(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"], p["su"], T, K, N)
    return g / (1.0 + np.exp(-g)) * u


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("T,K,N,seed", TC_SWIGLU_SHAPES)
def test_tc_swiglu_parity(nq, bits, T, K, N, seed):
    p = _swiglu_problem(bits, T, K, N, 950 + seed)
    h = gu.host_f64(_swiglu_dev(nq, bits, p, K, N))
    h_ref = _swiglu_ref(bits, p, T, K, N)
    for t in range(T):
        assert gu.rel_err(h[t], h_ref[t]) <= gu.TOL, t
    nq.device_error()


def test_tc_swiglu_matches_slices_and_is_deterministic(nq):
    T, K, N = 40, 2048, 1152
    p = _swiglu_problem(4, T, K, N, 960)
    h1 = _swiglu_dev(nq, 4, p, K, N)
    h2 = _swiglu_dev(nq, 4, p, K, N)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    prev = nq.tensor_core_batches(0)
    try:
        hs = _swiglu_dev(nq, 4, p, K, N)
    finally:
        nq.tensor_core_batches(prev)
    h_ref = _swiglu_ref(4, p, T, K, N)
    for h in (h1, hs):
        hh = gu.host_f64(h)
        for t in range(T):
            assert gu.rel_err(hh[t], h_ref[t]) <= gu.TOL
    nq.device_error()


def test_tc_swiglu_zero_point_gate_gives_exact_zero(nq):
    """Gate codes equal to z make G exactly 0, so H = silu(0) * U is exactly 0 everywhere."""
    T, K, N = 24, 1024, 272
    p = _swiglu_problem(4, T, K, N, 961)
    q = dict(p, wg=np.full_like(p["wg"], 0x88888888))
    assert torch.count_nonzero(_swiglu_dev(nq, 4, q, K, N).float()) == 0


@pytest.mark.parametrize("T", [16, 64])
@pytest.mark.parametrize("bits", [4, 5])
def test_tc_swiglu_full_size_sampled(nq, bits, T):
    """The SwiGLU gate/up block of the bench (K=5120, N=17408), full-size launches, sampled rows."""
    K, N = 5120, 17408
    p = _swiglu_problem(bits, T, K, N, 970 + bits + T)
    h = gu.host_f64(_swiglu_dev(nq, bits, p, K, N))
    rows = gu.sample_rows(N, 128, 12)
    if bits == 4:
        g, u, _ = oracle.swiglu_q4_rows(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, rows)
    else:
        g, u, _ = oracle.swiglu_q5_rows(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"], p["su"], T, K, rows)
    h_ref = (g / (1.0 + np.exp(-g)) * u).T
    for t in range(T):
        assert gu.rel_err(h[t, rows], h_ref[t]) <= gu.TOL, t
    nq.device_error()
