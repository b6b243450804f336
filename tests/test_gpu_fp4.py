"""GPU parity of the NVFP4 weight path (e2m1 elements, e4m3 scale per 16, fp32 tensor scale)
against the fp64 CPU oracle on the same seeded inputs: the decoded weights bit for bit
(through the kernels' own decoder), the projection within max|y - y_ref| / max|y_ref| <= 5e-3
(per token row)."""
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


def pack(nq, p, K, N):
    return nq.pack_fp4(gu.dev_u32(p["codes"]), torch.from_numpy(np.ascontiguousarray(p["sf"])).cuda(), K, N)


@pytest.mark.parametrize("K,N,seed", [(64, 16, 0), (256, 48, 1), (640, 272, 2), (5120, 17408, 3)])
def test_fp4_dequant_bit_exact(nq, K, N, seed):
    p = si.fp4_problem(1, K, N, 500 + seed)
    w = pack(nq, p, K, N)
    w_gpu = nq.dequant_fp4_debug(*w, p["g"], K, N).cpu().numpy()
    w_ref = oracle.dequant_fp4(p["codes"], p["sf"], p["g"], K, N)
    assert np.array_equal(w_gpu.view(np.uint32), w_ref.view(np.uint32))


def test_fp4_dequant_every_code_and_scale_edges(nq):
    """Every e2m1 code at every fragment position, under e4m3 scales that include the
    subnormals (0x01..0x07), the smallest normal, 1.0, the largest finite value (448), and a
    tensor scale that is not a power of two."""
    K, N = 256, 32
    k = np.arange(K)
    n = np.arange(N)[:, None]
    c = (k[None, :] * 5 + 3 * n) % 16
    codes = np.zeros((N, K // 8), np.uint32)
    for i in range(8):
        codes |= c[:, i::8].astype(np.uint32) << np.uint32(4 * i)
    edge = np.array([0x01, 0x02, 0x07, 0x08, 0x38, 0x7E, 0x3F, 0x10, 0x55, 0x5E], np.uint8)
    sf = np.ascontiguousarray(edge[(np.arange(N)[:, None] + np.arange(K // 16)[None, :]) % len(edge)])
    g = 0.3
    p = {"codes": codes, "sf": sf}
    w = pack(nq, p, K, N)
    w_gpu = nq.dequant_fp4_debug(*w, g, K, N).cpu().numpy()
    w_ref = oracle.dequant_fp4(codes, sf, g, K, N)
    assert np.array_equal(w_gpu.view(np.uint32), w_ref.view(np.uint32))


FP4_GEMM_SHAPES = [(1, 256, 128, 0), (2, 640, 48, 1), (3, 192, 80, 2), (5, 1024, 272, 3), (8, 5120, 96, 4),
                   (8, 17408, 48, 5), (7, 6208, 32, 6), (12, 512, 64, 7), (1, 17408, 32, 8)]


@pytest.mark.parametrize("T,K,N,seed", FP4_GEMM_SHAPES)
def test_fp4_gemm_parity(nq, T, K, N, seed):
    p = si.fp4_problem(T, K, N, 520 + seed)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(p["x"]), *w, p["g"], N))
    y_ref = oracle.gemm_fp4(p["x"], p["codes"], p["sf"], p["g"], T, K, N)
    for t in range(T):
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


@pytest.mark.parametrize("T", [1, 8])
def test_fp4_decode_shape_full_size_sampled(nq, T):
    """The 27B-class FFN up-projection shape (K=5120, N=17408) in NVFP4, full-size launch,
    sampled output rows."""
    K, N = 5120, 17408
    p = si.fp4_problem(T, K, N, 540 + T)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(p["x"]), *w, p["g"], N))
    rows = gu.sample_rows(N, 256, 7)
    y_ref = oracle.gemm_fp4_rows(p["x"], p["codes"], p["sf"], p["g"], T, K, rows).T
    assert gu.rel_err(y[:, rows], y_ref) <= gu.TOL


def test_fp4_activation_range_outliers(nq):
    T, K, N = 6, 1280, 96
    p = si.fp4_problem(T, K, N, 560)
    g = np.random.default_rng(561)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, 5] = 3.0e38
    x[1, :] *= 1.0e6
    x[2, 100:200] = 70000.0
    x[3, :] *= 1.0e-30
    xb = si.bf16_bits(x)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(xb), *w, p["g"], N))
    y_ref = oracle.gemm_fp4(xb, p["codes"], p["sf"], p["g"], T, K, N)
    for t in range(T):
        assert np.all(np.isfinite(y[t]))
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


def test_fp4_deterministic(nq):
    T, K, N = 8, 6208, 272
    p = si.fp4_problem(T, K, N, 570)
    w = pack(nq, p, K, N)
    x = gu.dev_bf16(p["x"])
    y1 = nq.gemm_fp4(x, *w, p["g"], N)
    y2 = nq.gemm_fp4(x, *w, p["g"], N)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    nq.device_error()


# ---------------------------------------------------------------- 8 < T <= 64: tensor cores
# The decoded weights e2m1 x e4m3 x 2^-20 are exact in bf16; the epilogue multiplies by
# 2^20 g.

FP4_TC_SHAPES = [(9, 640, 272, 0), (16, 5120, 384, 1), (33, 512, 144, 2), (64, 17408, 96, 3), (40, 6208, 1040, 4)]


@pytest.mark.parametrize("T,K,N,seed", FP4_TC_SHAPES)
def test_fp4_tc_parity(nq, T, K, N, seed):
    assert nq.tensor_core_batches(-1) == 1
    p = si.fp4_problem(T, K, N, 600 + seed)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(p["x"]), *w, p["g"], N))
    y_ref = oracle.gemm_fp4(p["x"], p["codes"], p["sf"], p["g"], T, K, N)
    for t in range(T):
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t
    nq.device_error()


@pytest.mark.parametrize("T", [16, 64])
def test_fp4_tc_full_size_sampled(nq, T):
    K, N = 5120, 17408
    p = si.fp4_problem(T, K, N, 610 + T)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(p["x"]), *w, p["g"], N))
    rows = gu.sample_rows(N, 128, 13)
    y_ref = oracle.gemm_fp4_rows(p["x"], p["codes"], p["sf"], p["g"], T, K, rows).T
    for t in range(T):
        assert gu.rel_err(y[t, rows], y_ref[t]) <= gu.TOL, t


def test_fp4_tc_matches_slices_and_is_deterministic(nq):
    T, K, N = 24, 2048, 1152
    p = si.fp4_problem(T, K, N, 620)
    w = pack(nq, p, K, N)
    x = gu.dev_bf16(p["x"])
    y1 = nq.gemm_fp4(x, *w, p["g"], N)
    y2 = nq.gemm_fp4(x, *w, p["g"], N)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    prev = nq.tensor_core_batches(0)
    try:
        ys = nq.gemm_fp4(x, *w, p["g"], N)
    finally:
        nq.tensor_core_batches(prev)
    y_ref = oracle.gemm_fp4(p["x"], p["codes"], p["sf"], p["g"], T, K, N)
    for y in (y1, ys):
        yh = gu.host_f64(y)
        for t in range(T):
            assert gu.rel_err(yh[t], y_ref[t]) <= gu.TOL, t
    nq.device_error()


def test_fp4_tc_activation_outliers(nq):
    """Activations up to the bf16 maximum times weights up to 2688: the 2^-20 in the decoded
    weights keeps every group partial finite."""
    T, K, N = 20, 1280, 160
    p = si.fp4_problem(T, K, N, 630)
    g = np.random.default_rng(631)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, 5] = 3.0e38
    x[1, :] *= 1.0e6
    x[3, :] *= 1.0e-30
    x[17, 700] = -2.0e37
    xb = si.bf16_bits(x)
    w = pack(nq, p, K, N)
    y = gu.host_f64(nq.gemm_fp4(gu.dev_bf16(xb), *w, p["g"], N))
    y_ref = oracle.gemm_fp4(xb, p["codes"], p["sf"], p["g"], T, K, N)
    for t in range(T):
        assert np.all(np.isfinite(y[t])), t
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


# ---------------------------------------------------------------- NVFP4 SwiGLU blocks
# The gate/up block of an NVFP4 MLP, gate and up with different tensor scales: one launch for
# T <= 8, two tensor-core launches (gate -> fp32 G, up -> bf16 silu(G) * U) for 8 < T <= 64.
# H against silu(g) * u from the oracle's fp64 g and u, at the parity bar of the other blocks.

def _swiglu_fp4(nq, p, T, K, N):
    wg = nq.pack_fp4(gu.dev_u32(p["cg"]), torch.from_numpy(np.ascontiguousarray(p["sfg"])).cuda(), K, N)
    wu = nq.pack_fp4(gu.dev_u32(p["cu"]), torch.from_numpy(np.ascontiguousarray(p["sfu"])).cuda(), K, N)
    return wg, wu


SWIGLU_FP4_SHAPES = [(1, 256, 48, 0), (2, 640, 16, 1), (3, 1024, 272, 2), (4, 320, 112, 3), (8, 6208, 32, 4),
                     (6, 17408, 64, 5), (9, 640, 272, 6), (16, 1024, 1040, 7), (33, 5120, 384, 8),
                     (64, 512, 144, 9), (48, 17408, 96, 10)]


@pytest.mark.parametrize("T,K,N,seed", SWIGLU_FP4_SHAPES)
def test_swiglu_fp4_parity(nq, T, K, N, seed):
    p = si.swiglu_fp4_problem(T, K, N, 700 + seed)
    wg, wu = _swiglu_fp4(nq, p, T, K, N)
    h = gu.host_f64(nq.swiglu_fp4(gu.dev_bf16(p["x"]), *wg, p["gg"], *wu, p["gu"], N))
    g, u, _ = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL
    nq.device_error()


@pytest.mark.parametrize("T", [8, 16])
def test_swiglu_fp4_full_size_sampled(nq, T):
    """The NVFP4 SwiGLU block at the 27B-class MLP shape (K=5120, N=17408), sampled rows."""
    K, N = 5120, 17408
    p = si.swiglu_fp4_problem(T, K, N, 720 + T)
    wg, wu = _swiglu_fp4(nq, p, T, K, N)
    h = gu.host_f64(nq.swiglu_fp4(gu.dev_bf16(p["x"]), *wg, p["gg"], *wu, p["gu"], N))
    rows = gu.sample_rows(N, 256, 17)
    g, u, _ = oracle.swiglu_fp4_rows(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, rows)
    assert gu.rel_err(h[:, rows], (g / (1.0 + np.exp(-g)) * u).T) <= gu.TOL


def test_swiglu_fp4_scales_are_per_matrix_and_deterministic(nq):
    """Swapping the two tensor scales changes H (each scale belongs to its matrix); equal calls
    give equal bits; tensor-core batches agree with 8-token slices within the bar."""
    T, K, N = 20, 1024, 272
    p = si.swiglu_fp4_problem(T, K, N, 740)
    wg, wu = _swiglu_fp4(nq, p, T, K, N)
    x = gu.dev_bf16(p["x"])
    h1 = nq.swiglu_fp4(x, *wg, p["gg"], *wu, p["gu"], N)
    h2 = nq.swiglu_fp4(x, *wg, p["gg"], *wu, p["gu"], N)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    hs = nq.swiglu_fp4(x, *wg, p["gu"], *wu, p["gg"], N)
    assert not torch.equal(h1.view(torch.int16), hs.view(torch.int16))
    prev = nq.tensor_core_batches(0)
    try:
        h_sl = nq.swiglu_fp4(x, *wg, p["gg"], *wu, p["gu"], N)
    finally:
        nq.tensor_core_batches(prev)
    g, u, _ = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    ref = g / (1.0 + np.exp(-g)) * u
    for h in (h1, h_sl):
        assert gu.rel_err(gu.host_f64(h), ref) <= gu.TOL
    for T8 in (3, 8):                       # the 8-token kernel with the swapped scales as well
        q = si.swiglu_fp4_problem(T8, K, N, 741 + T8)
        qg, qu = _swiglu_fp4(nq, q, T8, K, N)
        hq = gu.host_f64(nq.swiglu_fp4(gu.dev_bf16(q["x"]), *qg, q["gu"], *qu, q["gg"], N))
        g, u, _ = oracle.swiglu_fp4(q["x"], q["cg"], q["sfg"], q["gu"], q["cu"], q["sfu"], q["gg"], T8, K, N)
        assert gu.rel_err(hq, g / (1.0 + np.exp(-g)) * u) <= gu.TOL
    nq.device_error()
