"""Pins of the CPU oracle against things other than itself (CPU only).

- decoders against the library casts of NumPy (fp16) and PyTorch (bf16), exhaustively;
- hand-derived closed-form fixtures in tests/golden/;
- the independent NumPy twin (byte-view unpack, BLAS contraction);
- invariants: zero-point codes give exact zeros, one-hot X selects a weight column,
  all-zero codes give -z*s, linearity in X, the Q5 planes reduce to the Q4 rule;
- planted mistakes in a copy of the oracle source are caught by these pins.
"""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from oracle import twin
from tests.golden import fixtures as fx


# ---------------------------------------------------------------- scalar decoders

def test_fp16_decoder_exhaustive_vs_numpy():
    L = oracle.lib()
    ours = np.array([L.orc_fp16_to_f64(h) for h in range(65536)])
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros too
    assert math.copysign(1.0, L.orc_fp16_to_f64(0x8000)) == -1.0


def test_bf16_decoder_exhaustive_vs_torch():
    L = oracle.lib()
    ours = np.array([L.orc_bf16_to_f64(b) for b in range(65536)])
    ref = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_round_bf16_vs_torch_cast():
    """fp32-representable inputs: a single RNE rounding to bf16 must equal PyTorch's cast."""
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(5000) * 1e30).astype(np.float32),
        (g.standard_normal(5000) * 1e-39).astype(np.float32),       # bf16 subnormals
        np.array([3.3895314e38, -3.3895314e38, 1e-45, 0.0, -0.0], np.float32),
        # exact ties between neighbouring bf16 values: 1 + (2m+1) * 2^-8
        (1.0 + (2 * np.arange(64) + 1) * 2.0**-8).astype(np.float32),
    ])
    ours = np.array([oracle.round_bf16(float(v)) for v in vals], np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_bf16_ties_to_even_by_hand():
    # 1 + 2^-8 lies halfway between 1 (even mantissa) and 1 + 2^-7: goes to 1.
    assert oracle.round_bf16(1.0 + 2.0**-8) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1+2^-7 (odd) and 1+2^-6 (even): goes up.
    assert oracle.round_bf16(1.0 + 3 * 2.0**-8) == 0x3F82
    # past the largest finite bf16 by half a quantum -> +inf
    assert oracle.round_bf16(2.0**128) == 0x7F80
    assert oracle.round_bf16(-0.0) == 0x8000


# ---------------------------------------------------------------- golden fixtures

def _spot_w(w, spots):
    for sp in spots:
        assert w[sp["n"], sp["k"]] == np.float32(sp["w"]), sp


def test_golden_q4_closed_form():
    f = fx.load("q4_closed_form.json")
    wq, s, x = fx.words(f["wq_rows_hex"]), fx.halves(f["s_rows_hex"]), fx.x_bits(f)
    _spot_w(oracle.dequant_q4(wq, s, f["K"], f["N"]), f["w_expected_spot"])
    y = oracle.gemm_q4(x, wq, s, f["T"], f["K"], f["N"])
    assert np.array_equal(y, np.array(f["y_expected"]))


def test_golden_q5_closed_form():
    f = fx.load("q5_closed_form.json")
    wn, wh, s, x = fx.words(f["wn_rows_hex"]), fx.words(f["wh_rows_hex"]), fx.halves(f["s_rows_hex"]), fx.x_bits(f)
    _spot_w(oracle.dequant_q5(wn, wh, s, f["K"], f["N"]), f["w_expected_spot"])
    y = oracle.gemm_q5(x, wn, wh, s, f["T"], f["K"], f["N"])
    assert np.array_equal(y, np.array(f["y_expected"]))


def test_golden_fp16_scale_edges():
    f = fx.load("fp16_scale_edges.json")
    wq, s, x = fx.words(f["wq_rows_hex"]), fx.halves(f["s_rows_hex"]), fx.x_bits(f)
    _spot_w(oracle.dequant_q4(wq, s, f["K"], f["N"]), f["w_expected_spot"])
    y = oracle.gemm_q4(x, wq, s, f["T"], f["K"], f["N"])
    assert np.array_equal(y, np.array(f["y_expected"]))


def test_golden_swiglu_closed_form():
    f = fx.load("swiglu_closed_form.json")
    wg, wu = fx.words(f["wg_rows_hex"]), fx.words(f["wu_rows_hex"])
    sg, su = fx.halves(f["sg_rows_hex"]), fx.halves(f["su_rows_hex"])
    x = fx.x_bits(f)
    g, u, h = oracle.swiglu_q4(x, wg, sg, wu, su, f["T"], f["K"], f["N"])
    assert np.array_equal(g, np.array(f["g_expected"]))
    assert np.array_equal(u, np.array(f["u_expected"]))
    assert np.array_equal(h, fx.halves(f["h_expected_hex"]))


# ---------------------------------------------------------------- the twin

# up to 64 tokens: the larger speculative-verify batches (several requests x draft tokens)
TWIN_SHAPES = [(1, 256, 128, 0), (3, 192, 48, 11), (8, 640, 80, 12), (5, 64, 16, 13), (9, 128, 32, 14),
               (64, 192, 48, 15)]


@pytest.mark.parametrize("T,K,N,seed", TWIN_SHAPES)
def test_q4_dequant_and_gemm_vs_twin(T, K, N, seed):
    p = si.q4_problem(T, K, N, seed)
    w = oracle.dequant_q4(p["wq"], p["s"], K, N)
    w_twin = twin.weights(twin.codes_q4(p["wq"], K), p["s"], 8)
    assert np.array_equal(w.view(np.uint32), w_twin.view(np.uint32))   # bit-exact
    y = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    y_twin = twin.gemm_q4(p["x"], p["wq"], p["s"], K)
    assert np.max(np.abs(y - y_twin)) <= 1e-12 * np.max(np.abs(y_twin))


@pytest.mark.parametrize("T,K,N,seed", TWIN_SHAPES)
def test_q5_dequant_and_gemm_vs_twin(T, K, N, seed):
    p = si.q5_problem(T, K, N, seed)
    w = oracle.dequant_q5(p["wn"], p["wh"], p["s"], K, N)
    w_twin = twin.weights(twin.codes_q5(p["wn"], p["wh"], K), p["s"], 16)
    assert np.array_equal(w.view(np.uint32), w_twin.view(np.uint32))
    y = oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)
    y_twin = twin.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], K)
    assert np.max(np.abs(y - y_twin)) <= 1e-12 * np.max(np.abs(y_twin))


def test_token_rows_are_independent():
    """Row t of Y depends only on row t of X: a 40-token batch equals its 8-token slices
    computed separately (and the rows variant agrees), for both code widths."""
    T, K, N = 40, 256, 48
    p = si.q4_problem(T, K, N, 16)
    y = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    for t0 in range(0, T, 8):
        part = oracle.gemm_q4(np.ascontiguousarray(p["x"][t0:t0 + 8]), p["wq"], p["s"], 8, K, N)
        assert np.array_equal(y[t0:t0 + 8], part)
    rows = np.arange(N, dtype=np.int32)
    assert np.array_equal(oracle.gemm_q4_rows(p["x"], p["wq"], p["s"], T, K, rows).T, y)
    q = si.q5_problem(T, K, N, 17)
    y5 = oracle.gemm_q5(q["x"], q["wn"], q["wh"], q["s"], T, K, N)
    part = oracle.gemm_q5(np.ascontiguousarray(q["x"][32:]), q["wn"], q["wh"], q["s"], 8, K, N)
    assert np.array_equal(y5[32:], part)


def test_rows_variant_matches_full():
    p = si.q4_problem(4, 320, 64, 21)
    y = oracle.gemm_q4(p["x"], p["wq"], p["s"], 4, 320, 64)
    rows = [0, 17, 63, 5]
    yr = oracle.gemm_q4_rows(p["x"], p["wq"], p["s"], 4, 320, rows)
    assert np.array_equal(yr, y[:, rows].T)
    q = si.q5_problem(2, 192, 32, 22)
    y5 = oracle.gemm_q5(q["x"], q["wn"], q["wh"], q["s"], 2, 192, 32)
    y5r = oracle.gemm_q5_rows(q["x"], q["wn"], q["wh"], q["s"], 2, 192, [31, 0])
    assert np.array_equal(y5r, y5[:, [31, 0]].T)


def test_swiglu_vs_twin():
    T, K, N = 8, 256, 48
    p = si.swiglu_problem(T, K, N, 31)
    g, u, h = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    g_t = twin.gemm_q4(p["x"], p["wg"], p["sg"], K)
    u_t = twin.gemm_q4(p["x"], p["wu"], p["su"], K)
    assert np.max(np.abs(g - g_t)) <= 1e-12 * np.max(np.abs(g_t))
    assert np.max(np.abs(u - u_t)) <= 1e-12 * np.max(np.abs(u_t))
    h_t = twin.silu(g_t) * u_t
    h_ours = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    # one bf16 rounding of nearly equal fp64 values: at most one quantum apart
    assert np.all(np.abs(h_ours - h_t) <= 2.0**-7 * np.abs(h_t) + 1e-30)
    gr, ur, hr = oracle.swiglu_q4_rows(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, [3, 40])
    assert np.array_equal(hr, h[:, [3, 40]].T) and np.array_equal(gr, g[:, [3, 40]].T)


def test_swiglu_q5_vs_twin():
    T, K, N = 5, 320, 32
    p = si.swiglu_q5_problem(T, K, N, 37)
    g, u, h = oracle.swiglu_q5(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"], p["su"],
                               T, K, N)
    g_t = twin.gemm_q5(p["x"], p["wgn"], p["wgh"], p["sg"], K)
    u_t = twin.gemm_q5(p["x"], p["wun"], p["wuh"], p["su"], K)
    assert np.max(np.abs(g - g_t)) <= 1e-12 * np.max(np.abs(g_t))
    assert np.max(np.abs(u - u_t)) <= 1e-12 * np.max(np.abs(u_t))
    h_t = twin.silu(g_t) * u_t
    h_ours = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(h_ours - h_t) <= 2.0**-7 * np.abs(h_t) + 1e-30)
    rows = [31, 0, 9]
    gr, ur, hr = oracle.swiglu_q5_rows(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"],
                                       p["su"], T, K, rows)
    assert np.array_equal(hr, h[:, rows].T) and np.array_equal(ur, u[:, rows].T)


def test_swiglu_q5_closed_forms():
    """Codes equal to the zero point (16: nibble 0, high bit 1) contribute exactly nothing:
    an all-16 gate gives g = 0, so h = silu(0) * u is a zero carrying u's sign; an all-16 up
    gives u = 0 and h a zero carrying g's sign.
    A single code 17 (q - z = +1) in gate group 0 with a scale of 1 leaves g = x[t, k0]."""
    T, K, N = 3, 128, 16
    p = si.swiglu_q5_problem(T, K, N, 41)
    zn = np.zeros_like(p["wgn"])
    zh = np.full_like(p["wgh"], 0xFFFFFFFF)
    g, u, h = oracle.swiglu_q5(p["x"], zn, zh, p["sg"], p["wun"], p["wuh"], p["su"], T, K, N)
    assert np.all(g == 0.0) and np.array_equal(h, np.where(u < 0, 0x8000, 0).astype(np.uint16))
    g, u, h = oracle.swiglu_q5(p["x"], p["wgn"], p["wgh"], p["sg"], zn, zh, p["su"], T, K, N)
    assert np.all(u == 0.0) and np.array_equal(h, np.where(g < 0, 0x8000, 0).astype(np.uint16))
    wgn = zn.copy()
    wgn[:, 0] = 1 << 4 * 3          # row n, k0 = 3: nibble 1 with high bit 1 -> q = 17
    sg = p["sg"].copy()
    sg[:, 0] = np.float16(1.0).view(np.uint16)
    g, u, h = oracle.swiglu_q5(p["x"], wgn, zh, sg, p["wun"], p["wuh"], p["su"], T, K, N)
    xk0 = torch.from_numpy(p["x"][:, 3].view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(g, np.repeat(xk0[:, None], N, axis=1))


def test_silu_closed_forms():
    assert oracle.silu_mul(0.0, 5.0) == 0.0
    assert oracle.silu_mul(50.0, 1.0) == pytest.approx(50.0, rel=1e-15)   # silu(g) -> g
    assert abs(oracle.silu_mul(-50.0, 1.0)) < 1e-19                      # silu(g) -> 0
    gs = np.linspace(-20, 20, 401)
    ours = np.array([oracle.silu_mul(v, 1.0) for v in gs])
    assert np.max(np.abs(ours - twin.silu(gs))) <= 1e-14


# ---------------------------------------------------------------- invariants

def test_all_zero_codes_give_minus_z_times_scale():
    K, N = 128, 32
    s = si.scales(np.random.default_rng(3), N, K)
    sf = twin.scales_f32(s)
    w4 = oracle.dequant_q4(np.zeros((N, K // 8), np.uint32), s, K, N)
    assert np.array_equal(w4, np.repeat(-8.0 * sf, 64, axis=1))
    w5 = oracle.dequant_q5(np.zeros((N, K // 8), np.uint32), np.zeros((N, K // 32), np.uint32), s, K, N)
    assert np.array_equal(w5, np.repeat(-16.0 * sf, 64, axis=1))


def test_zero_point_codes_give_exact_zero_output():
    T, K, N = 8, 256, 16
    p = si.q4_problem(T, K, N, 4)
    y = oracle.gemm_q4(p["x"], np.full((N, K // 8), 0x88888888, np.uint32), p["s"], T, K, N)
    assert np.all(y == 0.0)
    y5 = oracle.gemm_q5(p["x"], np.zeros((N, K // 8), np.uint32), np.full((N, K // 32), 0xFFFFFFFF, np.uint32),
                        p["s"], T, K, N)
    assert np.all(y5 == 0.0)


def test_one_hot_x_with_unit_scales_selects_codes():
    K, N = 192, 24
    p = si.q4_problem(1, K, N, 5)
    s1 = np.full((N, K // 64), 0x3C00, np.uint16)         # 1.0
    codes = twin.codes_q4(p["wq"], K)
    for k in (0, 1, 63, 64, 130, 191):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = oracle.gemm_q4(x, p["wq"], s1, 1, K, N)
        assert np.array_equal(y[0], (codes[:, k] - 8).astype(np.float64))
    q = si.q5_problem(1, K, N, 6)
    codes5 = twin.codes_q5(q["wn"], q["wh"], K)
    for k in (0, 31, 32, 100):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = oracle.gemm_q5(x, q["wn"], q["wh"], s1, 1, K, N)
        assert np.array_equal(y[0], (codes5[:, k] - 16).astype(np.float64))


def test_linearity_in_x():
    """Y(2*X1 - X2) = 2*Y(X1) - Y(X2) with small-integer X, where every X is exact in bf16."""
    T, K, N = 4, 256, 32
    p = si.q4_problem(T, K, N, 8)
    g = np.random.default_rng(9)
    a = g.integers(-8, 9, size=(T, K)).astype(np.float32)
    b = g.integers(-8, 9, size=(T, K)).astype(np.float32)
    xa, xb, xc = si.bf16_bits(a), si.bf16_bits(b), si.bf16_bits(2 * a - b)
    ya = oracle.gemm_q4(xa, p["wq"], p["s"], T, K, N)
    yb = oracle.gemm_q4(xb, p["wq"], p["s"], T, K, N)
    yc = oracle.gemm_q4(xc, p["wq"], p["s"], T, K, N)
    assert np.max(np.abs(yc - (2 * ya - yb))) <= 1e-12 * np.max(np.abs(yc))


def test_q5_planes_reduce_to_q4_rule():
    K, N = 128, 16
    p = si.q5_problem(1, K, N, 10)
    zero_hi = np.zeros((N, K // 32), np.uint32)
    w5 = oracle.dequant_q5(p["wn"], zero_hi, p["s"], K, N)
    w4 = oracle.dequant_q4(p["wn"], p["s"], K, N)
    sf = np.repeat(twin.scales_f32(p["s"]), 64, axis=1)
    assert np.array_equal(w5, w4 - 8.0 * sf)          # s*(nib-16) = s*(nib-8) - 8s, exact here
    one_hi = np.full((N, K // 32), 0xFFFFFFFF, np.uint32)
    w5z = oracle.dequant_q5(np.zeros((N, K // 8), np.uint32), one_hi, p["s"], K, N)
    assert np.all(w5z == 0.0)


def test_dequant_is_exact_product():
    """Every dequantised weight equals the exact real product s*(q-z) (checked in fp64)."""
    K, N = 256, 64
    p = si.q5_problem(1, K, N, 14)
    w = oracle.dequant_q5(p["wn"], p["wh"], p["s"], K, N).astype(np.float64)
    exact = np.repeat(twin.scales_f32(p["s"]).astype(np.float64), 64, axis=1) * \
        (twin.codes_q5(p["wn"], p["wh"], K) - 16)
    assert np.array_equal(w, exact)


# ---------------------------------------------------------------- NVFP4

def test_e4m3_decoder_exhaustive_vs_torch():
    ours = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    ref = twin.e4m3_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))   # -0 stays -0


def test_e2m1_decoder_all_codes():
    ours = np.array([oracle.e2m1_to_f64(c) for c in range(16)])
    assert np.array_equal(ours, twin.e2m1_f32(np.arange(16, dtype=np.uint8)).astype(np.float64))
    # the format's value set: eight magnitudes, the negative codes mirror the positive ones
    assert list(ours[:8]) == sorted(ours[:8]) and ours[1] == 0.5 and ours[2] == 1.0 and ours[7] == 6.0
    assert np.array_equal(ours[8:], -ours[:8]) and np.signbit(ours[8]) and ours[8] == 0.0


FP4_SHAPES = [(1, 256, 32, 0), (3, 192, 48, 1), (8, 640, 16, 2), (20, 64, 32, 3)]


@pytest.mark.parametrize("T,K,N,seed", FP4_SHAPES)
def test_fp4_dequant_and_gemm_vs_twin(T, K, N, seed):
    p = si.fp4_problem(T, K, N, 60 + seed)
    w = oracle.dequant_fp4(p["codes"], p["sf"], p["g"], K, N)
    w_twin = twin.weights_fp4(p["codes"], p["sf"], p["g"], K)
    assert np.array_equal(w.view(np.uint32), w_twin.view(np.uint32))
    y = oracle.gemm_fp4(p["x"], p["codes"], p["sf"], p["g"], T, K, N)
    y_twin = twin.gemm_fp4(p["x"], p["codes"], p["sf"], p["g"], K)
    assert np.max(np.abs(y - y_twin)) <= 1e-12 * np.max(np.abs(y_twin))
    rows = np.array([0, N - 1, N // 2], np.int32)
    assert np.array_equal(oracle.gemm_fp4_rows(p["x"], p["codes"], p["sf"], p["g"], T, K, rows).T, y[:, rows])


def test_fp4_block_structure():
    """One scale per 16 elements: a block scale of 2 doubles exactly its own 16 weights; the
    tensor scale multiplies every weight; the weights are the exact products (fp64 check)."""
    K, N = 128, 16
    p = si.fp4_problem(1, K, N, 70, g=1.0)
    w = oracle.dequant_fp4(p["codes"], p["sf"], 1.0, K, N).astype(np.float64)
    sf2 = p["sf"].copy()
    sf2[3, 5] = 0x40                                   # e4m3 2.0
    sf1 = p["sf"].copy()
    sf1[3, 5] = 0x38                                   # e4m3 1.0
    w2 = oracle.dequant_fp4(p["codes"], sf2, 1.0, K, N).astype(np.float64)
    w1 = oracle.dequant_fp4(p["codes"], sf1, 1.0, K, N).astype(np.float64)
    assert np.array_equal(w2[3, 80:96], 2.0 * w1[3, 80:96])
    mask = np.ones_like(w, bool)
    mask[3, 80:96] = False
    assert np.array_equal(w2[mask], w[mask])
    wg = oracle.dequant_fp4(p["codes"], p["sf"], 0.25, K, N).astype(np.float64)
    assert np.array_equal(wg, 0.25 * w)
    exact = np.repeat(twin.e4m3_f32(p["sf"]).astype(np.float64), 16, axis=1) * \
        twin.e2m1_f32(twin.codes_q4(p["codes"], K).astype(np.uint8)).astype(np.float64)
    assert np.array_equal(w, exact)


def test_swiglu_fp4_vs_twin():
    """The NVFP4 gate/up block against the NumPy twin, with different gate and up tensor scales
    (a swapped or shared scale would fail), and its row variant against the full block."""
    T, K, N = 6, 256, 32
    p = si.swiglu_fp4_problem(T, K, N, 43)
    assert p["gg"] != p["gu"]
    g, u, h = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    g_t = twin.gemm_fp4(p["x"], p["cg"], p["sfg"], p["gg"], K)
    u_t = twin.gemm_fp4(p["x"], p["cu"], p["sfu"], p["gu"], K)
    assert np.max(np.abs(g - g_t)) <= 1e-12 * np.max(np.abs(g_t))
    assert np.max(np.abs(u - u_t)) <= 1e-12 * np.max(np.abs(u_t))
    h_t = twin.silu(g_t) * u_t
    h_ours = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(h_ours - h_t) <= 2.0**-7 * np.abs(h_t) + 1e-30)
    rows = [31, 0, 7]
    gr, ur, hr = oracle.swiglu_fp4_rows(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, rows)
    assert np.array_equal(hr, h[:, rows].T) and np.array_equal(gr, g[:, rows].T) and np.array_equal(ur, u[:, rows].T)


def test_swiglu_fp4_closed_forms():
    """Code 0 is +0: an all-zero gate gives g = 0 and h a zero carrying u's sign; an all-zero up
    gives u = 0 and h a zero carrying g's sign. Doubling the up tensor scale doubles u exactly."""
    T, K, N = 2, 128, 16
    p = si.swiglu_fp4_problem(T, K, N, 47)
    z = np.zeros_like(p["cg"])
    g, u, h = oracle.swiglu_fp4(p["x"], z, p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    assert np.all(g == 0.0) and np.array_equal(h, np.where(u < 0, 0x8000, 0).astype(np.uint16))
    g, u, h = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], z, p["sfu"], p["gu"], T, K, N)
    assert np.all(u == 0.0) and np.array_equal(h, np.where(g < 0, 0x8000, 0).astype(np.uint16))
    _, u1, _ = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], p["gu"], T, K, N)
    _, u2, _ = oracle.swiglu_fp4(p["x"], p["cg"], p["sfg"], p["gg"], p["cu"], p["sfu"], 2 * p["gu"], T, K, N)
    assert np.array_equal(u2, 2.0 * u1)


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = [
    ("nibble order reversed", "(4 * (k & 7))) & 0xFu);\n}", "(4 * (7 - (k & 7)))) & 0xFu);\n}"),
    ("zero point 7", "wrow[k] = dequant(s, K, n, k, q4_code(wq, K, n, k), 8)", "wrow[k] = dequant(s, K, n, k, q4_code(wq, K, n, k), 7)"),
    ("group of 32", "(k >> 6)]);", "(k >> 5) % (K / 64)]);"),
    ("q5 high bit ignored", "return nib | (hi << 4);", "return nib | (0 << 4);"),
    ("x row stride transposed", "orc_bf16_to_f64(x[(size_t)t * K + k]);\n        out[t] = acc;\n    }\n}\n\nstatic void row_q5",
     "orc_bf16_to_f64(x[(size_t)k * T + t]);\n        out[t] = acc;\n    }\n}\n\nstatic void row_q5"),
    ("fp16 subnormal off by one", "ldexp((double)f, -24)", "ldexp((double)f, -23)"),
    ("fp4 block of 32", "sf[(size_t)n * (K / 16) + (k >> 4)]", "sf[(size_t)n * (K / 16) + (k >> 5)]"),
    ("e2m1 exponent bias 0", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e4m3 subnormal scale", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
]


def _build_mutant(src: str, tmp: str) -> "ctypes.CDLL":
    import ctypes
    c = os.path.join(tmp, "m.c")
    so = os.path.join(tmp, "m.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-o", so, c, "-lm"])
    L = ctypes.CDLL(so)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.orc_gemm_q4.argtypes = [P, P, P, I, I, I, P]
    L.orc_gemm_q5.argtypes = [P, P, P, P, I, I, I, P]
    L.orc_gemm_fp4.argtypes = [P, P, P, ctypes.c_float, I, I, I, P]
    return L


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    """Plant one plausible mistake in a copy of the oracle; the twin and fixtures must see it."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as tmp:
        L = _build_mutant(src.replace(old, new), tmp)
        caught = False
        # random problems vs the twin (T=3 so a transposed X stride reads the wrong rows)
        T, K, N = 3, 256, 32
        p = si.q4_problem(T, K, N, 40)
        y = np.empty((T, N))
        L.orc_gemm_q4(oracle._p(p["x"]), oracle._p(p["wq"]), oracle._p(p["s"]), T, K, N, oracle._p(y))
        caught |= not np.allclose(y, twin.gemm_q4(p["x"], p["wq"], p["s"], K), rtol=1e-9, atol=0)
        q = si.q5_problem(T, K, N, 41)
        y5 = np.empty((T, N))
        L.orc_gemm_q5(oracle._p(q["x"]), oracle._p(q["wn"]), oracle._p(q["wh"]), oracle._p(q["s"]), T, K, N,
                      oracle._p(y5))
        caught |= not np.allclose(y5, twin.gemm_q5(q["x"], q["wn"], q["wh"], q["s"], K), rtol=1e-9, atol=0)
        # the fp16-edge fixture
        f = fx.load("fp16_scale_edges.json")
        wq, s, x = fx.words(f["wq_rows_hex"]), fx.halves(f["s_rows_hex"]), fx.x_bits(f)
        yf = np.empty((f["T"], f["N"]))
        L.orc_gemm_q4(oracle._p(x), oracle._p(wq), oracle._p(s), f["T"], f["K"], f["N"], oracle._p(yf))
        caught |= not np.array_equal(yf, np.array(f["y_expected"]))
        # NVFP4 vs its twin, with block scales that include e4m3 subnormals
        r = si.fp4_problem(T, K, N, 42)
        r["sf"][:, ::3] = np.arange(1, 8, dtype=np.uint8)[np.arange(r["sf"][:, ::3].size) % 7].reshape(
            r["sf"][:, ::3].shape)
        y4 = np.empty((T, N))
        L.orc_gemm_fp4(oracle._p(r["x"]), oracle._p(r["codes"]), oracle._p(r["sf"]), r["g"], T, K, N,
                       oracle._p(y4))
        caught |= not np.allclose(y4, twin.gemm_fp4(r["x"], r["codes"], r["sf"], r["g"], K), rtol=1e-9, atol=0)
        assert caught, name
