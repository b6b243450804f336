"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU oracle on the
same seeded inputs. Dequantised weights must match bit for bit, through both decoders the
kernels use; outputs within max|y - y_ref| / max|y_ref| <= 5e-3. The bf16 output rounding
alone is up to 2^-8 (3.9e-3) relative to |y| (8 significant bits, half an ulp of 2^-7), so
the bound leaves about 1.1e-3 for fp32 accumulation in any order, where ~1e-6 is expected."""
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


# ---------------------------------------------------------------- dequant: bit-exact

DEQ_SHAPES = [(256, 128, 0), (192, 48, 1), (64, 16, 2), (640, 272, 3), (5120, 6144, 4)]


def _dequant_case(nq, bits, operands, K, N, seed):
    if bits == 4:
        p = si.q4_problem(1, K, N, seed)
        w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
        w_gpu = nq.dequant_q4_debug(*w, K, N, operands=operands).cpu().numpy()
        w_ref = oracle.dequant_q4(p["wq"], p["s"], K, N)
    else:
        p = si.q5_problem(1, K, N, seed)
        w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
        w_gpu = nq.dequant_q5_debug(*w, K, N, operands=operands).cpu().numpy()
        w_ref = oracle.dequant_q5(p["wn"], p["wh"], p["s"], K, N)
    assert w_gpu.shape == w_ref.shape
    assert np.array_equal(w_gpu.view(np.uint32), w_ref.view(np.uint32))


# Both decoders: fp16 operands (the T <= 2 kernels: 1024 + q / 1024 + 16 q) and bf16
# operands (the T >= 3 kernels: 128 + q), each dumped through the same decode routine the
# projection kernels call, compared bit for bit with the CPU definition.
@pytest.mark.parametrize("operands", ["f16", "bf16"])
@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("K,N,seed", DEQ_SHAPES)
def test_dequant_bit_exact(nq, bits, operands, K, N, seed):
    _dequant_case(nq, bits, operands, K, N, seed)


# the full decode / verify weight shapes (K=5120 with N=17408 Q4 and N=6144 Q5)
@pytest.mark.parametrize("operands", ["f16", "bf16"])
@pytest.mark.parametrize("bits,K,N,seed", [(4, 5120, 17408, 1), (5, 5120, 6144, 2)])
def test_dequant_bit_exact_full_size(nq, bits, operands, K, N, seed):
    _dequant_case(nq, bits, operands, K, N, seed)


def test_dequant_every_code_both_decoders(nq):
    """Every code value at every position of a tile: codes cycle through 0..15 (Q4) and
    0..31 (Q5) with the high plane driven by bit 4, so each nibble slot, each high-bit
    position and each K step of the fragment layout sees every value, under scales that
    include fp16 subnormals, the largest finite fp16 and negative values."""
    K, N = 256, 32
    k = np.arange(K)
    n = np.arange(N)[:, None]
    q4 = (k[None, :] + 3 * n) % 16
    q5 = (k[None, :] * 7 + 5 * n) % 32
    wq = np.zeros((N, K // 8), np.uint32)
    wn = np.zeros((N, K // 8), np.uint32)
    wh = np.zeros((N, K // 32), np.uint32)
    for i in range(8):
        wq |= (q4[:, i::8].astype(np.uint32) << np.uint32(4 * i))
        wn |= ((q5[:, i::8] & 15).astype(np.uint32) << np.uint32(4 * i))
    for i in range(32):
        wh |= ((q5[:, i::32] >> 4).astype(np.uint32) << np.uint32(i))
    scale_bits = np.array([0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0xBC00, 0x8001, 0x2E66], np.uint16)
    s = scale_bits[(np.arange(N)[:, None] + np.arange(K // 64)[None, :]) % len(scale_bits)]
    s = np.ascontiguousarray(s)
    ref4 = oracle.dequant_q4(wq, s, K, N)
    ref5 = oracle.dequant_q5(wn, wh, s, K, N)
    w4 = gu.pack_q4(nq, wq, s, K, N)
    w5 = gu.pack_q5(nq, wn, wh, s, K, N)
    for operands in ("f16", "bf16"):
        g4 = nq.dequant_q4_debug(*w4, K, N, operands=operands).cpu().numpy()
        g5 = nq.dequant_q5_debug(*w5, K, N, operands=operands).cpu().numpy()
        assert np.array_equal(g4.view(np.uint32), ref4.view(np.uint32)), operands
        assert np.array_equal(g5.view(np.uint32), ref5.view(np.uint32)), operands


# ---------------------------------------------------------------- projections, small/ragged

GEMM_SHAPES = [
    # T, K, N, seed: tiny case, ragged row tiles (odd tile count), one group, several
    # chunks, every T, K slabs at T=8 (K > 6144) with a ragged last slab
    (1, 256, 128, 0), (3, 192, 48, 1), (5, 640, 80, 2), (7, 64, 16, 3), (8, 1024, 272, 4),
    (2, 4096, 496, 5), (4, 2048, 1040, 6), (6, 320, 4112, 7), (8, 6208, 48, 8), (8, 17408, 64, 9),
    (1, 17408, 32, 10), (8, 12352, 112, 11),
]


@pytest.mark.parametrize("T,K,N,seed", GEMM_SHAPES)
def test_gemm_q4_parity(nq, T, K, N, seed):
    p = si.q4_problem(T, K, N, seed)
    wq = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *wq, N))
    y_ref = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    assert gu.rel_err(y, y_ref) <= gu.TOL


@pytest.mark.parametrize("T,K,N,seed", GEMM_SHAPES)
def test_gemm_q5_parity(nq, T, K, N, seed):
    p = si.q5_problem(T, K, N, seed + 100)
    wq = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(p["x"]), *wq, N))
    y_ref = oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)
    assert gu.rel_err(y, y_ref) <= gu.TOL


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemm_every_T(nq, T):
    K, N = 1536, 208
    p = si.q4_problem(T, K, N, 50 + T)
    wq = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *wq, N))
    assert gu.rel_err(y, oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)) <= gu.TOL
    q = si.q5_problem(T, K, N, 60 + T)
    wq5 = gu.pack_q5(nq, q["wn"], q["wh"], q["s"], K, N)
    y5 = gu.host_f64(nq.gemm_q5(gu.dev_bf16(q["x"]), *wq5, N))
    assert gu.rel_err(y5, oracle.gemm_q5(q["x"], q["wn"], q["wh"], q["s"], T, K, N)) <= gu.TOL


SWIGLU_SHAPES = [(8, 256, 48, 0), (1, 640, 16, 1), (5, 1024, 272, 2), (8, 6208, 32, 3), (3, 17408, 48, 4)]


@pytest.mark.parametrize("T,K,N,seed", SWIGLU_SHAPES)
def test_swiglu_q4_parity(nq, T, K, N, seed):
    p = si.swiglu_problem(T, K, N, seed)
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    h = gu.host_f64(nq.swiglu_q4(gu.dev_bf16(p["x"]), *wg, *wu, N))
    g, u, h_ref_bits = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    h_exact = g / (1.0 + np.exp(-g)) * u
    assert gu.rel_err(h, h_exact) <= gu.TOL


SWIGLU_Q5_SHAPES = [(8, 256, 48, 0), (1, 640, 16, 1), (2, 1024, 272, 2), (4, 17408, 64, 3),
                    (8, 6208, 32, 4), (6, 320, 112, 5), (3, 5120, 1040, 6)]


def _swiglu_q5_dev(nq, p, T, K, N):
    wg = gu.pack_q5(nq, p["wgn"], p["wgh"], p["sg"], K, N)
    wu = gu.pack_q5(nq, p["wun"], p["wuh"], p["su"], K, N)
    return nq.swiglu_q5(gu.dev_bf16(p["x"]), *wg, *wu, N)


@pytest.mark.parametrize("T,K,N,seed", SWIGLU_Q5_SHAPES)
def test_swiglu_q5_parity(nq, T, K, N, seed):
    p = si.swiglu_q5_problem(T, K, N, seed + 200)
    h = gu.host_f64(_swiglu_q5_dev(nq, p, T, K, N))
    g, u, _ = oracle.swiglu_q5(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"], p["su"],
                               T, K, N)
    assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL


def test_swiglu_q5_zero_point_codes_give_zero(nq):
    """Gate codes all equal to z = 16 make g exactly 0, so every h is a zero; the same for
    up codes. The kernel's zero-point correction must cancel exactly, not approximately."""
    T, K, N = 8, 1024, 64
    p = si.swiglu_q5_problem(T, K, N, 250)
    zn, zh = np.zeros_like(p["wgn"]), np.full_like(p["wgh"], 0xFFFFFFFF)
    q = dict(p, wgn=zn, wgh=zh)
    assert np.all(gu.host_f64(_swiglu_q5_dev(nq, q, T, K, N)) == 0.0)
    q = dict(p, wun=zn, wuh=zh)
    assert np.all(gu.host_f64(_swiglu_q5_dev(nq, q, T, K, N)) == 0.0)


def test_swiglu_q5_block_full_size_sampled(nq):
    """The gate/up block of the SwiGLU workload (T=8, K=5120, N=17408) with 5-bit weights,
    in the launch configuration of the full size, checked on sampled output rows; then the
    down projection (Q5, K=17408 -> N=5120) on the GPU's own H."""
    c = si.SWIGLU_Q4
    T, K, N = c["T"], c["K"], c["N"]
    p = si.swiglu_q5_problem(T, K, N, c["seed"] + 500)
    h_dev = _swiglu_q5_dev(nq, p, T, K, N)
    rows = gu.sample_rows(N, 256, 2)
    g, u, _ = oracle.swiglu_q5_rows(p["x"], p["wgn"], p["wgh"], p["sg"], p["wun"], p["wuh"],
                                    p["su"], T, K, rows)
    assert gu.rel_err(gu.host_f64(h_dev)[:, rows], (g / (1.0 + np.exp(-g)) * u).T) <= gu.TOL
    d = si.SWIGLU_DOWN
    pd = si.q5_problem(T, d["K"], d["N"], c["seed"] + 1500)
    wd = gu.pack_q5(nq, pd["wn"], pd["wh"], pd["s"], d["K"], d["N"])
    y = gu.host_f64(nq.gemm_q5(h_dev, *wd, d["N"]))
    h_bits = h_dev.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = gu.sample_rows(d["N"], 256, 3)
    y_ref = oracle.gemm_q5_rows(h_bits, pd["wn"], pd["wh"], pd["s"], T, d["K"], rows)
    assert gu.rel_err(y[:, rows], y_ref.T) <= gu.TOL


# ---------------------------------------------------------------- the five workloads

def test_workload_tiny_q4(nq):
    c = si.TINY_Q4
    p = si.q4_problem(c["T"], c["K"], c["N"], c["seed"])
    wq = gu.pack_q4(nq, p["wq"], p["s"], c["K"], c["N"])
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *wq, c["N"]))
    assert gu.rel_err(y, oracle.gemm_q4(p["x"], p["wq"], p["s"], c["T"], c["K"], c["N"])) <= gu.TOL


def test_workload_decode_q4_full(nq):
    c = si.DECODE_Q4
    p = si.q4_problem(c["T"], c["K"], c["N"], c["seed"])
    wq = gu.pack_q4(nq, p["wq"], p["s"], c["K"], c["N"])
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *wq, c["N"]))
    assert gu.rel_err(y, oracle.gemm_q4(p["x"], p["wq"], p["s"], c["T"], c["K"], c["N"])) <= gu.TOL


@pytest.mark.parametrize("T", [8, 1, 2, 4])
def test_workload_verify_q5_full(nq, T):
    c = si.VERIFY_Q5
    p = si.q5_problem(T, c["K"], c["N"], c["seed"])
    wq = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], c["K"], c["N"])
    y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(p["x"]), *wq, c["N"]))
    y_ref = oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, c["K"], c["N"])
    assert gu.rel_err(y, y_ref) <= gu.TOL


def test_workload_swiglu_block_full(nq):
    """Gate/up fused with the silu epilogue, then the down projection on the GPU's own H."""
    c = si.SWIGLU_Q4
    T, K, N = c["T"], c["K"], c["N"]
    p = si.swiglu_problem(T, K, N, c["seed"])
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    h_dev = nq.swiglu_q4(gu.dev_bf16(p["x"]), *wg, *wu, N)
    rows = gu.sample_rows(N, 384, 1)
    g, u, _ = oracle.swiglu_q4_rows(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, rows)
    h_exact = (g / (1.0 + np.exp(-g)) * u).T           # [T][rows]
    h = gu.host_f64(h_dev)
    assert gu.rel_err(h[:, rows], h_exact) <= gu.TOL
    # down projection K=17408 -> N=5120 on the GPU's H (decoupled from H's rounding)
    d = si.SWIGLU_DOWN
    pd = si.q4_problem(T, d["K"], d["N"], c["seed"] + 1000)
    wd = gu.pack_q4(nq, pd["wq"], pd["s"], d["K"], d["N"])
    y = gu.host_f64(nq.gemm_q4(h_dev, *wd, d["N"]))
    h_bits = h_dev.view(torch.int16).cpu().numpy().view(np.uint16)
    y_ref = oracle.gemm_q4(h_bits, pd["wq"], pd["s"], T, d["K"], d["N"])
    assert gu.rel_err(y, y_ref) <= gu.TOL


def test_swiglu_q4_fused_decode_full_size_sampled(nq):
    """The fused gate/up call at T=1 with the decode shape (K=5120, N=17408): the call the
    layer-stack benchmark times at T=1, in its full-size launch configuration, on sampled
    rows (both halves of row tiles, both tiles of row pairs, first and last rows)."""
    T, K, N = 1, 5120, 17408
    p = si.swiglu_problem(T, K, N, 31)
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    h = gu.host_f64(nq.swiglu_q4(gu.dev_bf16(p["x"]), *wg, *wu, N))
    rows = gu.sample_rows(N, 512, 5)
    g, u, _ = oracle.swiglu_q4_rows(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, rows)
    assert gu.rel_err(h[:, rows], (g / (1.0 + np.exp(-g)) * u).T) <= gu.TOL


@pytest.mark.parametrize("layer", [0, 63])
@pytest.mark.parametrize("T", [1, 8])
def test_workload_layer_stack_sampled(nq, layer, T):
    """One layer of the 64-layer sweep: all six projections, sampled output rows."""
    x_full = si.activations(si.rng(si.layer_seed(layer, 99)), T, 17408)
    for j, (name, K, N) in enumerate(si.LAYER_Q4 + si.LAYER_Q5):
        bits = 4 if j < 3 else 5
        rows = gu.sample_rows(N, 128, j)
        x = np.ascontiguousarray(x_full[:, :K])
        if bits == 4:
            p = si.q4_problem(T, K, N, si.layer_seed(layer, j))
            wq = gu.pack_q4(nq, p["wq"], p["s"], K, N)
            y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(x), *wq, N))
            y_ref = oracle.gemm_q4_rows(x, p["wq"], p["s"], T, K, rows).T
        else:
            p = si.q5_problem(T, K, N, si.layer_seed(layer, j))
            wq = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
            y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(x), *wq, N))
            y_ref = oracle.gemm_q5_rows(x, p["wn"], p["wh"], p["s"], T, K, rows).T
        assert gu.rel_err(y[:, rows], y_ref) <= gu.TOL, name


# ---------------------------------------------------------------- properties and edges

def test_deterministic_and_zero_point_exact(nq):
    T, K, N = 8, 6208, 272       # two K slabs, split-K fix-up
    p = si.q4_problem(T, K, N, 77)
    wq = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y1 = nq.gemm_q4(x, *wq, N)
    y2 = nq.gemm_q4(x, *wq, N)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # all codes at the zero point: exactly zero output, however K is split
    z4 = gu.pack_q4(nq, np.full((N, K // 8), 0x88888888, np.uint32), p["s"], K, N)
    assert torch.count_nonzero(nq.gemm_q4(x, *z4, N).float()) == 0
    z5 = gu.pack_q5(nq, np.zeros((N, K // 8), np.uint32), np.full((N, K // 32), 0xFFFFFFFF, np.uint32),
                         p["s"], K, N)
    assert torch.count_nonzero(nq.gemm_q5(x, *z5, N).float()) == 0


def test_one_hot_x_selects_codes(nq):
    """Unit scales and a one-hot X give Y = q - z exactly (small integers are exact in bf16)."""
    K, N = 640, 48
    p = si.q4_problem(1, K, N, 78)
    s1 = np.full((N, K // 64), 0x3C00, np.uint16)
    wq = gu.pack_q4(nq, p["wq"], s1, K, N)
    codes = oracle.dequant_q4(p["wq"], s1, K, N)     # = q - 8 with unit scales
    x = np.zeros((8, K), np.uint16)
    ks = [0, 1, 63, 64, 300, 500, 638, 639]
    for t, k in enumerate(ks):
        x[t, k] = 0x3F80
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(x), *wq, N))
    for t, k in enumerate(ks):
        assert np.array_equal(y[t], codes[:, k].astype(np.float64))


def test_empty_and_k0(nq):
    N = 32
    x = torch.zeros((2, 0), dtype=torch.bfloat16, device="cuda")
    y = torch.full((2, N), 7.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    # K == 0: Y is an empty sum -> zeros
    from weight_only_groupwise_gb300.nq import _ptr, _stream, lib
    x16 = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = lib().nq_gemm_q4(_ptr(x16), _ptr(dummy), _ptr(dummy), _ptr(y), 2, 0, N, _stream(None))
    assert rc == 0
    assert torch.count_nonzero(y.float()) == 0
    # T == 0: nothing written
    y.fill_(3.0)
    rc = lib().nq_gemm_q5(_ptr(x16), _ptr(dummy), _ptr(dummy), _ptr(y), 0, 64, N, _stream(None))
    assert rc == 0 and bool((y.float() == 3.0).all())


def test_errors_leave_output_untouched(nq):
    T, K, N = 2, 128, 32
    p = si.q4_problem(T, K, N, 79)
    wq = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    x = gu.dev_bf16(p["x"])
    y = torch.full((T, N), 5.0, dtype=torch.bfloat16, device="cuda")
    from weight_only_groupwise_gb300.nq import NqError
    with pytest.raises(NqError) as e:
        nq.gemm_q4(x, *wq, N + 1, out=y)        # N % 16 != 0
    assert e.value.status == -2
    xo = torch.empty(T * K + 8, dtype=torch.bfloat16, device="cuda")[1:1 + T * K].view(T, K)
    with pytest.raises(NqError) as e:
        nq.gemm_q4(xo, *wq, N, out=y)           # misaligned X
    assert e.value.status == -3
    with pytest.raises(NqError) as e:
        nq.gemm_q4(x, *wq, N, out=x.view(-1)[:T * N].view(T, N))  # Y aliases X
    assert e.value.status == -4
    with pytest.raises(NqError) as e:                           # Y aliases the scales
        nq.gemm_q4(x, wq[0], wq[1], N, out=wq[1][:T * N * 2].view(torch.bfloat16).view(T, N))
    assert e.value.status == -4
    torch.cuda.synchronize()
    assert bool((y.float() == 5.0).all())
    nq.device_error()                               # no device-side wait ran out


@pytest.mark.parametrize("bits", [4, 5])
def test_activation_range_outliers(nq, bits):
    """Activations far outside fp16's range (outliers up to 3e38, values down to 1e-30) still
    give results within tolerance: the kernels scale each token's slab by a power of two."""
    T, K, N = 6, 1280, 96
    p = si.q4_problem(T, K, N, 91) if bits == 4 else si.q5_problem(T, K, N, 91)
    g = np.random.default_rng(92)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, 5] = 3.0e38                      # near the bf16 maximum
    x[1, :] *= 1.0e6                      # a whole token of large activations
    x[2, 100:200] = 70000.0               # just past the fp16 maximum
    x[3, :] *= 1.0e-30                    # tiny token
    x[4, 7] = -4.0e4
    xb = si.bf16_bits(x)
    if bits == 4:
        w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
        y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(xb), *w, N))
        y_ref = oracle.gemm_q4(xb, p["wq"], p["s"], T, K, N)
    else:
        w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
        y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(xb), *w, N))
        y_ref = oracle.gemm_q5(xb, p["wn"], p["wh"], p["s"], T, K, N)
    for t in range(T):   # per token: each row has its own magnitude
        assert np.all(np.isfinite(y[t]))
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


@pytest.mark.parametrize("bits", [4, 5])
def test_activation_outlier_in_a_later_slab(nq, bits):
    """T=8 with K=17408 runs in three K slabs. One token carries an outlier near the bf16
    maximum in the last slab only, in its last K group; another token is scaled by 1e30 in
    the middle slab. Each slab's range check must see its own outliers."""
    T, K, N = 8, 17408, 48
    p = si.q4_problem(T, K, N, 93) if bits == 4 else si.q5_problem(T, K, N, 93)
    g = np.random.default_rng(94)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[5, K - 3] = -2.5e38
    x[2, 7000:9000] *= 1.0e30
    xb = si.bf16_bits(x)
    if bits == 4:
        w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
        y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(xb), *w, N))
        y_ref = oracle.gemm_q4(xb, p["wq"], p["s"], T, K, N)
    else:
        w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
        y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(xb), *w, N))
        y_ref = oracle.gemm_q5(xb, p["wn"], p["wh"], p["s"], T, K, N)
    for t in range(T):
        assert np.all(np.isfinite(y[t]))
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t


SLAB_CLUSTER_SHAPES = [
    # bits, T, K, N: two, three and four K slabs, a shorter last slab, SwiGLU pairs
    (4, 8, 17408, 64), (5, 8, 17408, 48), (4, 3, 17408, 48), (5, 4, 17408, 32),
    (4, 8, 6208, 80), (4, 8, 24576, 16),
]


@pytest.mark.parametrize("bits,T,K,N", SLAB_CLUSTER_SHAPES)
def test_slab_cluster_parity(nq, bits, T, K, N):
    """The slab-cluster launch (on for this test only) against the oracle."""
    prev = nq.slab_clusters(1)
    try:
        seed = 300 + T + K // 64
        if bits == 4:
            p = si.q4_problem(T, K, N, seed)
            w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
            y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *w, N))
            y_ref = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
        else:
            p = si.q5_problem(T, K, N, seed)
            w = gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N)
            y = gu.host_f64(nq.gemm_q5(gu.dev_bf16(p["x"]), *w, N))
            y_ref = oracle.gemm_q5(p["x"], p["wn"], p["wh"], p["s"], T, K, N)
        assert gu.rel_err(y, y_ref) <= gu.TOL
        s = si.swiglu_problem(T, K, 32, seed + 1)
        wg = gu.pack_q4(nq, s["wg"], s["sg"], K, 32)
        wu = gu.pack_q4(nq, s["wu"], s["su"], K, 32)
        h = gu.host_f64(nq.swiglu_q4(gu.dev_bf16(s["x"]), *wg, *wu, 32))
        g, u, _ = oracle.swiglu_q4(s["x"], s["wg"], s["sg"], s["wu"], s["su"], T, K, 32)
        assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL
        nq.device_error()
    finally:
        nq.slab_clusters(prev)


# ---------------------------------------------------------------- larger verify batches

# T > 8 (several concurrent requests' verify rows): one launch per slice of 8 tokens; the
# ragged last slice, a single extra token and the 64-token maximum.
LARGE_T_SHAPES = [(9, 640, 48, 0), (16, 1024, 272, 1), (24, 256, 16, 2), (33, 6208, 80, 3), (64, 512, 64, 4),
                  (40, 17408, 32, 5)]


@pytest.mark.parametrize("T,K,N,seed", LARGE_T_SHAPES)
def test_large_batches_parity(nq, T, K, N, seed):
    p = si.q4_problem(T, K, N, 400 + seed)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *w, N))
    y_ref = oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)
    for t in range(T):
        assert gu.rel_err(y[t], y_ref[t]) <= gu.TOL, t
    q = si.q5_problem(T, K, N, 450 + seed)
    w5 = gu.pack_q5(nq, q["wn"], q["wh"], q["s"], K, N)
    y5 = gu.host_f64(nq.gemm_q5(gu.dev_bf16(q["x"]), *w5, N))
    assert gu.rel_err(y5, oracle.gemm_q5(q["x"], q["wn"], q["wh"], q["s"], T, K, N)) <= gu.TOL


@pytest.mark.parametrize("T", [12, 64])
def test_large_batches_swiglu(nq, T):
    K, N = 1024, 96
    p = si.swiglu_problem(T, K, N, 470 + T)
    wg = gu.pack_q4(nq, p["wg"], p["sg"], K, N)
    wu = gu.pack_q4(nq, p["wu"], p["su"], K, N)
    h = gu.host_f64(nq.swiglu_q4(gu.dev_bf16(p["x"]), *wg, *wu, N))
    g, u, _ = oracle.swiglu_q4(p["x"], p["wg"], p["sg"], p["wu"], p["su"], T, K, N)
    assert gu.rel_err(h, g / (1.0 + np.exp(-g)) * u) <= gu.TOL
    v = si.swiglu_q5_problem(T, K, N, 480 + T)
    h5 = gu.host_f64(_swiglu_q5_dev(nq, v, T, K, N))
    g5, u5, _ = oracle.swiglu_q5(v["x"], v["wgn"], v["wgh"], v["sg"], v["wun"], v["wuh"], v["su"], T, K, N)
    assert gu.rel_err(h5, g5 / (1.0 + np.exp(-g5)) * u5) <= gu.TOL


def test_large_batch_decode_shape_sampled(nq):
    """T=64 (eight requests x eight verify tokens) on the decode weight shape K=5120,
    N=17408, in its full-size launch configuration, on sampled output rows."""
    T, K, N = 64, 5120, 17408
    p = si.q4_problem(T, K, N, 490)
    w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
    y = gu.host_f64(nq.gemm_q4(gu.dev_bf16(p["x"]), *w, N))
    rows = gu.sample_rows(N, 96, 6)
    y_ref = oracle.gemm_q4_rows(p["x"], p["wq"], p["s"], T, K, rows).T
    assert gu.rel_err(y[:, rows], y_ref) <= gu.TOL


# ---------------------------------------------------------------- grouped projections

GROUPED_CASES = [
    # bits, T, K, [N per group]: the q-gate + kv pair of a layer (scaled down), odd tile counts,
    # four groups, K slabs at T=8, several 8-token slices
    (5, 8, 1024, [192, 32]), (4, 1, 640, [48, 16, 80]), (5, 3, 5120, [96, 48, 16, 272]),
    (4, 8, 17408, [64, 48]), (5, 12, 512, [32, 112]), (4, 2, 256, [16]),
    # 8 < T <= 64: one tensor-core launch per matrix (K split across blocks for the small N)
    (4, 40, 5120, [192, 48, 272]), (5, 64, 1024, [16, 144]),
]


@pytest.mark.parametrize("bits,T,K,Ns", GROUPED_CASES)
def test_grouped_projections_parity(nq, bits, T, K, Ns):
    x = si.activations(si.rng(700 + T + K), T, K)
    groups, refs = [], []
    for j, N in enumerate(Ns):
        if bits == 4:
            p = si.q4_problem(T, K, N, 710 + j)
            groups.append((*gu.pack_q4(nq, p["wq"], p["s"], K, N), N))
            refs.append(oracle.gemm_q4(x, p["wq"], p["s"], T, K, N))
        else:
            p = si.q5_problem(T, K, N, 720 + j)
            groups.append((*gu.pack_q5(nq, p["wn"], p["wh"], p["s"], K, N), N))
            refs.append(oracle.gemm_q5(x, p["wn"], p["wh"], p["s"], T, K, N))
    fn = nq.gemm_q4_grouped if bits == 4 else nq.gemm_q5_grouped
    ys = fn(gu.dev_bf16(x), groups)
    for y, r in zip(ys, refs):
        y = gu.host_f64(y)
        for t in range(T):
            assert gu.rel_err(y[t], r[t]) <= gu.TOL, t
    nq.device_error()


def test_grouped_slices_when_tensor_cores_are_off(nq):
    """With tensor-core batches off, a grouped call with T > 8 runs as 8-token slices of one
    grouped launch: the same results within the tolerance."""
    T, K, Ns = 20, 1024, [48, 112]
    x = si.activations(si.rng(790), T, K)
    groups, refs = [], []
    for j, N in enumerate(Ns):
        p = si.q4_problem(T, K, N, 791 + j)
        groups.append((*gu.pack_q4(nq, p["wq"], p["s"], K, N), N))
        refs.append(oracle.gemm_q4(x, p["wq"], p["s"], T, K, N))
    prev = nq.tensor_core_batches(0)
    try:
        ys = nq.gemm_q4_grouped(gu.dev_bf16(x), groups)
    finally:
        nq.tensor_core_batches(prev)
    for y, r in zip(ys, refs):
        y = gu.host_f64(y)
        for t in range(T):
            assert gu.rel_err(y[t], r[t]) <= gu.TOL, t
    nq.device_error()


def test_grouped_layer_qkv_full_size_sampled(nq):
    """The layer's q-gate (5120 x 6144) and kv (5120 x 1024) Q5 projections as one grouped
    launch at T=8, full size, sampled rows of both outputs."""
    T, K = 8, 5120
    x = si.activations(si.rng(730), T, K)
    pq = si.q5_problem(T, K, 6144, 731)
    pk = si.q5_problem(T, K, 1024, 732)
    groups = [(*gu.pack_q5(nq, pq["wn"], pq["wh"], pq["s"], K, 6144), 6144),
              (*gu.pack_q5(nq, pk["wn"], pk["wh"], pk["s"], K, 1024), 1024)]
    yq, yk = nq.gemm_q5_grouped(gu.dev_bf16(x), groups)
    for y, p, N, seed in ((yq, pq, 6144, 8), (yk, pk, 1024, 9)):
        rows = gu.sample_rows(N, 128, seed)
        ref = oracle.gemm_q5_rows(x, p["wn"], p["wh"], p["s"], T, K, rows).T
        assert gu.rel_err(gu.host_f64(y)[:, rows], ref) <= gu.TOL
