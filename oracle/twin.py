"""Brute-force NumPy twin of the oracle, written independently of oracle.c.

TEST INFRASTRUCTURE ONLY. Used to pin the C oracle: it unpacks the canonical layout
through byte views (NumPy's little-endian reinterpretation and ``unpackbits``) instead of
shifts on words, decodes fp16 with NumPy's own float16 type, and contracts with a BLAS
fp64 matmul. The two agreeing means neither has a dropped term, a wrong index or a
transposed operand that the other does not share.
"""
from __future__ import annotations

import numpy as np
import torch


def codes_q4(wq: np.ndarray, K: int) -> np.ndarray:
    """[N][K] int codes from uint32 [N][K/8]: byte b of a word holds k=2b (low) and 2b+1 (high)."""
    b = np.ascontiguousarray(wq, dtype="<u4").view(np.uint8).reshape(wq.shape[0], K // 2)
    q = np.empty((wq.shape[0], K), np.int64)
    q[:, 0::2] = b & 0x0F
    q[:, 1::2] = b >> 4
    return q


def codes_q5(wn: np.ndarray, wh: np.ndarray, K: int) -> np.ndarray:
    nib = codes_q4(wn, K)
    hb = np.ascontiguousarray(wh, dtype="<u4").view(np.uint8).reshape(wh.shape[0], K // 8)
    hi = np.unpackbits(hb, axis=1, bitorder="little").astype(np.int64)  # [N][K]
    return nib + 16 * hi


def scales_f32(s: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(s, dtype=np.uint16).view(np.float16).astype(np.float32)


def weights(codes: np.ndarray, s: np.ndarray, z: int) -> np.ndarray:
    """fp32 W[n][k] = s[n][k//64] * (q - z), one fp32 multiply per element."""
    sf = np.repeat(scales_f32(s), 64, axis=1)
    return sf * (codes - z).astype(np.float32)


def x_f64(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def gemm(x: np.ndarray, w32: np.ndarray) -> np.ndarray:
    """Y[T][N] = X[T][K] @ W[N][K]^T in fp64 (BLAS)."""
    return x_f64(x) @ w32.astype(np.float64).T


def gemm_q4(x, wq, s, K):
    return gemm(x, weights(codes_q4(wq, K), s, 8))


def gemm_q5(x, wn, wh, s, K):
    return gemm(x, weights(codes_q5(wn, wh, K), s, 16))


def silu(g: np.ndarray) -> np.ndarray:
    """silu via the logistic function of torch (a library routine), in fp64."""
    return np.asarray(g) * torch.sigmoid(torch.from_numpy(np.asarray(g, np.float64))).numpy()


# ---------------------------------------------------------------- NVFP4

def e4m3_f32(b: np.ndarray) -> np.ndarray:
    """e4m3 ("fn") bit patterns -> fp32 through PyTorch's float8_e4m3fn type."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def e2m1_f32(c: np.ndarray) -> np.ndarray:
    """e2m1 codes -> fp32 without a formula of our own: the fields of a 4-bit code widen into
    an e4m3 bit pattern (same sign; exponent re-biased from 1 to 7; mantissa moved to the top
    of e4m3's three bits; the one subnormal, 0.5, is the normal e4m3 2^-1), which PyTorch
    decodes."""
    c = np.asarray(c, dtype=np.uint8)
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    E = np.where(e == 0, np.where(m == 1, 6, 0), e + 6).astype(np.uint8)
    M = np.where(e == 0, 0, m << 2).astype(np.uint8)
    return e4m3_f32(((s << 7) | (E << 3) | M).astype(np.uint8))


def weights_fp4(codes: np.ndarray, sf: np.ndarray, g: float, K: int) -> np.ndarray:
    """fp32 W[n][k] = g * (scale * element); the inner product is exact in fp32."""
    elem = e2m1_f32(codes_q4(codes, K).astype(np.uint8))
    scale = np.repeat(e4m3_f32(sf), 16, axis=1)
    return np.float32(g) * (scale * elem)


def gemm_fp4(x, codes, sf, g, K):
    return gemm(x, weights_fp4(codes, sf, g, K))
