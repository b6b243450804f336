"""Seeded synthetic inputs for the groupwise int4/int5 small-batch projection.

This module only draws random numbers and stores them in the library's canonical
input types (uint32 code words, fp16 and bf16 bit patterns). Conversions to fp16 and
bf16 are done by NumPy / PyTorch library casts. It holds none of the method's
arithmetic: no unpacking, no dequantisation, no contraction. The CPU oracle and the
CUDA path are both fed from here and from nowhere else.

Canonical layouts (the library's format definition, also stated in include/nq.h):
  X     bf16   [T][K]      row-major activations
  Wq    uint32 [N][K/8]    Q4 codes, nibble i (bits 4i..4i+3) of word j = q[n, 8j+i]
  Wn    uint32 [N][K/8]    Q5 low nibbles, same rule
  Wh    uint32 [N][K/32]   Q5 high bits, bit i of word j = bit 4 of q[n, 32j+i]
  S     fp16   [N][K/64]   one scale per (output row n, 64-wide K group)

Value distributions (the workloads of the pages' T=8 verify / decode projections):
  codes  uniform on [0, 15] (Q4) or [0, 31] (Q5). Eight independent uniform 4-bit
         fields are exactly a uniform 32-bit word, so whole words are drawn.
  scales fp16(0.01 * exp(z)), z ~ N(0, 0.25) read as variance 0.25 (sigma = 0.5)
  X      bf16(x), x ~ N(0, 1)
Draw order inside one generator: code words (nibble plane, then high plane for Q5),
then scale normals, then activation normals.
"""
from __future__ import annotations

import numpy as np
import torch

SCALE_BASE = 0.01
SCALE_SIGMA = 0.5
GROUP = 64


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, PyTorch cast) as uint16 bit patterns."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def fp16_bits(x: np.ndarray) -> np.ndarray:
    """fp64/fp32 -> fp16 (round to nearest even, NumPy cast) as uint16 bit patterns."""
    return np.asarray(x).astype(np.float16).view(np.uint16).copy()


def code_words(g: np.random.Generator, rows: int, words: int) -> np.ndarray:
    return g.integers(0, 2**32, size=(rows, words), dtype=np.uint32)


def scales(g: np.random.Generator, N: int, K: int) -> np.ndarray:
    z = g.standard_normal((N, K // GROUP))
    return fp16_bits(SCALE_BASE * np.exp(SCALE_SIGMA * z))


def activations(g: np.random.Generator, T: int, K: int) -> np.ndarray:
    return bf16_bits(g.standard_normal((T, K)).astype(np.float32))


def q4_problem(T: int, K: int, N: int, seed: int) -> dict:
    """One seeded Q4 projection: codes, then scales, then X, from one generator."""
    g = rng(seed)
    wq = code_words(g, N, K // 8)
    s = scales(g, N, K)
    x = activations(g, T, K)
    return {"bits": 4, "T": T, "K": K, "N": N, "x": x, "wq": wq, "s": s}


def q5_problem(T: int, K: int, N: int, seed: int) -> dict:
    """One seeded Q5 projection: nibble plane, high plane, scales, then X."""
    g = rng(seed)
    wn = code_words(g, N, K // 8)
    wh = code_words(g, N, K // 32)
    s = scales(g, N, K)
    x = activations(g, T, K)
    return {"bits": 5, "T": T, "K": K, "N": N, "x": x, "wn": wn, "wh": wh, "s": s}


def swiglu_problem(T: int, K: int, N: int, seed: int) -> dict:
    """Gate and up Q4 weights (each [N][K]) and X, from one generator."""
    g = rng(seed)
    wg = code_words(g, N, K // 8)
    wu = code_words(g, N, K // 8)
    sg = scales(g, N, K)
    su = scales(g, N, K)
    x = activations(g, T, K)
    return {"T": T, "K": K, "N": N, "x": x, "wg": wg, "sg": sg, "wu": wu, "su": su}


def swiglu_q5_problem(T: int, K: int, N: int, seed: int) -> dict:
    """Gate and up Q5 weights (nibble and high planes each) and X, from one generator."""
    g = rng(seed)
    wgn = code_words(g, N, K // 8)
    wgh = code_words(g, N, K // 32)
    wun = code_words(g, N, K // 8)
    wuh = code_words(g, N, K // 32)
    sg = scales(g, N, K)
    su = scales(g, N, K)
    x = activations(g, T, K)
    return {"T": T, "K": K, "N": N, "x": x, "wgn": wgn, "wgh": wgh, "sg": sg, "wun": wun,
            "wuh": wuh, "su": su}


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3 ("fn", round to nearest even, PyTorch cast) as uint8 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


FP4_BLOCK = 16
FP4_GLOBAL_SCALE = 0.0078125  # 2^-7: the per-tensor fp32 scale of the synthetic NVFP4 weights


def fp4_problem(T: int, K: int, N: int, seed: int, g: float = FP4_GLOBAL_SCALE) -> dict:
    """One seeded NVFP4 projection: e2m1 code words (uniform 32-bit words: every 4-bit code,
    both zeros included, equally likely), then one e4m3 block scale per 16 elements of a row
    (fp32 exp(N(0, 0.25)) cast to e4m3), then X ~ N(0,1) in bf16; g is the tensor scale."""
    rg = rng(seed)
    codes = code_words(rg, N, K // 8)
    sf = e4m3_bits(np.exp(SCALE_SIGMA * rg.standard_normal((N, K // FP4_BLOCK))).astype(np.float32))
    x = activations(rg, T, K)
    return {"T": T, "K": K, "N": N, "x": x, "codes": codes, "sf": sf, "g": float(g)}


FP4_UP_SCALE = 0.005859375  # 3 * 2^-9: a tensor scale for the up matrix that differs from the gate's


def swiglu_fp4_problem(T: int, K: int, N: int, seed: int, gg: float = FP4_GLOBAL_SCALE,
                       gu: float = FP4_UP_SCALE) -> dict:
    """The NVFP4 gate/up block: gate codes, up codes, gate block scales, up block scales (the
    draws of fp4_problem, twice), then X; gg, gu are the two tensor scales."""
    rg = rng(seed)
    cg = code_words(rg, N, K // 8)
    cu = code_words(rg, N, K // 8)
    sfg = e4m3_bits(np.exp(SCALE_SIGMA * rg.standard_normal((N, K // FP4_BLOCK))).astype(np.float32))
    sfu = e4m3_bits(np.exp(SCALE_SIGMA * rg.standard_normal((N, K // FP4_BLOCK))).astype(np.float32))
    x = activations(rg, T, K)
    return {"T": T, "K": K, "N": N, "x": x, "cg": cg, "sfg": sfg, "gg": float(gg), "cu": cu, "sfu": sfu,
            "gu": float(gu)}


# The five workloads. Shapes are those of a 27B-class dense decoder layer.
TINY_Q4 = dict(T=1, K=256, N=128, seed=0)                  # tiny Q4 correctness case
DECODE_Q4 = dict(T=1, K=5120, N=17408, seed=1)             # decode GEMV, FFN up-projection
VERIFY_Q5 = dict(T=8, K=5120, N=6144, seed=2)              # T=8 verify, attention gate/value
SWIGLU_Q4 = dict(T=8, K=5120, N=17408, seed=3)             # gate+up, then down K=17408,N=5120
SWIGLU_DOWN = dict(K=17408, N=5120)
LAYER_Q4 = [("gate", 5120, 17408), ("up", 5120, 17408), ("down", 17408, 5120)]
LAYER_Q5 = [("qgate", 5120, 6144), ("kv", 5120, 1024), ("out", 6144, 5120)]
N_LAYERS = 64


def layer_seed(layer: int, proj: int) -> int:
    """Per-layer, per-projection seed of the layer-stack sweep."""
    return 1000 * layer + proj


# ---------------------------------------------------------------- device-side generators
# Same recipe, drawn on the GPU with a seeded torch generator: used where the volume makes
# host generation slow (the benchmark's rotated weight copies and the 64-layer stack).
# Parity tests use the host generators above.

def device_code_words(rows: int, words: int, gen: "torch.Generator", device) -> "torch.Tensor":
    return torch.randint(-2**31, 2**31, (rows, words), dtype=torch.int64, generator=gen,
                         device=device).to(torch.int32)


def device_scales(N: int, K: int, gen, device) -> "torch.Tensor":
    z = torch.randn((N, K // GROUP), generator=gen, device=device, dtype=torch.float32)
    return (SCALE_BASE * torch.exp(SCALE_SIGMA * z)).to(torch.float16).view(torch.int16)


def device_fp4_scales(N: int, K: int, gen, device) -> "torch.Tensor":
    z = torch.randn((N, K // FP4_BLOCK), generator=gen, device=device, dtype=torch.float32)
    return torch.exp(SCALE_SIGMA * z).to(torch.float8_e4m3fn).view(torch.uint8)


def device_activations(T: int, K: int, gen, device) -> "torch.Tensor":
    return torch.randn((T, K), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
