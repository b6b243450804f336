"""CPU oracle for the weight-only groupwise int4/int5 projection.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers. The product path never imports this package.

``oracle.c`` is the definition written out in fp64 on the canonical layout (see its header).
``twin.py`` is a second, independently written NumPy evaluation used to pin the C oracle.
This module only compiles ``oracle.c`` and marshals NumPy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP) into oracle/liborc.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L.orc_fp16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_fp16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_round_bf16.restype = ctypes.c_uint16
        L.orc_silu_mul.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_silu_mul.restype = ctypes.c_double
        L.orc_dequant_q4.argtypes = [P, P, I, I, P]
        L.orc_dequant_q5.argtypes = [P, P, P, I, I, P]
        L.orc_gemm_q4.argtypes = [P, P, P, I, I, I, P]
        L.orc_gemm_q5.argtypes = [P, P, P, P, I, I, I, P]
        L.orc_gemm_q4_rows.argtypes = [P, P, P, I, I, P, I, P]
        L.orc_gemm_q5_rows.argtypes = [P, P, P, P, I, I, P, I, P]
        L.orc_swiglu_q4.argtypes = [P, P, P, P, P, I, I, I, P, P, P]
        L.orc_swiglu_q4_rows.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P]
        L.orc_swiglu_q5.argtypes = [P, P, P, P, P, P, P, I, I, I, P, P, P]
        L.orc_swiglu_q5_rows.argtypes = [P, P, P, P, P, P, P, I, I, P, I, P, P, P]
        L.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_to_f64.restype = ctypes.c_double
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_f64.restype = ctypes.c_double
        L.orc_dequant_fp4.argtypes = [P, P, ctypes.c_float, I, I, P]
        L.orc_gemm_fp4.argtypes = [P, P, P, ctypes.c_float, I, I, I, P]
        L.orc_gemm_fp4_rows.argtypes = [P, P, P, ctypes.c_float, I, I, P, I, P]
        F = ctypes.c_float
        L.orc_swiglu_fp4.argtypes = [P, P, P, F, P, P, F, I, I, I, P, P, P]
        L.orc_swiglu_fp4_rows.argtypes = [P, P, P, F, P, P, F, I, I, P, I, P, P, P]
        L.orc_num_threads.restype = I
        L.orc_set_num_threads.argtypes = [I]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def fp16_to_f64(h: int) -> float:
    return lib().orc_fp16_to_f64(int(h))


def bf16_to_f64(b: int) -> float:
    return lib().orc_bf16_to_f64(int(b))


def round_bf16(v: float) -> int:
    return int(lib().orc_round_bf16(float(v)))


def silu_mul(g: float, u: float) -> float:
    return lib().orc_silu_mul(float(g), float(u))


def dequant_q4(wq, s, K: int, N: int) -> np.ndarray:
    wq, s = _c(wq, np.uint32), _c(s, np.uint16)
    w = np.empty((N, K), np.float32)
    lib().orc_dequant_q4(_p(wq), _p(s), K, N, _p(w))
    return w


def dequant_q5(wn, wh, s, K: int, N: int) -> np.ndarray:
    wn, wh, s = _c(wn, np.uint32), _c(wh, np.uint32), _c(s, np.uint16)
    w = np.empty((N, K), np.float32)
    lib().orc_dequant_q5(_p(wn), _p(wh), _p(s), K, N, _p(w))
    return w


def gemm_q4(x, wq, s, T: int, K: int, N: int) -> np.ndarray:
    x, wq, s = _c(x, np.uint16), _c(wq, np.uint32), _c(s, np.uint16)
    y = np.empty((T, N), np.float64)
    lib().orc_gemm_q4(_p(x), _p(wq), _p(s), T, K, N, _p(y))
    return y


def gemm_q5(x, wn, wh, s, T: int, K: int, N: int) -> np.ndarray:
    x, wn, wh, s = _c(x, np.uint16), _c(wn, np.uint32), _c(wh, np.uint32), _c(s, np.uint16)
    y = np.empty((T, N), np.float64)
    lib().orc_gemm_q5(_p(x), _p(wn), _p(wh), _p(s), T, K, N, _p(y))
    return y


def gemm_q4_rows(x, wq, s, T: int, K: int, rows) -> np.ndarray:
    """Y[t, rows[i]] as an array [len(rows)][T]."""
    x, wq, s = _c(x, np.uint16), _c(wq, np.uint32), _c(s, np.uint16)
    r = _c(rows, np.int32)
    y = np.empty((len(r), T), np.float64)
    lib().orc_gemm_q4_rows(_p(x), _p(wq), _p(s), T, K, _p(r), len(r), _p(y))
    return y


def gemm_q5_rows(x, wn, wh, s, T: int, K: int, rows) -> np.ndarray:
    x, wn, wh, s = _c(x, np.uint16), _c(wn, np.uint32), _c(wh, np.uint32), _c(s, np.uint16)
    r = _c(rows, np.int32)
    y = np.empty((len(r), T), np.float64)
    lib().orc_gemm_q5_rows(_p(x), _p(wn), _p(wh), _p(s), T, K, _p(r), len(r), _p(y))
    return y


def swiglu_q4(x, wg, sg, wu, su, T: int, K: int, N: int):
    """(G fp64 [T][N], U fp64 [T][N], H bf16 bits [T][N])."""
    x = _c(x, np.uint16)
    wg, wu = _c(wg, np.uint32), _c(wu, np.uint32)
    sg, su = _c(sg, np.uint16), _c(su, np.uint16)
    g = np.empty((T, N), np.float64)
    u = np.empty((T, N), np.float64)
    h = np.empty((T, N), np.uint16)
    lib().orc_swiglu_q4(_p(x), _p(wg), _p(sg), _p(wu), _p(su), T, K, N, _p(g), _p(u), _p(h))
    return g, u, h


def swiglu_q4_rows(x, wg, sg, wu, su, T: int, K: int, rows):
    """(G, U, H) on selected rows, each [len(rows)][T]."""
    x = _c(x, np.uint16)
    wg, wu = _c(wg, np.uint32), _c(wu, np.uint32)
    sg, su = _c(sg, np.uint16), _c(su, np.uint16)
    r = _c(rows, np.int32)
    g = np.empty((len(r), T), np.float64)
    u = np.empty((len(r), T), np.float64)
    h = np.empty((len(r), T), np.uint16)
    lib().orc_swiglu_q4_rows(_p(x), _p(wg), _p(sg), _p(wu), _p(su), T, K, _p(r), len(r),
                             _p(g), _p(u), _p(h))
    return g, u, h


def swiglu_q5(x, wgn, wgh, sg, wun, wuh, su, T: int, K: int, N: int):
    """(G, U, H) for 5-bit gate and up weights, as swiglu_q4."""
    x = _c(x, np.uint16)
    wgn, wgh, wun, wuh = (_c(a, np.uint32) for a in (wgn, wgh, wun, wuh))
    sg, su = _c(sg, np.uint16), _c(su, np.uint16)
    g = np.empty((T, N), np.float64)
    u = np.empty((T, N), np.float64)
    h = np.empty((T, N), np.uint16)
    lib().orc_swiglu_q5(_p(x), _p(wgn), _p(wgh), _p(sg), _p(wun), _p(wuh), _p(su), T, K, N,
                        _p(g), _p(u), _p(h))
    return g, u, h


def swiglu_q5_rows(x, wgn, wgh, sg, wun, wuh, su, T: int, K: int, rows):
    """(G, U, H) on selected rows, each [len(rows)][T]."""
    x = _c(x, np.uint16)
    wgn, wgh, wun, wuh = (_c(a, np.uint32) for a in (wgn, wgh, wun, wuh))
    sg, su = _c(sg, np.uint16), _c(su, np.uint16)
    r = _c(rows, np.int32)
    g = np.empty((len(r), T), np.float64)
    u = np.empty((len(r), T), np.float64)
    h = np.empty((len(r), T), np.uint16)
    lib().orc_swiglu_q5_rows(_p(x), _p(wgn), _p(wgh), _p(sg), _p(wun), _p(wuh), _p(su), T, K,
                             _p(r), len(r), _p(g), _p(u), _p(h))
    return g, u, h


def e2m1_to_f64(c: int) -> float:
    return lib().orc_e2m1_to_f64(int(c))


def e4m3_to_f64(b: int) -> float:
    return lib().orc_e4m3_to_f64(int(b))


def dequant_fp4(codes, sf, g: float, K: int, N: int) -> np.ndarray:
    """NVFP4 weights in fp32 [N][K]: codes uint32 [N][K/8], e4m3 scales uint8 [N][K/16]."""
    codes, sf = _c(codes, np.uint32), _c(sf, np.uint8)
    w = np.empty((N, K), np.float32)
    lib().orc_dequant_fp4(_p(codes), _p(sf), float(g), K, N, _p(w))
    return w


def gemm_fp4(x, codes, sf, g: float, T: int, K: int, N: int) -> np.ndarray:
    x, codes, sf = _c(x, np.uint16), _c(codes, np.uint32), _c(sf, np.uint8)
    y = np.empty((T, N), np.float64)
    lib().orc_gemm_fp4(_p(x), _p(codes), _p(sf), float(g), T, K, N, _p(y))
    return y


def gemm_fp4_rows(x, codes, sf, g: float, T: int, K: int, rows) -> np.ndarray:
    """Y[t, rows[i]] as an array [len(rows)][T]."""
    x, codes, sf = _c(x, np.uint16), _c(codes, np.uint32), _c(sf, np.uint8)
    r = _c(rows, np.int32)
    y = np.empty((len(r), T), np.float64)
    lib().orc_gemm_fp4_rows(_p(x), _p(codes), _p(sf), float(g), T, K, _p(r), len(r), _p(y))
    return y


def swiglu_fp4(x, cg, sfg, gg: float, cu, sfu, gu: float, T: int, K: int, N: int):
    """NVFP4 gate/up block: (G fp64 [T][N], U fp64 [T][N], H bf16 bits [T][N])."""
    x = _c(x, np.uint16)
    cg, cu = _c(cg, np.uint32), _c(cu, np.uint32)
    sfg, sfu = _c(sfg, np.uint8), _c(sfu, np.uint8)
    g = np.empty((T, N), np.float64)
    u = np.empty((T, N), np.float64)
    h = np.empty((T, N), np.uint16)
    lib().orc_swiglu_fp4(_p(x), _p(cg), _p(sfg), float(gg), _p(cu), _p(sfu), float(gu), T, K, N, _p(g), _p(u), _p(h))
    return g, u, h


def swiglu_fp4_rows(x, cg, sfg, gg: float, cu, sfu, gu: float, T: int, K: int, rows):
    """(G, U, H) of the NVFP4 block on selected rows, each [len(rows)][T]."""
    x = _c(x, np.uint16)
    cg, cu = _c(cg, np.uint32), _c(cu, np.uint32)
    sfg, sfu = _c(sfg, np.uint8), _c(sfu, np.uint8)
    r = _c(rows, np.int32)
    g = np.empty((len(r), T), np.float64)
    u = np.empty((len(r), T), np.float64)
    h = np.empty((len(r), T), np.uint16)
    lib().orc_swiglu_fp4_rows(_p(x), _p(cg), _p(sfg), float(gg), _p(cu), _p(sfu), float(gu), T, K, _p(r), len(r),
                              _p(g), _p(u), _p(h))
    return g, u, h


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))
