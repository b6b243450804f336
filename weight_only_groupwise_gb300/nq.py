"""Thin ctypes binding of libnq.so (include/nq.h). Argument marshalling only: every step of
the projection runs in the library's CUDA kernels. PyTorch provides device memory and the
current stream. There is no fallback: if the library is missing or the device is not a GB300
(sm_103), the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnq.so")
_lib = None

STATUS = {0: "NQ_OK", -1: "NQ_ERR_NULL", -2: "NQ_ERR_SHAPE", -3: "NQ_ERR_ALIGN", -4: "NQ_ERR_ALIAS",
          -5: "NQ_ERR_CUDA", -6: "NQ_ERR_DEVICE", -7: "NQ_ERR_TIMEOUT", -8: "NQ_ERR_SCRATCH"}


class NqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libnq.so (built by weight_only_groupwise_gb300.build). Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run weight_only_groupwise_gb300.build.build() "
                               "(the CUDA library is required; there is no CPU path)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.nq_status_string.argtypes = [I]
        L.nq_status_string.restype = ctypes.c_char_p
        L.nq_version.restype = I
        for f in ("nq_packed_bytes_q4", "nq_packed_bytes_q5"):
            getattr(L, f).argtypes = [I, I]
            getattr(L, f).restype = S
        L.nq_pack_q4.argtypes = [P, P, I, I, P, P]
        L.nq_pack_q5.argtypes = [P, P, P, I, I, P, P]
        L.nq_gemm_q4.argtypes = [P, P, P, I, I, I, P]
        L.nq_gemm_q5.argtypes = [P, P, P, I, I, I, P]
        L.nq_gemm_q4_noalloc.argtypes = [P, P, P, I, I, I, P]
        L.nq_swiglu_q4.argtypes = [P, P, P, P, I, I, I, P]
        L.nq_swiglu_q5.argtypes = [P, P, P, P, I, I, I, P]
        L.nq_dequant_q4_debug.argtypes = [P, P, I, I, P]
        L.nq_dequant_q5_debug.argtypes = [P, P, I, I, P]
        L.nq_reserve.argtypes = [I, I, I]
        L.nq_device_error.argtypes = []
        L.nq_shutdown.argtypes = []
        L.nq_shutdown.restype = None
        L.nq_plan_info.argtypes = [I, I, I, I, I, I, P]
        L.nq_plan_segments.argtypes = [I, I, I, I, I, I, I, P, ctypes.c_int64]
        L.nq_plan_segments.restype = ctypes.c_int64
        L.nq_slab_clusters.argtypes = [I]
        L.nq_slab_clusters.restype = I
        L.nq_plan_cluster_info.argtypes = [I, I, I, I, I, I, P]
        L.nq_plan_cluster_segments.argtypes = [I, I, I, I, I, I, I, P, ctypes.c_int64]
        L.nq_plan_cluster_segments.restype = ctypes.c_int64
        for f in ("nq_pack_q4", "nq_pack_q5", "nq_gemm_q4", "nq_gemm_q5", "nq_gemm_q4_noalloc", "nq_swiglu_q4",
                  "nq_swiglu_q5",
                  "nq_dequant_q4_debug", "nq_dequant_q5_debug", "nq_reserve", "nq_device_error",
                  "nq_plan_info", "nq_plan_cluster_info"):
            getattr(L, f).restype = I
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().nq_status_string(int(status)).decode()


def _check(status: int) -> None:
    if status != 0:
        raise NqError(status, status_string(status))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


# ---------------------------------------------------------------- sizes

def packed_bytes_q4(K: int, N: int) -> int:
    return int(lib().nq_packed_bytes_q4(K, N))


def packed_bytes_q5(K: int, N: int) -> int:
    return int(lib().nq_packed_bytes_q5(K, N))


# ---------------------------------------------------------------- repack

def pack_q4(wq_canon: torch.Tensor, s_canon: torch.Tensor, K: int, N: int, stream=None) -> torch.Tensor:
    """Canonical Q4 codes (4-byte words [N][K/8]) and fp16 scales ([N][K/64]) on the GPU ->
    packed weight (uint8 tensor holding codes and scales)."""
    dev = _cuda(wq_canon, "wq_canon").device
    _cuda(s_canon, "s_canon")
    w = torch.empty(max(packed_bytes_q4(K, N), 16), dtype=torch.uint8, device=dev)
    _check(lib().nq_pack_q4(_ptr(wq_canon), _ptr(s_canon), K, N, _ptr(w), _stream(stream)))
    return w


def pack_q5(wn_canon, wh_canon, s_canon, K: int, N: int, stream=None) -> torch.Tensor:
    dev = _cuda(wn_canon, "wn_canon").device
    _cuda(wh_canon, "wh_canon")
    _cuda(s_canon, "s_canon")
    w = torch.empty(max(packed_bytes_q5(K, N), 16), dtype=torch.uint8, device=dev)
    _check(lib().nq_pack_q5(_ptr(wn_canon), _ptr(wh_canon), _ptr(s_canon), K, N, _ptr(w), _stream(stream)))
    return w


# ---------------------------------------------------------------- projections

def _out(x: torch.Tensor, N: int, out):
    T = x.shape[0]
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    return _cuda(out, "out")


def gemm_q4(x: torch.Tensor, w: torch.Tensor, N: int, out=None, stream=None):
    """Y[T,N] (bf16) = X[T,K] (bf16) * dequant(packed Q4 weight)."""
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_q4(_ptr(x), _ptr(w), _ptr(y), T, K, N, _stream(stream)))
    return y


def gemm_q5(x: torch.Tensor, w: torch.Tensor, N: int, out=None, stream=None):
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_q5(_ptr(x), _ptr(w), _ptr(y), T, K, N, _stream(stream)))
    return y


def swiglu_q4(x, wg, wu, N: int, out=None, stream=None):
    """H[T,N] = bf16(silu(X*Wg) * (X*Wu)) with both weights packed Q4."""
    _cuda(x, "x")
    T, K = x.shape
    h = _out(x, N, out)
    _check(lib().nq_swiglu_q4(_ptr(x), _ptr(wg), _ptr(wu), _ptr(h), T, K, N, _stream(stream)))
    return h


def swiglu_q5(x, wg, wu, N: int, out=None, stream=None):
    """H[T,N] = bf16(silu(X*Wg) * (X*Wu)) with both weights packed Q5."""
    _cuda(x, "x")
    T, K = x.shape
    h = _out(x, N, out)
    _check(lib().nq_swiglu_q5(_ptr(x), _ptr(wg), _ptr(wu), _ptr(h), T, K, N, _stream(stream)))
    return h


def dequant_q4_debug(w, K: int, N: int, stream=None) -> torch.Tensor:
    out = torch.empty((N, K), dtype=torch.float32, device=w.device)
    _check(lib().nq_dequant_q4_debug(_ptr(w), _ptr(out), K, N, _stream(stream)))
    return out


def dequant_q5_debug(w, K: int, N: int, stream=None) -> torch.Tensor:
    out = torch.empty((N, K), dtype=torch.float32, device=w.device)
    _check(lib().nq_dequant_q5_debug(_ptr(w), _ptr(out), K, N, _stream(stream)))
    return out


# ---------------------------------------------------------------- runtime / plan

def reserve(T_max: int, K_max: int, N_max: int) -> None:
    _check(lib().nq_reserve(T_max, K_max, N_max))


def device_error() -> None:
    _check(lib().nq_device_error())


def shutdown() -> None:
    lib().nq_shutdown()


PLAN_KEYS = ("ctas", "units", "slabs", "slab_groups", "pairs", "ws_slots", "stages", "chunk_groups")


def plan_info(bits: int, mode: int, T: int, K: int, N: int, num_sms: int) -> dict:
    out = (ctypes.c_int64 * 8)()
    _check(lib().nq_plan_info(bits, mode, T, K, N, num_sms, ctypes.cast(out, ctypes.c_void_p)))
    return dict(zip(PLAN_KEYS, list(out)))


def plan_segments(bits: int, mode: int, T: int, K: int, N: int, num_sms: int, cta: int) -> list:
    n = lib().nq_plan_segments(bits, mode, T, K, N, num_sms, cta, None, 0)
    if n < 0:
        _check(int(n))
    buf = (ctypes.c_int64 * (4 * max(n, 1)))()
    lib().nq_plan_segments(bits, mode, T, K, N, num_sms, cta, ctypes.cast(buf, ctypes.c_void_p), n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def slab_clusters(enable: int = -1) -> int:
    """Turn slab clusters on (1) / off (0) for later calls, or query (-1); returns the
    previous setting."""
    return int(lib().nq_slab_clusters(enable))


CLUSTER_KEYS = ("ctas", "cluster", "slab_groups", "pairs", "ws_slots", "stages", "cluster_units", "clusters")


def plan_cluster_info(bits: int, mode: int, T: int, K: int, N: int, clusters: int) -> dict:
    """The slab-cluster plan of a shape (host only); raises NqError if the shape has none."""
    out = (ctypes.c_int64 * 8)()
    _check(lib().nq_plan_cluster_info(bits, mode, T, K, N, clusters, ctypes.cast(out, ctypes.c_void_p)))
    return dict(zip(CLUSTER_KEYS, list(out)))


def plan_cluster_segments(bits: int, mode: int, T: int, K: int, N: int, clusters: int, cta: int):
    """Real (slab, pair, ga, gb) runs of block `cta` of a slab-cluster plan, in order."""
    n = lib().nq_plan_cluster_segments(bits, mode, T, K, N, clusters, cta, None, 0)
    if n < 0:
        _check(int(n))
    buf = (ctypes.c_int64 * (4 * max(n, 1)))()
    lib().nq_plan_cluster_segments(bits, mode, T, K, N, clusters, cta, ctypes.cast(buf, ctypes.c_void_p), n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


# C names, for callers that prefer them
nq_pack_q4, nq_pack_q5 = pack_q4, pack_q5
nq_gemm_q4, nq_gemm_q5, nq_swiglu_q4 = gemm_q4, gemm_q5, swiglu_q4
nq_dequant_q4_debug, nq_dequant_q5_debug = dequant_q4_debug, dequant_q5_debug
nq_reserve, nq_device_error, nq_shutdown = reserve, device_error, shutdown
nq_plan_info, nq_plan_segments = plan_info, plan_segments
