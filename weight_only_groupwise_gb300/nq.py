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


class NqGroup(ctypes.Structure):
    """struct nq_group of include/nq.h."""
    _fields_ = [("Wq", ctypes.c_void_p), ("S", ctypes.c_void_p), ("Y", ctypes.c_void_p), ("N", ctypes.c_int)]


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
        L.nq_scale_bytes.argtypes = [I, I]
        L.nq_scale_bytes.restype = S
        L.nq_pack_q4.argtypes = [P, P, I, I, P, P, P]
        L.nq_pack_q5.argtypes = [P, P, P, I, I, P, P, P]
        L.nq_gemm_q4.argtypes = [P, P, P, P, I, I, I, P]
        L.nq_gemm_q5.argtypes = [P, P, P, P, I, I, I, P]
        L.nq_gemm_q4_noalloc.argtypes = [P, P, P, P, I, I, I, P]
        L.nq_swiglu_q4.argtypes = [P, P, P, P, P, P, I, I, I, P]
        L.nq_swiglu_q5.argtypes = [P, P, P, P, P, P, I, I, I, P]
        for f in ("nq_dequant_q4_debug", "nq_dequant_q5_debug", "nq_dequant_q4_debug_bf16",
                  "nq_dequant_q5_debug_bf16"):
            getattr(L, f).argtypes = [P, P, P, I, I, P]
            getattr(L, f).restype = I
        L.nq_packed_bytes_fp4.argtypes = [I, I]
        L.nq_packed_bytes_fp4.restype = S
        L.nq_scale_bytes_fp4.argtypes = [I, I]
        L.nq_scale_bytes_fp4.restype = S
        L.nq_pack_fp4.argtypes = [P, P, I, I, P, P, P]
        L.nq_pack_fp4.restype = I
        L.nq_gemm_fp4.argtypes = [P, P, P, ctypes.c_float, P, I, I, I, P]
        L.nq_gemm_fp4.restype = I
        L.nq_swiglu_fp4.argtypes = [P, P, P, ctypes.c_float, P, P, ctypes.c_float, P, I, I, I, P]
        L.nq_swiglu_fp4.restype = I
        L.nq_dequant_fp4_debug.argtypes = [P, P, ctypes.c_float, P, I, I, P]
        L.nq_dequant_fp4_debug.restype = I
        for f in ("nq_gemm_q4_grouped", "nq_gemm_q5_grouped"):
            getattr(L, f).argtypes = [P, P, I, I, I, P]
            getattr(L, f).restype = I
        L.nq_reserve.argtypes = [I, I, I]
        L.nq_device_error.argtypes = []
        L.nq_wait_limit.argtypes = [ctypes.c_longlong]
        L.nq_wait_limit.restype = ctypes.c_longlong
        L.nq_shutdown.argtypes = []
        L.nq_shutdown.restype = None
        L.nq_plan_info.argtypes = [I, I, I, I, I, I, P]
        L.nq_plan_segments.argtypes = [I, I, I, I, I, I, I, P, ctypes.c_int64]
        L.nq_plan_segments.restype = ctypes.c_int64
        L.nq_tensor_core_batches.argtypes = [I]
        L.nq_tensor_core_batches.restype = I
        L.nq_plan_tc_info.argtypes = [I, I, I, I, I, P]
        L.nq_plan_tc_info.restype = I
        L.nq_route_info.argtypes = [I, I, I, I, I, I, P]
        L.nq_route_info.restype = I
        L.nq_slab_clusters.argtypes = [I]
        L.nq_slab_clusters.restype = I
        L.nq_plan_cluster_info.argtypes = [I, I, I, I, I, I, P]
        L.nq_plan_cluster_segments.argtypes = [I, I, I, I, I, I, I, P, ctypes.c_int64]
        L.nq_plan_cluster_segments.restype = ctypes.c_int64
        L.nq_program_create.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        L.nq_program_gemm.argtypes = [P, I, P, P, P, P, I, I, I]
        L.nq_program_gemm_fp4.argtypes = [P, P, P, P, ctypes.c_float, P, I, I, I]
        L.nq_program_swiglu.argtypes = [P, I, P, P, P, P, P, P, I, I, I]
        L.nq_program_grouped.argtypes = [P, I, P, P, I, I, I]
        L.nq_program_swiglu_fp4.argtypes = [P, P, P, P, ctypes.c_float, P, P, ctypes.c_float, P, I, I, I]
        L.nq_program_build.argtypes = [P]
        L.nq_program_launch.argtypes = [P, P]
        L.nq_program_info.argtypes = [P, P]
        for f in ("nq_program_create", "nq_program_gemm", "nq_program_gemm_fp4", "nq_program_swiglu", "nq_program_swiglu_fp4",
                  "nq_program_grouped", "nq_program_build", "nq_program_launch", "nq_program_info"):
            getattr(L, f).restype = I
        L.nq_program_destroy.argtypes = [P]
        L.nq_program_destroy.restype = None
        for f in ("nq_pack_q4", "nq_pack_q5", "nq_gemm_q4", "nq_gemm_q5", "nq_gemm_q4_noalloc", "nq_swiglu_q4",
                  "nq_swiglu_q5", "nq_reserve", "nq_device_error", "nq_plan_info", "nq_plan_cluster_info"):
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


def scale_bytes(K: int, N: int) -> int:
    return int(lib().nq_scale_bytes(K, N))


# ---------------------------------------------------------------- repack

def _packed_pair(code_bytes: int, K: int, N: int, dev):
    wq = torch.empty(max(code_bytes, 16), dtype=torch.uint8, device=dev)
    s = torch.empty(max(scale_bytes(K, N), 16), dtype=torch.uint8, device=dev)
    return wq, s


def pack_q4(wq_canon: torch.Tensor, s_canon: torch.Tensor, K: int, N: int, stream=None):
    """Canonical Q4 codes (4-byte words [N][K/8]) and fp16 scales ([N][K/64]) on the GPU ->
    (packed codes, packed scales), two uint8 device tensors."""
    dev = _cuda(wq_canon, "wq_canon").device
    _cuda(s_canon, "s_canon")
    wq, s = _packed_pair(packed_bytes_q4(K, N), K, N, dev)
    _check(lib().nq_pack_q4(_ptr(wq_canon), _ptr(s_canon), K, N, _ptr(wq), _ptr(s), _stream(stream)))
    return wq, s


def pack_q5(wn_canon, wh_canon, s_canon, K: int, N: int, stream=None):
    """Canonical Q5 nibble plane, high plane and fp16 scales -> (packed codes, packed scales)."""
    dev = _cuda(wn_canon, "wn_canon").device
    _cuda(wh_canon, "wh_canon")
    _cuda(s_canon, "s_canon")
    wq, s = _packed_pair(packed_bytes_q5(K, N), K, N, dev)
    _check(lib().nq_pack_q5(_ptr(wn_canon), _ptr(wh_canon), _ptr(s_canon), K, N, _ptr(wq), _ptr(s),
                            _stream(stream)))
    return wq, s


# ---------------------------------------------------------------- projections

def _out(x: torch.Tensor, N: int, out):
    T = x.shape[0]
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    return _cuda(out, "out")


def gemm_q4(x: torch.Tensor, wq: torch.Tensor, s: torch.Tensor, N: int, out=None, stream=None):
    """Y[T,N] (bf16) = X[T,K] (bf16) * dequant(packed Q4 codes wq, packed scales s)."""
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_q4(_ptr(x), _ptr(wq), _ptr(s), _ptr(y), T, K, N, _stream(stream)))
    return y


def gemm_q5(x: torch.Tensor, wq: torch.Tensor, s: torch.Tensor, N: int, out=None, stream=None):
    """Y[T,N] (bf16) = X[T,K] (bf16) * dequant(packed Q5 codes wq, packed scales s)."""
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_q5(_ptr(x), _ptr(wq), _ptr(s), _ptr(y), T, K, N, _stream(stream)))
    return y


def gemm_q4_noalloc(x: torch.Tensor, wq: torch.Tensor, s: torch.Tensor, N: int, out=None, stream=None):
    """gemm_q4 with its scratch in the library's fixed device array (no allocation by the
    library; `out` is allocated here by torch when not given)."""
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_q4_noalloc(_ptr(x), _ptr(wq), _ptr(s), _ptr(y), T, K, N, _stream(stream)))
    return y


def _grouped(fn, x, groups, outs, stream):
    _cuda(x, "x")
    T, K = x.shape
    if outs is None:
        outs = [torch.empty((T, N), dtype=torch.bfloat16, device=x.device) for (_, _, N) in groups]
    arr = (NqGroup * len(groups))()
    for i, ((wq, s, N), y) in enumerate(zip(groups, outs)):
        _cuda(y, "out")
        arr[i] = NqGroup(wq.data_ptr(), s.data_ptr(), y.data_ptr(), N)
    _check(fn(_ptr(x), ctypes.cast(arr, ctypes.c_void_p), len(groups), T, K, _stream(stream)))
    return outs


def gemm_q4_grouped(x, groups, outs=None, stream=None):
    """[Y_g] for groups [(packed codes, packed scales, N_g), ...] sharing X, one launch."""
    return _grouped(lib().nq_gemm_q4_grouped, x, groups, outs, stream)


def gemm_q5_grouped(x, groups, outs=None, stream=None):
    return _grouped(lib().nq_gemm_q5_grouped, x, groups, outs, stream)


def swiglu_q4(x, wg, sg, wu, su, N: int, out=None, stream=None):
    """H[T,N] = bf16(silu(X*Wg) * (X*Wu)) with both weights packed Q4 (codes, scales)."""
    _cuda(x, "x")
    T, K = x.shape
    h = _out(x, N, out)
    _check(lib().nq_swiglu_q4(_ptr(x), _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(h), T, K, N,
                              _stream(stream)))
    return h


def swiglu_q5(x, wg, sg, wu, su, N: int, out=None, stream=None):
    """H[T,N] = bf16(silu(X*Wg) * (X*Wu)) with both weights packed Q5 (codes, scales)."""
    _cuda(x, "x")
    T, K = x.shape
    h = _out(x, N, out)
    _check(lib().nq_swiglu_q5(_ptr(x), _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(h), T, K, N,
                              _stream(stream)))
    return h


def _dequant(fn, wq, s, K: int, N: int, stream):
    out = torch.empty((N, K), dtype=torch.float32, device=wq.device)
    _check(fn(_ptr(wq), _ptr(s), _ptr(out), K, N, _stream(stream)))
    return out


def dequant_q4_debug(wq, s, K: int, N: int, operands: str = "f16", stream=None) -> torch.Tensor:
    """fp32 [N][K] dump of a packed Q4 pair through the decoder of the fp16-operand kernels
    (T <= 2, operands="f16") or of the bf16-operand kernels (T >= 3, operands="bf16")."""
    f = lib().nq_dequant_q4_debug if operands == "f16" else lib().nq_dequant_q4_debug_bf16
    return _dequant(f, wq, s, K, N, stream)


def dequant_q5_debug(wq, s, K: int, N: int, operands: str = "f16", stream=None) -> torch.Tensor:
    f = lib().nq_dequant_q5_debug if operands == "f16" else lib().nq_dequant_q5_debug_bf16
    return _dequant(f, wq, s, K, N, stream)


# ---------------------------------------------------------------- NVFP4

def packed_bytes_fp4(K: int, N: int) -> int:
    return int(lib().nq_packed_bytes_fp4(K, N))


def scale_bytes_fp4(K: int, N: int) -> int:
    return int(lib().nq_scale_bytes_fp4(K, N))


def pack_fp4(codes_canon: torch.Tensor, sf_canon: torch.Tensor, K: int, N: int, stream=None):
    """Canonical NVFP4 codes (4-byte words [N][K/8]) and e4m3 scales (bytes [N][K/16]) on the
    GPU -> (packed codes, packed scales), two uint8 device tensors."""
    dev = _cuda(codes_canon, "codes_canon").device
    _cuda(sf_canon, "sf_canon")
    wq = torch.empty(max(packed_bytes_fp4(K, N), 16), dtype=torch.uint8, device=dev)
    s = torch.empty(max(scale_bytes_fp4(K, N), 16), dtype=torch.uint8, device=dev)
    _check(lib().nq_pack_fp4(_ptr(codes_canon), _ptr(sf_canon), K, N, _ptr(wq), _ptr(s), _stream(stream)))
    return wq, s


def gemm_fp4(x: torch.Tensor, wq: torch.Tensor, s: torch.Tensor, global_scale: float, N: int, out=None,
             stream=None):
    """Y[T,N] (bf16) = X[T,K] (bf16) * NVFP4 weight (packed codes wq, packed scales s, tensor
    scale global_scale)."""
    _cuda(x, "x")
    T, K = x.shape
    y = _out(x, N, out)
    _check(lib().nq_gemm_fp4(_ptr(x), _ptr(wq), _ptr(s), ctypes.c_float(global_scale), _ptr(y), T, K, N,
                             _stream(stream)))
    return y


def swiglu_fp4(x, wg, sg, gate_scale: float, wu, su, up_scale: float, N: int, out=None, stream=None):
    """H[T,N] = bf16(silu(X*Wg) * (X*Wu)) with NVFP4 gate and up weights (packed codes, packed
    scales, tensor scale each)."""
    _cuda(x, "x")
    T, K = x.shape
    h = _out(x, N, out)
    _check(lib().nq_swiglu_fp4(_ptr(x), _ptr(wg), _ptr(sg), ctypes.c_float(gate_scale), _ptr(wu), _ptr(su),
                               ctypes.c_float(up_scale), _ptr(h), T, K, N, _stream(stream)))
    return h


def dequant_fp4_debug(wq, s, global_scale: float, K: int, N: int, stream=None) -> torch.Tensor:
    out = torch.empty((N, K), dtype=torch.float32, device=wq.device)
    _check(lib().nq_dequant_fp4_debug(_ptr(wq), _ptr(s), ctypes.c_float(global_scale), _ptr(out), K, N,
                                      _stream(stream)))
    return out


# ---------------------------------------------------------------- recorded programs

PROGRAM_KEYS = ("calls", "kernels", "builds", "failed_call")


class Program:
    """A sequence of projection calls recorded once and replayed as one CUDA graph
    (nq_program_* of include/nq.h). The library records the tensors' device addresses, not
    their contents: write new activations into the same X tensor and launch again. The
    program keeps a reference to every tensor it records, so they stay allocated while it can
    be launched. Outputs not given are allocated here (torch) and returned."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(lib().nq_program_create(ctypes.byref(h)))
        self._h = h
        self._keep = []

    def _rec(self, status, *tensors):
        _check(status)
        self._keep.extend(t for t in tensors if t is not None)

    def _gemm(self, bits, x, wq, s, N, out):
        _cuda(x, "x")
        T, K = x.shape
        y = _out(x, N, out)
        self._rec(lib().nq_program_gemm(self._h, bits, _ptr(x), _ptr(wq), _ptr(s), _ptr(y), T, K, N), x, wq, s, y)
        return y

    def gemm_q4(self, x, wq, s, N: int, out=None):
        return self._gemm(4, x, wq, s, N, out)

    def gemm_q5(self, x, wq, s, N: int, out=None):
        return self._gemm(5, x, wq, s, N, out)

    def gemm_fp4(self, x, wq, s, global_scale: float, N: int, out=None):
        _cuda(x, "x")
        T, K = x.shape
        y = _out(x, N, out)
        self._rec(lib().nq_program_gemm_fp4(self._h, _ptr(x), _ptr(wq), _ptr(s), ctypes.c_float(global_scale),
                                            _ptr(y), T, K, N), x, wq, s, y)
        return y

    def _swiglu(self, bits, x, wg, sg, wu, su, N, out):
        _cuda(x, "x")
        T, K = x.shape
        h = _out(x, N, out)
        self._rec(lib().nq_program_swiglu(self._h, bits, _ptr(x), _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(h),
                                          T, K, N), x, wg, sg, wu, su, h)
        return h

    def swiglu_q4(self, x, wg, sg, wu, su, N: int, out=None):
        return self._swiglu(4, x, wg, sg, wu, su, N, out)

    def swiglu_q5(self, x, wg, sg, wu, su, N: int, out=None):
        return self._swiglu(5, x, wg, sg, wu, su, N, out)

    def swiglu_fp4(self, x, wg, sg, gate_scale: float, wu, su, up_scale: float, N: int, out=None):
        _cuda(x, "x")
        T, K = x.shape
        h = _out(x, N, out)
        self._rec(lib().nq_program_swiglu_fp4(self._h, _ptr(x), _ptr(wg), _ptr(sg), ctypes.c_float(gate_scale),
                                              _ptr(wu), _ptr(su), ctypes.c_float(up_scale), _ptr(h), T, K, N),
                  x, wg, sg, wu, su, h)
        return h

    def _grouped(self, bits, x, groups, outs):
        _cuda(x, "x")
        T, K = x.shape
        if outs is None:
            outs = [torch.empty((T, N), dtype=torch.bfloat16, device=x.device) for (_, _, N) in groups]
        arr = (NqGroup * len(groups))()
        for i, ((wq, s, N), y) in enumerate(zip(groups, outs)):
            _cuda(y, "out")
            arr[i] = NqGroup(wq.data_ptr(), s.data_ptr(), y.data_ptr(), N)
        self._rec(lib().nq_program_grouped(self._h, bits, _ptr(x), ctypes.cast(arr, ctypes.c_void_p), len(groups),
                                           T, K), x, *[t for (wq, s, _) in groups for t in (wq, s)], *outs)
        return outs

    def grouped_q4(self, x, groups, outs=None):
        return self._grouped(4, x, groups, outs)

    def grouped_q5(self, x, groups, outs=None):
        return self._grouped(5, x, groups, outs)

    def build(self) -> None:
        _check(lib().nq_program_build(self._h))

    def launch(self, stream=None) -> None:
        _check(lib().nq_program_launch(self._h, _stream(stream)))

    def info(self) -> dict:
        out = (ctypes.c_int64 * 4)()
        _check(lib().nq_program_info(self._h, ctypes.cast(out, ctypes.c_void_p)))
        return dict(zip(PROGRAM_KEYS, list(out)))

    def close(self) -> None:
        if self._h is not None and self._h.value:
            lib().nq_program_destroy(self._h)
        self._h = None
        self._keep = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- runtime / plan

def reserve(T_max: int, K_max: int, N_max: int) -> None:
    _check(lib().nq_reserve(T_max, K_max, N_max))


def device_error() -> None:
    _check(lib().nq_device_error())


def wait_limit(ns: int = 0) -> int:
    """Set (ns > 0) or query (ns <= 0) the bound of device-side waits; returns the previous."""
    return int(lib().nq_wait_limit(int(ns)))


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


def tensor_core_batches(enable: int = -1) -> int:
    """Large batches (8 < T <= 64) on the tensor-core kernel (1) or in 8-token slices (0); -1
    queries. Returns the previous setting."""
    return int(lib().nq_tensor_core_batches(enable))


TC_KEYS = ("ctas", "row_blocks", "k_pieces", "tokens_padded", "stages", "smem_bytes", "groups", "stage_groups")


def plan_tc_info(bits: int, T: int, K: int, N: int, num_sms: int) -> dict:
    out = (ctypes.c_int64 * 8)()
    _check(lib().nq_plan_tc_info(bits, T, K, N, num_sms, ctypes.cast(out, ctypes.c_void_p)))
    return dict(zip(TC_KEYS, list(out)))


ROUTE_KEYS = ("kernel", "launches", "operands", "split", "ctas", "k_split", "stages", "tokens_padded")
ROUTE_NAMES = {"kernel": ("mma.sync 8-token", "tcgen05"), "operands": ("fp16", "bf16"),
               "split": ("stream-K", "whole row pairs", "slab clusters", "row blocks x K pieces")}


def route_info(bits: int, mode: int, T: int, K: int, N: int, num_sms: int) -> dict:
    """The kernel and variant a call of this shape takes with the current settings (host
    only): ROUTE_KEYS, with the kernel, operand type and split also given by name."""
    out = (ctypes.c_int64 * 8)()
    _check(lib().nq_route_info(bits, mode, T, K, N, num_sms, ctypes.cast(out, ctypes.c_void_p)))
    d = dict(zip(ROUTE_KEYS, list(out)))
    for k, names in ROUTE_NAMES.items():
        d[k + "_name"] = names[d[k]]
    return d


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
nq_gemm_q4, nq_gemm_q5, nq_gemm_q4_noalloc = gemm_q4, gemm_q5, gemm_q4_noalloc
nq_swiglu_q4, nq_swiglu_q5 = swiglu_q4, swiglu_q5
nq_gemm_q4_grouped, nq_gemm_q5_grouped = gemm_q4_grouped, gemm_q5_grouped
nq_dequant_q4_debug, nq_dequant_q5_debug = dequant_q4_debug, dequant_q5_debug
nq_pack_fp4, nq_gemm_fp4, nq_dequant_fp4_debug = pack_fp4, gemm_fp4, dequant_fp4_debug
nq_swiglu_fp4 = swiglu_fp4
nq_reserve, nq_device_error, nq_shutdown, nq_wait_limit = reserve, device_error, shutdown, wait_limit
nq_plan_info, nq_plan_segments = plan_info, plan_segments
