"""The C ABI library loads and exports every function include/nq.h declares, and its
host-only calls (sizes, status strings, argument checks that fail before any CUDA call,
plan inspection) behave as documented. No GPU compute here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from weight_only_groupwise_gb300 import build
    build.build()
    from weight_only_groupwise_gb300 import nq
    return nq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(nq_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("nq_pack_q4", "nq_pack_q5", "nq_gemm_q4", "nq_gemm_q5", "nq_swiglu_q4",
                 "nq_swiglu_q5", "nq_dequant_q4_debug", "nq_dequant_q5_debug",
                 "nq_dequant_q4_debug_bf16", "nq_dequant_q5_debug_bf16", "nq_status_string",
                 "nq_packed_bytes_q4", "nq_packed_bytes_q5", "nq_scale_bytes", "nq_wait_limit",
                 "nq_pack_fp4", "nq_gemm_fp4", "nq_dequant_fp4_debug", "nq_packed_bytes_fp4", "nq_scale_bytes_fp4"):
        assert must in names


def test_projection_signatures_take_scales_separately():
    """The projection calls take (X, Wq, S, Y, T, K, N, stream); the SwiGLU calls
    (X, Wg, Sg, Wu, Su, H, T, K, N, stream); pack writes (wq_packed, s_packed)."""
    src = open(os.path.join(ROOT, "include", "nq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    flat = " ".join(src.split())
    assert ("nq_status nq_gemm_q4(const void* X, const void* Wq, const void* S, void* Y, int T, int K, "
            "int N, void* stream);") in flat
    assert ("nq_status nq_swiglu_q4(const void* X, const void* Wg, const void* Sg, const void* Wu, "
            "const void* Su, void* H, int T, int K, int N, void* stream);") in flat
    assert ("nq_status nq_pack_q4(const uint32_t* wq_canon, const uint16_t* s_canon, int K, int N, "
            "void* wq_packed, void* s_packed, void* stream);") in flat
    assert ("nq_status nq_dequant_q5_debug(const void* Wq, const void* S, float* out, int K, int N, "
            "void* stream);") in flat


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_sizes_and_strings(L):
    from weight_only_groupwise_gb300 import nq
    # packed codes and packed scales: exactly the algorithmic bytes, nothing else
    assert nq.packed_bytes_q4(5120, 17408) == 5120 * 17408 // 2
    assert nq.packed_bytes_q5(5120, 6144) == 5120 * 6144 * 5 // 8
    assert nq.scale_bytes(5120, 17408) == 17408 * 80 * 2
    assert nq.packed_bytes_q4(100, 16) == 0          # K % 64 != 0
    assert nq.packed_bytes_q4(64, 8) == 0            # N % 16 != 0
    assert nq.scale_bytes(64, 8) == 0
    assert nq.packed_bytes_fp4(5120, 17408) == 5120 * 17408 // 2
    assert nq.scale_bytes_fp4(5120, 17408) == 17408 * 5120 // 16
    assert nq.scale_bytes_fp4(96, 16) == 0
    for s in range(-8, 1):
        assert nq.status_string(s).startswith("NQ_")
    assert nq.status_string(-99) == "NQ_ERR_UNKNOWN"
    assert L.nq_version() >> 16 == 2


def test_wait_limit_set_and_query(L):
    from weight_only_groupwise_gb300 import nq
    base = nq.wait_limit(0)
    assert base > 0
    assert nq.wait_limit(12345) == base
    assert nq.wait_limit(-1) == 12345
    assert nq.wait_limit(base) == 12345
    assert nq.wait_limit(0) == base


def test_shape_errors_are_reported_before_any_cuda_call(L):
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(64)
    p16 = P((ctypes.addressof(buf) + 15) & ~15)
    assert L.nq_gemm_q4(p16, p16, p16, p16, 65, 64, 16, None) == -2    # T > 64
    assert L.nq_gemm_q4(p16, p16, p16, p16, -1, 64, 16, None) == -2
    assert L.nq_gemm_q5(p16, p16, p16, p16, 1, 96, 16, None) == -2     # K % 64
    assert L.nq_gemm_q4(p16, p16, p16, p16, 1, 64, 24, None) == -2     # N % 16
    assert L.nq_gemm_q4_noalloc(p16, p16, p16, p16, 65, 64, 16, None) == -2
    assert L.nq_swiglu_q4(p16, p16, p16, p16, p16, p16, 1, 65, 16, None) == -2
    assert L.nq_swiglu_q5(p16, p16, p16, p16, p16, p16, 65, 64, 16, None) == -2
    assert L.nq_swiglu_q5(p16, p16, p16, p16, p16, p16, 1, 64, 40, None) == -2
    assert L.nq_pack_q4(p16, p16, 63, 16, p16, p16, None) == -2
    assert L.nq_dequant_q5_debug(p16, p16, p16, 64, 17, None) == -2
    assert L.nq_dequant_q4_debug_bf16(p16, p16, p16, 32, 16, None) == -2
    assert L.nq_gemm_fp4(p16, p16, p16, ctypes.c_float(1.0), p16, 65, 64, 16, None) == -2
    assert L.nq_gemm_fp4(p16, p16, p16, ctypes.c_float(1.0), p16, 1, 64, 24, None) == -2
    assert L.nq_pack_fp4(p16, p16, 96, 16, p16, p16, None) == -2


def test_empty_problems_launch_nothing(L):
    # T == 0 or N == 0: NQ_OK without touching any pointer (NULLs are fine)
    assert L.nq_gemm_q4(None, None, None, None, 0, 64, 16, None) == 0
    assert L.nq_gemm_q5(None, None, None, None, 4, 64, 0, None) == 0
    assert L.nq_gemm_q4_noalloc(None, None, None, None, 0, 64, 16, None) == 0
    assert L.nq_swiglu_q4(None, None, None, None, None, None, 0, 64, 16, None) == 0
    assert L.nq_swiglu_q5(None, None, None, None, None, None, 3, 64, 0, None) == 0


def test_null_alignment_alias_errors(L):
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(8192)
    base = (ctypes.addressof(buf) + 15) & ~15
    # Q4 64 x 16: 512 code bytes and 32 scale bytes; Q5: 640 code bytes
    x, w, s, w2, s2, y = P(base), P(base + 1024), P(base + 2048), P(base + 3072), P(base + 4096), P(base + 5120)
    assert L.nq_gemm_q4(None, w, s, y, 1, 64, 16, None) == -1
    assert L.nq_gemm_q4(x, None, s, y, 1, 64, 16, None) == -1
    assert L.nq_gemm_q4(x, w, None, y, 1, 64, 16, None) == -1
    assert L.nq_gemm_q4_noalloc(x, w, None, y, 1, 64, 16, None) == -1
    assert L.nq_swiglu_q4(x, w, s, None, s2, y, 1, 64, 16, None) == -1
    assert L.nq_swiglu_q4(x, w, s, w2, None, y, 1, 64, 16, None) == -1
    assert L.nq_gemm_q4(P(base + 2), w, s, y, 1, 64, 16, None) == -3    # X misaligned
    assert L.nq_gemm_q4(x, w, P(base + 2056), y, 1, 64, 16, None) == -3  # S misaligned
    assert L.nq_gemm_q4(x, w, s, P(base + 5128), 1, 64, 16, None) == -3
    # Y overlapping X, the codes or the scales
    assert L.nq_gemm_q4(x, w, s, x, 1, 64, 16, None) == -4
    assert L.nq_gemm_q4(x, w, s, P(base + 1024 + 256), 1, 64, 16, None) == -4
    assert L.nq_gemm_q4(x, w, s, P(base + 2048 + 16), 1, 64, 16, None) == -4
    assert L.nq_gemm_q4_noalloc(x, w, s, P(base + 2048 + 16), 1, 64, 16, None) == -4
    assert L.nq_gemm_q5(x, w, s, P(base + 1024 + 608), 2, 64, 16, None) == -4
    assert L.nq_swiglu_q4(x, w, s, w2, s2, P(base + 4096 + 16), 1, 64, 16, None) == -4
    assert L.nq_swiglu_q5(x, w, s, P(base + 3080), s2, y, 1, 64, 16, None) == -3   # Wu misaligned
    # the packed Q5 64 x 16 codes are 640 bytes: H at Wu + 624 overlaps them
    assert L.nq_swiglu_q5(x, w, s, w2, s2, P(base + 3072 + 624), 1, 64, 16, None) == -4
    # NVFP4 64 x 16: 512 code bytes, 64 scale bytes
    g1 = ctypes.c_float(1.0)
    assert L.nq_gemm_fp4(x, w, None, g1, y, 1, 64, 16, None) == -1
    assert L.nq_gemm_fp4(x, w, s, g1, P(base + 5128), 1, 64, 16, None) == -3
    assert L.nq_gemm_fp4(x, w, s, g1, P(base + 2048 + 48), 1, 64, 16, None) == -4   # Y overlaps the scales
    assert L.nq_gemm_fp4(None, None, None, g1, None, 0, 64, 16, None) == 0
    # pack outputs overlapping an input or each other
    assert L.nq_pack_q4(x, s, 64, 16, x, s2, None) == -4
    assert L.nq_pack_q4(x, s, 64, 16, w2, P(base + 3072 + 256), None) == -4


def test_plan_info_matches_workloads(L):
    from weight_only_groupwise_gb300 import nq
    p = nq.plan_info(4, 0, 1, 5120, 17408, 152)
    assert p["ctas"] == 136 and p["pairs"] == 544 and p["units"] == 544 * 80 and p["slabs"] == 1  # 4 whole pairs each
    p = nq.plan_info(4, 0, 8, 17408, 5120, 152)   # T=8 down projection needs K slabs
    assert p["slabs"] == 3 and p["slab_groups"] * 3 >= 272
    p = nq.plan_info(4, 1, 8, 5120, 17408, 152)   # swiglu pairs gate/up tiles
    assert p["pairs"] == 1088
    p = nq.plan_info(5, 1, 8, 5120, 17408, 152)   # Q5 swiglu: same pairing, larger stages
    assert p["pairs"] == 1088 and p["stages"] >= 2


def test_slab_cluster_switch(L):
    """Query, set and restore the slab-cluster switch (host state only; no launch)."""
    prev = L.nq_slab_clusters(-1)
    assert prev in (0, 1)
    assert L.nq_slab_clusters(1) == prev
    assert L.nq_slab_clusters(-1) == 1
    assert L.nq_slab_clusters(0) == 1
    assert L.nq_slab_clusters(prev) == 0
    assert L.nq_slab_clusters(-1) == prev


def test_grouped_argument_errors(L):
    from weight_only_groupwise_gb300.nq import NqGroup
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(16384)
    base = (ctypes.addressof(buf) + 15) & ~15
    x = base
    gs = (NqGroup * 5)()
    # Q4 64 x 32: 1024 code bytes, 64 scale bytes; outputs 64 bytes each at T=1
    for i in range(5):
        gs[i] = NqGroup(base + 1024 + 2048 * i, base + 1024 + 2048 * i + 1536, base + 12288 + 128 * i, 32)
    arr = ctypes.cast(gs, P)
    assert L.nq_gemm_q4_grouped(P(x), None, 1, 1, 64, None) == -1
    assert L.nq_gemm_q4_grouped(P(x), arr, 0, 1, 64, None) == -2
    assert L.nq_gemm_q4_grouped(P(x), arr, 5, 1, 64, None) == -2
    assert L.nq_gemm_q5_grouped(P(x), arr, 2, 65, 64, None) == -2
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 96, None) == -2        # K % 64
    saved = gs[1].N
    gs[1].N = 40
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 64, None) == -2        # N % 16
    gs[1].N = 0
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 64, None) == -2        # empty group
    gs[1].N = saved
    assert L.nq_gemm_q4_grouped(None, arr, 2, 1, 64, None) == -1
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 0, 64, None) == 0         # T == 0: nothing to do
    y1 = gs[1].Y
    gs[1].Y = base + 12288 + 32                                        # overlaps group 0's Y
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 64, None) == -4
    gs[1].Y = gs[0].Wq + 16                                            # overlaps group 0's codes
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 64, None) == -4
    gs[1].Y = y1 + 2                                                   # misaligned
    assert L.nq_gemm_q4_grouped(P(x), arr, 2, 1, 64, None) == -3
