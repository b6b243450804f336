"""Host logic of the stream-K work split (CPU only): every (slab, pair, group) unit is
processed by exactly one block, blocks get equal shares, and the split-K partial slots are
unique and inside the workspace the plan reserves."""
import pytest

SHAPES = [
    # bits, mode, T, K, N
    (4, 0, 1, 256, 128), (4, 0, 1, 5120, 17408), (5, 0, 8, 5120, 6144), (4, 1, 8, 5120, 17408),
    (4, 0, 8, 17408, 5120), (5, 0, 8, 5120, 1024), (5, 0, 3, 6144, 5120), (4, 0, 8, 6208, 48),
    (4, 0, 5, 64, 16), (4, 0, 2, 1024, 272), (4, 1, 7, 17408, 48), (5, 0, 1, 64, 16),
    (5, 1, 8, 5120, 17408), (5, 1, 4, 17408, 64), (5, 1, 1, 640, 16),
]


@pytest.fixture(scope="module")
def nq():
    from weight_only_groupwise_gb300 import build
    build.build()
    from weight_only_groupwise_gb300 import nq
    return nq


@pytest.mark.parametrize("bits,mode,T,K,N", SHAPES)
@pytest.mark.parametrize("sms", [152, 148, 7, 1])
def test_partition_covers_every_unit_once(nq, bits, mode, T, K, N, sms):
    info = nq.plan_info(bits, mode, T, K, N, sms)
    G, RP, S, GS = K // 64, info["pairs"], info["slabs"], info["slab_groups"]
    assert info["ctas"] <= sms and info["units"] == RP * G
    seen = set()
    slots = set()
    per_cta = []
    fan_in = {}
    for c in range(info["ctas"]):
        segs = nq.plan_segments(bits, mode, T, K, N, sms, c)
        n_units = 0
        for (s, rp, ga, gb) in segs:
            assert 0 <= s < S and 0 <= rp < RP and s * GS <= ga < gb <= min(G, (s + 1) * GS)
            for g in range(ga, gb):
                assert (rp, g) not in seen
                seen.add((rp, g))
            # slot index s*RP + rp + c must be unique and inside the reserved slots
            slot = s * RP + rp + c
            assert slot not in slots and slot < info["ws_slots"]
            slots.add(slot)
            fan_in[rp] = fan_in.get(rp, 0) + 1
            n_units += gb - ga
        per_cta.append(n_units)
    assert len(seen) == RP * G
    assert max(per_cta) - min(per_cta) <= 1          # equal shares
    # every pair is covered by at least one run per slab
    assert all(fan_in[rp] >= S for rp in range(RP))
    # a run writes its output directly exactly when it is its pair's only contribution
    for c in range(info["ctas"]):
        segs = nq.plan_segments(bits, mode, T, K, N, sms, c)
        for (s, rp, ga, gb) in segs:
            complete = S == 1 and ga == 0 and gb == G
            assert complete == (fan_in[rp] == 1)
        # processing order: natural order with several slabs; with one slab the first and
        # last natural runs come first and the block ends on a complete run (if it has one)
        nat = sorted(segs, key=lambda x: (x[0], x[1], x[2]))
        if S > 1 or len(segs) <= 2:
            assert segs == nat
        else:
            assert segs[0] == nat[0] and segs[1] == nat[-1] and segs[2:] == nat[1:-1]
            assert segs[-1][2] == 0 and segs[-1][3] == G


@pytest.mark.parametrize("bits,T,K,N,sms,ctas", [
    (5, 8, 5120, 6144, 152, 96),     # 192 pairs: two whole pairs per block
    (5, 1, 5120, 6144, 152, 96),
    (4, 1, 1024, 2432, 152, 76),     # 76 pairs: one per block
    (4, 1, 5120, 17408, 152, 136),   # 544 pairs: four per block on 136 SMs
    (5, 8, 5120, 1024, 152, 32),     # 32 pairs: the rings of 32 blocks hold the whole problem
    (5, 1, 6144, 5120, 152, 80),     # 160 pairs, five stages per block: 80 blocks
    (5, 8, 6144, 5120, 152, 152),    # the same at T=8: two stages, too little in flight
    (4, 8, 17408, 5120, 152, 152),   # several slabs: stream-K
    (4, 1, 5120, 17408, 7, 7),       # 544 pairs on 7 SMs: 78 per block does not divide, stream-K
])
def test_whole_pairs_when_they_divide_evenly(nq, bits, T, K, N, sms, ctas):
    """With one slab and row pairs that divide evenly into at most four per block (the fewest
    that fit the SMs), the grid takes whole pairs per block (no segment is a partial run)
    when those blocks' rings hold at least 8 MB in flight or the whole problem."""
    info = nq.plan_info(bits, 0, T, K, N, sms)
    assert info["ctas"] == ctas
    if ctas < sms:
        G = K // 64
        for c in range(ctas):
            segs = nq.plan_segments(bits, 0, T, K, N, sms, c)
            assert all(ga == 0 and gb == G for (_, _, ga, gb) in segs)
            assert len(segs) == info["pairs"] // ctas


def test_many_pairs_per_block_stay_stream_k(nq):
    """The fused gate/up block of the SwiGLU workload has 1088 pairs: eight per block would
    leave 16 SMs idle, so the plan keeps stream-K over every SM."""
    assert nq.plan_info(4, 1, 8, 5120, 17408, 152)["ctas"] == 152
    assert nq.plan_info(5, 1, 8, 5120, 17408, 152)["ctas"] == 152


CLUSTER_SHAPES = [
    # bits, mode, T, K, N, clusters
    (4, 0, 8, 17408, 5120, 48), (5, 0, 8, 17408, 5120, 48), (4, 0, 4, 17408, 5120, 72),
    (4, 0, 3, 17408, 64, 50), (4, 0, 8, 6208, 48, 7), (4, 1, 8, 17408, 48, 48),
    (5, 1, 4, 17408, 64, 72), (4, 0, 8, 12352, 112, 3), (4, 0, 8, 24576, 16, 38),
]


@pytest.mark.parametrize("bits,mode,T,K,N,clusters", CLUSTER_SHAPES)
def test_cluster_partition_covers_every_unit_once(nq, bits, mode, T, K, N, clusters):
    """Slab clusters: block rank r only ever touches slab r; every (pair, group) of the
    real problem is processed by exactly one block; the ranks of a cluster walk the same
    runs (same pairs, same slab-local ranges before clipping to the shorter last slab)."""
    import numpy as np
    info = nq.plan_cluster_info(bits, mode, T, K, N, clusters)
    S, gs, RP, G = info["cluster"], info["slab_groups"], info["pairs"], K // 64
    assert 2 <= S <= 4 and gs % 8 == 0 and (S - 1) * gs < G <= S * gs
    assert info["ctas"] == info["clusters"] * S and info["clusters"] <= clusters
    assert info["stages"] >= 2
    # split-K between clusters: one ticket per pair, one partial slot per (pair, cluster) run
    # boundary, as a one-slab stream-K plan over the clusters
    assert info["ws_slots"] == info["pairs"] + info["clusters"]
    covered = np.zeros((RP, G), np.int32)
    runs = {}
    for cta in range(info["ctas"]):
        c, r = divmod(cta, S)
        segs = nq.plan_cluster_segments(bits, mode, T, K, N, clusters, cta)
        lo, hi = r * gs, min((r + 1) * gs, G)
        for (s, rp, ga, gb) in segs:
            assert s == r and lo <= ga <= gb <= hi
            covered[rp, ga:gb] += 1
        runs.setdefault(c, []).append([(rp, ga - lo) for (s, rp, ga, gb) in segs])
    assert (covered == 1).all()
    for c, per_rank in runs.items():
        pairs = [[rp for rp, _ in rr] for rr in per_rank]
        assert all(p == pairs[0] for p in pairs)
        starts0 = [a for _, a in per_rank[0]]
        assert all([a for _, a in rr] == starts0 or r == S - 1 for r, rr in enumerate(per_rank))


def test_no_cluster_plan_for_one_slab(nq):
    from weight_only_groupwise_gb300.nq import NqError
    with pytest.raises(NqError):
        nq.plan_cluster_info(4, 0, 1, 5120, 17408, 48)     # one slab
    with pytest.raises(NqError):
        nq.plan_cluster_info(4, 0, 2, 17408, 5120, 48)     # fp16 operands, one slab


# The limit of nq_gemm_q4_noalloc's fixed scratch (2048 partial slots, 4096 tickets) as
# stated in include/nq.h for a 152-SM GB300: the largest N per (T, K), from the planner.
NOALLOC_LIMITS = [
    # T, K, largest N
    (1, 5120, 60672), (1, 49152, 60672), (2, 24576, 60672), (3, 16384, 60672), (4, 12288, 60672),
    (6, 8192, 60672), (8, 6144, 60672), (4, 17408, 30336), (8, 12288, 30336), (8, 17408, 20224),
    (8, 24576, 15168),
]


def _noalloc_fits(nq, T, K, N, sms=152):
    p = nq.plan_info(4, 0, T, K, N, sms)
    return p["ws_slots"] <= 2048 and p["pairs"] <= 4096


@pytest.mark.parametrize("T,K,n_max", NOALLOC_LIMITS)
def test_noalloc_limits_stated_in_header(nq, T, K, n_max):
    assert _noalloc_fits(nq, T, K, n_max)
    assert not _noalloc_fits(nq, T, K, n_max + 16)


@pytest.mark.parametrize("T,k_max", [(1, 49152), (2, 24576), (3, 16384), (4, 12288), (5, 8192),
                                     (6, 8192), (7, 6144), (8, 6144)])
def test_one_slab_k_limits_stated_in_header(nq, T, k_max):
    assert nq.plan_info(4, 0, T, k_max, 512, 152)["slabs"] == 1
    assert nq.plan_info(4, 0, T, k_max + 64, 512, 152)["slabs"] == 2


@pytest.mark.parametrize("bits,T,K,N", [(4, 64, 5120, 17408), (5, 16, 5120, 6144), (4, 33, 17408, 5120),
                                        (5, 9, 64, 16), (4, 64, 192, 4096), (5, 48, 6208, 1040),
                                        (14, 40, 5120, 17408), (14, 64, 512, 144)])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_tc_plan(nq, bits, T, K, N, sms):
    """The tensor-core kernel's split: every (row block, K piece) is one block, the pieces of a
    row block cover its K groups once, at most one block per SM when there are enough row
    blocks, and the stages fit the shared memory."""
    p = nq.plan_tc_info(bits, T, K, N, sms)
    G = K // 64
    assert p["groups"] == G and p["row_blocks"] == -(-N // 128)
    assert p["ctas"] == p["row_blocks"] * p["k_pieces"]
    assert p["ctas"] <= max(sms, p["row_blocks"])
    bounds = [kp * G // p["k_pieces"] for kp in range(p["k_pieces"] + 1)]
    assert bounds[0] == 0 and bounds[-1] == G and all(b1 > b0 for b0, b1 in zip(bounds, bounds[1:]))
    assert p["tokens_padded"] in (16, 32, 64) and p["tokens_padded"] >= T > p["tokens_padded"] // 2 - (8 if T <= 16 else 0)
    assert 2 <= p["stages"] and p["smem_bytes"] <= 227 * 1024


# The routing of the pages' shapes on a 152-SM GB300, each choice the measured winner (the
# design notes give the times): (bits, mode, T, K, N) -> (kernel, launches, operands, split,
# blocks, K slabs or pieces). kernel 0 = mma.sync 8-token, 1 = tcgen05; operands 0 = fp16,
# 1 = bf16; split 0 = stream-K, 1 = whole row pairs, 3 = row blocks x K pieces.
ROUTES = [
    ((4, 0, 1, 5120, 17408), (0, 1, 0, 1, 136, 1)),    # decode Q4: fp16, four whole pairs per block
    ((4, 0, 2, 5120, 17408), (0, 1, 0, 1, 136, 1)),
    ((4, 0, 3, 5120, 17408), (0, 1, 1, 1, 136, 1)),    # T >= 3: bf16 operands
    ((4, 0, 8, 5120, 17408), (0, 1, 1, 1, 136, 1)),
    ((5, 0, 1, 5120, 6144), (0, 1, 0, 1, 96, 1)),      # spec-verify Q5: two whole pairs per block
    ((5, 0, 8, 5120, 6144), (0, 1, 1, 1, 96, 1)),
    ((5, 0, 8, 5120, 1024), (0, 1, 1, 1, 32, 1)),      # kv: one pair per block
    ((5, 0, 1, 6144, 5120), (0, 1, 0, 1, 80, 1)),      # out projection T=1: whole pairs
    ((5, 0, 8, 6144, 5120), (0, 1, 1, 0, 152, 1)),     # ... T=8: two stages only, stream-K
    ((4, 0, 8, 17408, 5120), (0, 1, 1, 0, 152, 3)),    # down projection T=8: three K slabs
    ((4, 1, 8, 5120, 17408), (0, 1, 1, 0, 152, 1)),    # fused gate/up: eight pairs per block, stream-K
    ((5, 1, 8, 5120, 17408), (0, 1, 1, 0, 152, 1)),
    ((14, 0, 1, 5120, 17408), (0, 1, 0, 1, 136, 1)),   # NVFP4: fp16 at every T
    ((14, 0, 8, 5120, 17408), (0, 1, 0, 1, 136, 1)),
    ((4, 0, 9, 5120, 17408), (1, 1, 1, 3, 136, 1)),    # T > 8: one tensor-core launch
    ((4, 0, 64, 5120, 17408), (1, 1, 1, 3, 136, 1)),
    ((5, 0, 16, 5120, 6144), (1, 1, 1, 3, 144, 3)),    # 48 row blocks x 3 K pieces
    ((4, 0, 16, 17408, 5120), (1, 1, 1, 3, 120, 3)),
    ((4, 1, 16, 5120, 17408), (1, 2, 1, 3, 136, 1)),   # SwiGLU: gate launch, then up launch
    ((14, 0, 40, 5120, 17408), (1, 1, 1, 3, 136, 1)),
    ((14, 1, 8, 5120, 17408), (0, 1, 0, 0, 152, 1)),   # NVFP4 SwiGLU: fp16, stream-K like Q4
    ((14, 1, 16, 5120, 17408), (1, 2, 1, 3, 136, 1)),  # ... and two tensor-core launches
]


@pytest.mark.parametrize("shape,route", ROUTES)
def test_routing_table(nq, shape, route):
    r = nq.route_info(*shape, 152)
    assert (r["kernel"], r["launches"], r["operands"], r["split"], r["ctas"], r["k_split"]) == route
    if r["kernel"] == 0:
        info = nq.plan_info(shape[0], shape[1], min(shape[2], 8), shape[3], shape[4], 152) if shape[0] != 14 else None
        if info:
            assert info["ctas"] == r["ctas"] and info["slabs"] == r["k_split"]
    else:
        tc = nq.plan_tc_info(shape[0], shape[2], shape[3], shape[4], 152)
        assert tc["ctas"] == r["ctas"] and tc["k_pieces"] == r["k_split"] and tc["tokens_padded"] == r["tokens_padded"]


def test_routing_without_tensor_core_batches(nq):
    prev = nq.tensor_core_batches(0)
    try:
        r = nq.route_info(4, 0, 20, 5120, 17408, 152)
        assert r["kernel"] == 0 and r["launches"] == 3 and r["operands"] == 1 and r["tokens_padded"] == 8
        assert nq.route_info(4, 1, 64, 5120, 17408, 152)["launches"] == 8
    finally:
        nq.tensor_core_batches(prev)
    assert nq.route_info(4, 0, 20, 5120, 17408, 152)["kernel"] == 1


def test_routing_rejects_bad_arguments(nq):
    from weight_only_groupwise_gb300.nq import NqError
    for args in [(3, 0, 1, 64, 16), (6, 1, 1, 64, 16), (4, 2, 1, 64, 16), (4, 0, 0, 64, 16), (4, 0, 65, 64, 16),
                 (4, 0, 1, 96, 16), (4, 0, 1, 64, 24)]:
        with pytest.raises(NqError):
            nq.route_info(*args, 152)
