"""Host-side accounting of bench.py (no GPU): the algorithmic bytes of each workload are the
codes + scales + X + Y of its calls, the launch counts per step match the routing of
include/nq.h, the ncu traffic record is read only for the kernel sources it was taken on, and
the pages' single-op numbers ride along as context."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes():
    # decode Q4 T=1: codes K*N/2 + fp16 scales N*K/32 + X 2TK + Y 2TN
    assert bench.proj_bytes(4, 1, 5120, 17408) == 44564480 + 2785280 + 10240 + 34816 == 47394816
    # verify Q5 T=8: codes 5KN/8
    assert bench.proj_bytes(5, 8, 5120, 6144) == 19660800 + 983040 + 81920 + 98304 == 20824064
    # NVFP4: codes K*N/2 + e4m3 scales N*K/16
    assert bench.fp4_bytes(1, 5120, 17408) == 44564480 + 5570560 + 10240 + 34816
    assert bench.weight_bytes(bench.FP4, 5120, 17408) == 44564480 + 5570560
    assert bench.workload_bytes(bench.WORKLOADS["decode_fp4"]) == bench.fp4_bytes(1, 5120, 17408)
    w4 = bench.WORKLOADS["swiglu_block_fp4"]
    assert bench.workload_bytes(w4) == (2 * (44564480 + 5570560) + 8 * 5120 * 2 + 8 * 17408 * 2
                                        + bench.fp4_bytes(8, 17408, 5120))
    # SwiGLU block: two weight sets on one X, one H
    w = bench.WORKLOADS["swiglu_block"]
    assert bench.workload_bytes(w) == (2 * (44564480 + 2785280) + 8 * 5120 * 2 + 8 * 17408 * 2
                                       + bench.proj_bytes(4, 8, 17408, 5120))


def test_launches_per_step_follow_the_routing():
    lp = bench.launches_per_step
    assert lp(dict(bench.WORKLOADS["decode_q4"])) == 1
    assert lp(dict(bench.WORKLOADS["swiglu_block"], T=8)) == 2             # fused gate/up, down
    assert lp(dict(bench.WORKLOADS["swiglu_block"], T=16)) == 3            # gate, up, down
    stack = bench.WORKLOADS["layer_stack"]
    assert lp(dict(stack, T=1)) == 4 * 64                                  # swiglu, down, grouped, out
    assert lp(dict(stack, T=16)) == lp(dict(stack, T=64)) == 6 * 64        # + gate/up split, 2 matrices


def test_traffic_record_only_for_its_sources(monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, e in rec.items():
        workload, T = key.split("@T")
        assert e["dram_bytes_per_launch"] > 0 and os.path.exists(os.path.join(ROOT, e["source"]))
        monkeypatch.setattr(bench, "kernel_hash", lambda h=e["kernel_hash"]: h)
        assert bench.ncu_traffic(workload, int(T)) == e["dram_bytes_per_launch"]
        monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
        assert bench.ncu_traffic(workload, int(T)) is None
    assert bench.ncu_traffic("decode_q4", 3) is None                       # no capture at T=3


def test_pages_context():
    c = bench.PAGES_CONTEXT
    assert c["t8_attention_q5_gate_value_us"] == {"before": 57.344, "after": 39.936}
    assert c["t8_gdn_qk_q4_us"] == {"before": 35.840, "after": 31.744}
