"""Recorded programs on the GPU: a decoder layer's projection calls (fused gate/up SwiGLU, the
down projection, the grouped q-gate/kv projections, the out projection, an NVFP4 projection)
recorded once and replayed as one CUDA graph write the same bits as the same calls made
eagerly on one stream, and the H of the replay matches the fp64 oracle. A replay reads X as
it is at launch time; a moved workspace makes the next launch build again."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

K, NH, NQ, NKV, KO = 640, 1088, 384, 64, 384   # a small layer: hidden 640, MLP 1088


@pytest.fixture(scope="module")
def nq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from weight_only_groupwise_gb300 import build
    build.build()
    from weight_only_groupwise_gb300 import nq
    return nq


def weights(nq, bits, K_, N_, seed):
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    wn = si.device_code_words(N_, K_ // 8, gen, dev)
    if bits == 5:
        wh = si.device_code_words(N_, K_ // 32, gen, dev)
    s = si.device_scales(N_, K_, gen, dev)
    return nq.pack_q4(wn, s, K_, N_) if bits == 4 else nq.pack_q5(wn, wh, s, K_, N_)


def fp4_weights(nq, K_, N_, seed):
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return nq.pack_fp4(si.device_code_words(N_, K_ // 8, gen, dev), si.device_fp4_scales(N_, K_, gen, dev), K_, N_)


class Layer:
    """The projections of one decoder layer (dims: hidden K, MLP NH, q-gate NQ, kv NKV, out
    input KO, NVFP4 output NF), with its activations and output buffers."""

    def __init__(self, nq, T, seed, dims=(K, NH, NQ, NKV, KO, 272)):
        dev = torch.device("cuda", 0)
        self.d = k, nh, nqg, nkv, ko, nf = dims
        self.gate, self.up = weights(nq, 4, k, nh, seed), weights(nq, 4, k, nh, seed + 1)
        self.down = weights(nq, 4, nh, k, seed + 2)
        self.qg, self.kv = weights(nq, 5, k, nqg, seed + 3), weights(nq, 5, k, nkv, seed + 4)
        self.out = weights(nq, 5, ko, k, seed + 5)
        self.f4 = fp4_weights(nq, k, nf, seed + 6)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + 7)
        self.x = si.device_activations(T, k, gen, dev)
        self.x6 = si.device_activations(T, ko, gen, dev)
        self.outs = [torch.empty((T, n), dtype=torch.bfloat16, device=dev) for n in (nh, k, nqg, nkv, k, nf)]

    def eager(self, nq):
        k, nh, nqg, nkv, ko, nf = self.d
        h = nq.swiglu_q4(self.x, *self.gate, *self.up, nh)
        yd = nq.gemm_q4(h, *self.down, k)
        yq, ykv = nq.gemm_q5_grouped(self.x, [(*self.qg, nqg), (*self.kv, nkv)])
        yo = nq.gemm_q5(self.x6, *self.out, k)
        yf = nq.gemm_fp4(self.x, *self.f4, si.FP4_GLOBAL_SCALE, nf)
        return [h, yd, yq, ykv, yo, yf]

    def record(self, nq):
        k, nh, nqg, nkv, ko, nf = self.d
        p = nq.Program()
        h, yd, yq, ykv, yo, yf = self.outs
        p.swiglu_q4(self.x, *self.gate, *self.up, nh, out=h)
        p.gemm_q4(h, *self.down, k, out=yd)
        p.grouped_q5(self.x, [(*self.qg, nqg), (*self.kv, nkv)], outs=[yq, ykv])
        p.gemm_q5(self.x6, *self.out, k, out=yo)
        p.gemm_fp4(self.x, *self.f4, si.FP4_GLOBAL_SCALE, nf, out=yf)
        return p


def same_bits(a, b):
    return all(torch.equal(u.view(torch.int16), v.view(torch.int16)) for u, v in zip(a, b))


@pytest.mark.parametrize("T", [1, 8, 40])
def test_program_replays_a_layer_bit_for_bit(nq, T):
    ly = Layer(nq, T, 900 + T)
    ref = ly.eager(nq)
    p = ly.record(nq)
    for o in ly.outs:
        o.fill_(0)
    p.launch()
    torch.cuda.synchronize()
    nq.device_error()
    assert same_bits(ly.outs, ref)
    i = p.info()
    # T <= 8: one launch per call; T = 40: the SwiGLU block and the grouped call are two
    # tensor-core launches each
    assert i["calls"] == 5 and i["builds"] == 1 and i["failed_call"] == -1
    assert i["kernels"] == (5 if T <= 8 else 7)
    # a replay reads X as it is at launch time
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    ly.x.copy_(si.device_activations(T, K, gen, ly.x.device))
    ly.x6.copy_(si.device_activations(T, KO, gen, ly.x.device))
    p.launch()
    ref2 = ly.eager(nq)
    torch.cuda.synchronize()
    assert same_bits(ly.outs, ref2) and not same_bits(ref, ref2)
    p.close()


@pytest.mark.parametrize("T", [8, 40])
def test_program_full_size_layer(nq, T):
    """One 27B-class layer at full size (the layer-stack shapes: gate/up 5120 x 17408, down
    17408 x 5120, q-gate 5120 x 6144, kv 5120 x 1024, out 6144 x 5120; NVFP4 5120 x 17408), in
    the launch configuration a replay of the stack uses: bit for bit the eager calls."""
    ly = Layer(nq, T, 990 + T, dims=(5120, 17408, 6144, 1024, 6144, 17408))
    ref = ly.eager(nq)
    p = ly.record(nq)
    for o in ly.outs:
        o.fill_(0)
    p.launch()
    torch.cuda.synchronize()
    nq.device_error()
    assert same_bits(ly.outs, ref)
    assert all(torch.isfinite(o.float()).all() for o in ly.outs)
    p.close()


def test_program_swiglu_matches_the_oracle(nq):
    """The replay's H against the fp64 oracle on host-drawn inputs, at the parity bar of the
    eager call."""
    T, K_, N_ = 8, 640, 272
    pr = si.swiglu_problem(T, K_, N_, 91)
    wg = gu.pack_q4(nq, pr["wg"], pr["sg"], K_, N_)
    wu = gu.pack_q4(nq, pr["wu"], pr["su"], K_, N_)
    x = gu.dev_bf16(pr["x"])
    h = torch.empty((T, N_), dtype=torch.bfloat16, device="cuda")
    p = nq.Program()
    p.swiglu_q4(x, *wg, *wu, N_, out=h)
    p.launch()
    torch.cuda.synchronize()
    g, u, _ = oracle.swiglu_q4(pr["x"], pr["wg"], pr["sg"], pr["wu"], pr["su"], T, K_, N_)
    h_exact = g / (1.0 + np.exp(-g)) * u
    assert gu.rel_err(gu.host_f64(h), h_exact) <= gu.TOL
    p.close()


def test_program_rebuilds_after_the_workspace_moves(nq):
    ly = Layer(nq, 8, 950)
    ref = ly.eager(nq)
    p = ly.record(nq)
    p.build()
    p.launch()
    torch.cuda.synchronize()
    assert same_bits(ly.outs, ref) and p.info()["builds"] == 1
    p.launch()
    assert p.info()["builds"] == 1          # nothing moved: the same graph
    torch.cuda.synchronize()
    nq.shutdown()                           # frees the workspace the graph points at
    for o in ly.outs:
        o.fill_(0)
    p.launch()                              # builds again on the new workspace
    torch.cuda.synchronize()
    nq.device_error()
    assert same_bits(ly.outs, ref) and p.info()["builds"] == 2
    p.close()


def test_program_on_another_stream_and_empty_program(nq):
    ly = Layer(nq, 3, 960)
    ref = ly.eager(nq)
    p = ly.record(nq)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    p.launch(stream=s)
    s.synchronize()
    assert same_bits(ly.outs, ref)
    p.close()
    e = nq.Program()
    e.build()
    e.launch()
    torch.cuda.synchronize()
    assert e.info() == {"calls": 0, "kernels": 0, "builds": 1, "failed_call": -1}
    e.close()


def test_program_recording_after_build_builds_again(nq):
    ly = Layer(nq, 8, 970)
    ref = ly.eager(nq)
    p = nq.Program()
    h, yd = ly.outs[0], ly.outs[1]
    p.swiglu_q4(ly.x, *ly.gate, *ly.up, NH, out=h)
    p.launch()
    assert p.info()["kernels"] == 1
    p.gemm_q4(h, *ly.down, K, out=yd)         # marks the program for building again
    p.launch()
    torch.cuda.synchronize()
    i = p.info()
    assert i["calls"] == 2 and i["kernels"] == 2 and i["builds"] == 2
    assert same_bits([h, yd], ref[:2])
    p.close()


@pytest.mark.parametrize("T", [8, 24])
def test_program_nvfp4_mlp_bit_for_bit(nq, T):
    """An NVFP4 MLP (SwiGLU block with its own gate and up tensor scales, then the down
    projection) replayed as a program writes the bits of the eager calls."""
    dev = torch.device("cuda", 0)
    wg, wu, wd = fp4_weights(nq, K, NH, 980), fp4_weights(nq, K, NH, 981), fp4_weights(nq, NH, K, 982)
    gen = torch.Generator(device=dev)
    gen.manual_seed(983)
    x = si.device_activations(T, K, gen, dev)
    gg, gu_, gd = 0.0078125, 0.005859375, 0.001953125
    h_ref = nq.swiglu_fp4(x, *wg, gg, *wu, gu_, NH)
    y_ref = nq.gemm_fp4(h_ref, *wd, gd, K)
    p = nq.Program()
    h = p.swiglu_fp4(x, *wg, gg, *wu, gu_, NH)
    y = p.gemm_fp4(h, *wd, gd, K)
    p.launch()
    torch.cuda.synchronize()
    nq.device_error()
    assert same_bits([h, y], [h_ref, y_ref])
    assert p.info()["kernels"] == (2 if T <= 8 else 3)
    p.close()


_FRESH_SCRIPT = r"""
import torch
import numpy as np
import oracle, seeded_inputs as si
from tests import gpu_util as gu
from weight_only_groupwise_gb300 import nq
# a fresh process whose first tensor-core and NVFP4 calls are made inside a program's capture
T, K, N = 24, 640, 272
p = si.q4_problem(T, K, N, 991)
w = gu.pack_q4(nq, p["wq"], p["s"], K, N)
x = gu.dev_bf16(p["x"])
q = si.swiglu_fp4_problem(T, K, N, 992)
wg = nq.pack_fp4(gu.dev_u32(q["cg"]), torch.from_numpy(np.ascontiguousarray(q["sfg"])).cuda(), K, N)
wu = nq.pack_fp4(gu.dev_u32(q["cu"]), torch.from_numpy(np.ascontiguousarray(q["sfu"])).cuda(), K, N)
xq = gu.dev_bf16(q["x"])
torch.cuda.synchronize()
prog = nq.Program()
y = prog.gemm_q4(x, *w, N)
h = prog.swiglu_fp4(xq, *wg, q["gg"], *wu, q["gu"], N)
prog.launch()
torch.cuda.synchronize()
nq.device_error()
assert prog.info()["kernels"] == 3, prog.info()
assert gu.rel_err(gu.host_f64(y), oracle.gemm_q4(p["x"], p["wq"], p["s"], T, K, N)) <= gu.TOL
g, u, _ = oracle.swiglu_fp4(q["x"], q["cg"], q["sfg"], q["gg"], q["cu"], q["sfu"], q["gu"], T, K, N)
assert gu.rel_err(gu.host_f64(h), g / (1.0 + np.exp(-g)) * u) <= gu.TOL
print("fresh-ok")
"""


def test_program_builds_in_a_fresh_process(nq):
    """A process whose first tensor-core calls are recorded: building the program reserves the
    workspace and looks up the tensor-map encoder before the capture, so the capture allocates
    nothing and queries nothing, and the replay matches the oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FRESH_SCRIPT], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "fresh-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
