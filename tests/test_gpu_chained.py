"""Ops launched back to back on one stream with no synchronisation between
them, each consuming the previous one's output (read after write) or
overwriting a buffer the previous one reads (write after read).

Every kernel is a programmatic dependent of the work before it: its CTAs may
start while that work drains, and must not touch global memory before it has
completed.  Intermediate buffers start as NaN, so a stage that read its input
too early gives NaN or a mismatch; each stage is checked against the oracle
applied to the GPU's own previous-stage result (read back at the end).
"""
import pytest
import torch

import oracle
from gen import synth
from tests import test_gpu_elementwise as ew
from tests._helpers import assert_norm_close

pytestmark = pytest.mark.gpu


def _nan_like(t):
    return torch.full_like(t, float("nan"))


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_read_after_write_chain(lib, dtype):
    T = synth.DTYPES[dtype]
    R, H = 2048, 4096
    d = synth.sln_inputs((R, H), dtype=dtype, has_bias=True, seed=21)
    ba = synth.bias_add_inputs((1, R, H), dtype, seed=22)
    sm = synth.bias_softmax_inputs((R, H), (4, H), dtype, data_std=2.0, seed=23)
    x, skip, gamma, beta, bias = (d[k].cuda() for k in ("input", "skip", "gamma", "beta", "bias"))
    b3, skip3, mask = ba["bias"].cuda(), ba["skip"].cuda(), sm["bias"].cuda()
    out1, out2, out3, out4 = (_nan_like(x) for _ in range(4))
    for _ in range(3):  # repeated, so that each chain also follows the previous one
        lib.ep_skip_layer_norm(x, skip, gamma, beta, bias, d["epsilon"], output=out1)
        lib.ep_quick_gelu(out1, 1.702, Y=out2)
        lib.ep_bias_add(out2.view(1, R, H), b3, skip3, Y=out3.view(1, R, H))
        lib.ep_bias_softmax(out3, mask, axis=1, is_inner_broadcast=0, output=out4)
    torch.cuda.synchronize()
    o1, o2, o3, o4 = (t.cpu() for t in (out1, out2, out3, out4))
    assert_norm_close(o1, oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"],
                                                 d["epsilon"])["output"], T)
    ew.check_quick_gelu(o2, o1, 1.702)
    ew.check_bias_add(o3.view(1, R, H), o2.view(1, R, H), ba["bias"], ba["skip"])
    assert_norm_close(o4, oracle.bias_softmax(o3, sm["bias"], axis=1, is_inner_broadcast=0), T)


def test_write_after_read(lib):
    # QuickGelu reads P, then BiasAdd overwrites P in place; then the softmax
    # reads Q (QuickGelu's output) while SkipLayerNorm overwrites Q's source
    R, H = 2048, 4096
    p0 = synth.quick_gelu_inputs(R * H, "f16", seed=31)["X"].view(1, R, H)
    ba = synth.bias_add_inputs((1, R, H), "f16", seed=32)
    d = synth.sln_inputs((R, H), dtype="f16", seed=33)
    P = p0.cuda()
    Q = _nan_like(P)
    lib.ep_quick_gelu(P, 1.702, Y=Q)
    lib.ep_bias_add(P, ba["bias"].cuda(), ba["skip"].cuda(), Y=P)        # writes what QuickGelu read
    lib.ep_skip_layer_norm(d["input"].cuda(), d["skip"].cuda(), d["gamma"].cuda(), d["beta"].cuda(), None,
                           d["epsilon"], output=P.view(R, H))             # and again
    torch.cuda.synchronize()
    ew.check_quick_gelu(Q.cpu(), p0, 1.702)
    assert_norm_close(P.view(R, H).cpu(), oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], None,
                                                                 d["epsilon"])["output"], torch.float16)


def test_split_softmax_after_producer(lib):
    # the split-row softmax (two launches) right after the op that writes its
    # input, and an op right after it that overwrites that input
    rows, cols = 8, 1 << 18
    q = synth.quick_gelu_inputs(rows * cols, "f32", seed=41)["X"].view(rows, cols)
    b = synth.bias_softmax_inputs((rows, cols), (1, cols), "f32", seed=42)["bias"]
    xd, bd = q.cuda(), b.cuda()
    z = _nan_like(xd)
    y = _nan_like(xd)
    ws = torch.empty(lib.ep_bias_softmax_workspace_size(torch.float32, (rows, cols), 1), dtype=torch.uint8,
                     device="cuda")
    lib.ep_quick_gelu(xd, 1.702, Y=z)
    lib.ep_bias_softmax(z, bd, axis=1, is_inner_broadcast=0, output=y, workspace=ws)
    lib.ep_quick_gelu(xd, -1.0, Y=z)                                       # overwrites the softmax input
    torch.cuda.synchronize()
    z1 = torch.from_numpy(oracle.quick_gelu(q, 1.702)).float()
    assert_norm_close(y.cpu(), oracle.bias_softmax(z1, b, axis=1, is_inner_broadcast=0), torch.float32)
    ew.check_quick_gelu(z.cpu(), q, -1.0)


def test_two_streams_at_once(lib):
    # two independent chains on two streams at the same time: the CTAs of both
    # grids share the SMs and each grid hands out only its own tiles.  The
    # kernels are deterministic, so the results must equal a sequential run's
    # bit for bit.
    R, H = 2048, 4096
    ins = [synth.sln_inputs((R, H), dtype="f16", has_bias=True, seed=60 + k) for k in range(2)]
    longs = [synth.bias_softmax_inputs((4, 1 << 18), (1, 1 << 18), "f32", data_std=2.0, seed=70 + k) for k in range(2)]

    def setup(k):
        d, lg = ins[k], longs[k]
        t = {n: d[n].cuda() for n in ("input", "skip", "gamma", "beta", "bias")}
        t["ld"], t["lb"] = lg["data"].cuda(), lg["bias"].cuda()
        t["o1"], t["o2"], t["o3"] = _nan_like(t["input"]), _nan_like(t["input"]), _nan_like(t["ld"])
        t["ws"] = torch.empty(lib.ep_bias_softmax_workspace_size(torch.float32, tuple(t["ld"].shape), 1),
                              dtype=torch.uint8, device="cuda")
        return t

    def chain(t, eps):
        for _ in range(4):
            lib.ep_skip_layer_norm(t["input"], t["skip"], t["gamma"], t["beta"], t["bias"], eps, output=t["o1"])
            lib.ep_quick_gelu(t["o1"], 1.702, Y=t["o2"])
            lib.ep_bias_softmax(t["ld"], t["lb"], axis=1, is_inner_broadcast=0, output=t["o3"], workspace=t["ws"])
            lib.ep_quick_gelu(t["o2"], 1.0, Y=t["o2"])                     # in place

    conc = [setup(k) for k in range(2)]
    seq = [setup(k) for k in range(2)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    for k, st in enumerate(streams):
        with torch.cuda.stream(st):
            chain(conc[k], ins[k]["epsilon"])
    torch.cuda.synchronize()
    for k in range(2):
        chain(seq[k], ins[k]["epsilon"])
    torch.cuda.synchronize()
    for k in range(2):
        for n in ("o1", "o2", "o3"):
            assert torch.equal(conc[k][n].view(torch.int16 if n != "o3" else torch.int32),
                               seq[k][n].view(torch.int16 if n != "o3" else torch.int32)), (k, n)
        d = ins[k]
        assert_norm_close(conc[k]["o1"].cpu(), oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"],
                                                                      d["bias"], d["epsilon"])["output"], torch.float16)
