"""The ops captured in a CUDA graph and replayed.

Each launch carries the programmatic-dependency attribute and the staged
kernels hand tiles out with launch control; both must survive stream
capture.  The kernels are deterministic (a tile's result does not depend on
which CTA computes it), so graph replays must reproduce the eager results
bit for bit.
"""
import pytest
import torch

import oracle
from gen import synth
from tests._helpers import assert_bit_exact, assert_norm_close

pytestmark = pytest.mark.gpu


def _chain(lib, t, ws):
    lib.ep_skip_layer_norm(t["x"], t["skip"], t["gamma"], t["beta"], t["bias"], 1e-5, output=t["o1"],
                           input_skip_bias_sum=t["sum"])
    lib.ep_quick_gelu(t["o1"], 1.702, Y=t["o2"])
    lib.ep_bias_add(t["o2"].view(1, *t["o2"].shape), t["b3"], t["skip3"], Y=t["o3"].view(1, *t["o3"].shape))
    lib.ep_bias_softmax(t["o3"], t["mask"], axis=1, is_inner_broadcast=0, output=t["o4"])
    lib.ep_bias_softmax(t["long"], t["long_bias"], axis=1, is_inner_broadcast=0, output=t["o5"], workspace=ws)


def test_graph_replay_matches_eager(lib):
    R, H = 1024, 4096
    d = synth.sln_inputs((R, H), dtype="f16", has_bias=True, seed=51)
    ba = synth.bias_add_inputs((1, R, H), "f16", seed=52)
    sm = synth.bias_softmax_inputs((R, H), (8, H), "f16", seed=53)
    lg = synth.bias_softmax_inputs((4, 1 << 18), (2, 1 << 18), "f32", data_std=2.0, seed=54)
    t = dict(x=d["input"].cuda(), skip=d["skip"].cuda(), gamma=d["gamma"].cuda(), beta=d["beta"].cuda(),
             bias=d["bias"].cuda(), b3=ba["bias"].cuda(), skip3=ba["skip"].cuda(), mask=sm["bias"].cuda(),
             long=lg["data"].cuda(), long_bias=lg["bias"].cuda())
    for k in ("o1", "sum", "o2", "o3", "o4"):
        t[k] = torch.empty(R, H, dtype=torch.float16, device="cuda")
    t["o5"] = torch.empty_like(t["long"])
    ws = torch.empty(lib.ep_bias_softmax_workspace_size(torch.float32, tuple(lg["data"].shape), 1),
                     dtype=torch.uint8, device="cuda")
    outs = ("o1", "sum", "o2", "o3", "o4", "o5")

    _chain(lib, t, ws)                                   # eager
    torch.cuda.synchronize()
    eager = {k: t[k].clone() for k in outs}

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _chain(lib, t, ws)                               # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _chain(lib, t, ws)
    for k in outs:
        t[k].fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for k in outs:
        assert_bit_exact(t[k].cpu(), eager[k].cpu())
    assert_norm_close(eager["o1"].cpu(), oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"],
                                                                d["bias"], 1e-5)["output"], torch.float16)
