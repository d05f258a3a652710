"""SkipLayerNormalization: CUDA path (through the C ABI) vs the float64 oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gen import synth
from tests._helpers import Guarded, assert_bit_exact, assert_norm_close, offset_copy

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16}


def run(lib, d, residual=False, offsets=None, guard=True, epsilon=None):
    """Run the GPU op on generated CPU inputs d; returns (out, sum) CPU tensors."""
    dev = {}
    keep = []
    offsets = offsets or {}
    for k in ("input", "skip", "gamma", "beta", "bias"):
        t = d[k]
        if t is None:
            dev[k] = None
        elif k in offsets:
            raw, v = offset_copy(t, offsets[k])
            keep.append(raw)
            dev[k] = v
        else:
            dev[k] = t.cuda()
    x = d["input"]
    go = Guarded(x.shape, x.dtype, offset_bytes=offsets.get("output", 0))
    gs = Guarded(x.shape, x.dtype, offset_bytes=offsets.get("sum", 0)) if residual else None
    eps = d["epsilon"] if epsilon is None else epsilon
    lib.ep_skip_layer_norm(dev["input"], dev["skip"], dev["gamma"], dev["beta"], dev["bias"], eps,
                           output=go.tensor, input_skip_bias_sum=gs.tensor if gs else None)
    torch.cuda.synchronize()
    if guard:
        go.check()
        if gs:
            gs.check()
    return go.tensor.cpu(), (gs.tensor.cpu() if gs else None)


def check(d, out, s, rows=None, epsilon=None):
    eps = d["epsilon"] if epsilon is None else epsilon
    H = d["input"].shape[-1]
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], eps, rows=rows)["output"]
    got = out.reshape(-1, H)
    if rows is not None:
        got = got[rows]
    err = assert_norm_close(got, o, d["input"].dtype)
    if s is not None:
        want = oracle.skip_bias_sum(d["input"], d["skip"], d["bias"], rows=rows)
        gs = s.reshape(-1, H)
        assert_bit_exact(gs[rows] if rows is not None else gs, want)
    return err


def _load_combos():
    with open(os.path.join(os.path.dirname(__file__), "golden", "sln_manifest_combinations.json")) as f:
        return json.load(f)["combinations"]


@pytest.mark.parametrize("combo", _load_combos(), ids=lambda c: f"r{c['rank']}-{c['T']}-beta{int(c['beta'])}-bias{int(c['bias'])}-res{int(c['residual'])}")
@pytest.mark.parametrize("H", [768, 771])
def test_manifest_combinations(lib, combo, H):
    if combo["H"] == "mult4" and H % 4:
        H = 772
    if combo["rank"] == 2:
        shapes = [((37, H), None)]
    else:
        shapes = [((3, 11, H), None), ((3, 11, H), (1, 11, H)), ((3, 11, H), (11, H))]
    for in_shape, skip_shape in shapes:
        d = synth.sln_inputs(in_shape, skip_shape, combo["T"], has_beta=combo["beta"], has_bias=combo["bias"], seed=H)
        out, s = run(lib, d, residual=combo["residual"])
        check(d, out, s)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("H", [1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 24, 31, 32, 33, 64, 127, 128, 129, 255, 256, 257, 500, 511, 512,
                               513, 1000, 1023, 1024, 1025, 2048, 2049, 4096, 4100, 8192, 8200, 12288, 16384])
def test_hidden_sizes(lib, dtype, H):
    rows = 19 if H <= 4096 else 5
    d = synth.sln_inputs((rows, H), None, dtype, has_beta=True, has_bias=True, seed=H)
    out, s = run(lib, d, residual=True)
    check(d, out, s)


@pytest.mark.parametrize("dtype,H", [("f32", 8), ("f32", 12), ("f16", 16), ("f16", 24), ("bf16", 16), ("bf16", 24)])
@pytest.mark.parametrize("skip_rows", [None, 7])
@pytest.mark.parametrize("simplified", [False, True])
def test_short_rows_one_thread(lib, dtype, H, skip_rows, simplified):
    # aligned rows of 2 or 3 fragments: one thread a row on the register kernel
    # (256 rows a CTA), with a broadcast skip, the residual output and the
    # statistics outputs
    rows = 256 * 5 + 37 if skip_rows is None else 7 * 187
    if skip_rows is None:
        d = synth.sln_inputs((rows, H), None, dtype, has_beta=not simplified, has_bias=True, seed=H + 9)
    else:
        d = synth.sln_inputs((rows // skip_rows, skip_rows, H), (1, skip_rows, H), dtype, has_beta=not simplified,
                             has_bias=True, seed=H + 9)
    out, s, mean, inv = run_ex(lib, d, simplified)
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                               simplified=simplified)
    assert_norm_close(out.reshape(-1, H), o["output"].reshape(-1, H), d["input"].dtype)
    assert_bit_exact(s.reshape(-1, H), oracle.skip_bias_sum(d["input"], d["skip"], d["bias"]).reshape(-1, H))
    np.testing.assert_allclose(mean.numpy().astype(np.float64).reshape(-1), o["mean"].reshape(-1), rtol=2e-5,
                               atol=2e-6)
    np.testing.assert_allclose(inv.numpy().astype(np.float64).reshape(-1), o["inv_std_dev"].reshape(-1), rtol=2e-5,
                               atol=0)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("H", [16385, 16392, 20000, 24576, 32768, 32776, 40000])
def test_long_rows(lib, dtype, H):
    # aligned rows up to 32768: 1024-thread register shapes; others and longer
    # rows: the three-pass kernel
    d = synth.sln_inputs((3, H), None, dtype, has_beta=True, has_bias=True, seed=H)
    out, s = run(lib, d, residual=True)
    check(d, out, s)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("beta,bias,res", [(False, False, False), (False, True, True), (True, False, True)])
def test_optional_inputs_superset(lib, dtype, beta, bias, res):
    d = synth.sln_inputs((4, 13, 96), (13, 96), dtype, has_beta=beta, has_bias=bias, seed=5)
    out, s = run(lib, d, residual=res)
    check(d, out, s)


@pytest.mark.parametrize("dtype,offs", [
    ("f16", {"input": 2}), ("f16", {"output": 6}), ("f16", {"gamma": 2, "sum": 2}),
    ("f32", {"skip": 4}), ("f32", {"input": 4, "output": 4, "sum": 8}), ("f32", {"bias": 12, "beta": 4}),
])
def test_misaligned_pointers(lib, dtype, offs):
    d = synth.sln_inputs((7, 256), None, dtype, has_beta=True, has_bias=True, seed=3)
    out, s = run(lib, d, residual=True, offsets=offs)
    check(d, out, s)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_in_place(lib, dtype):
    d = synth.sln_inputs((9, 1024), None, dtype, has_beta=True, has_bias=True, seed=9)
    x = d["input"].cuda()
    sk = d["skip"].cuda()
    lib.ep_skip_layer_norm(x, sk, d["gamma"].cuda(), d["beta"].cuda(), d["bias"].cuda(), d["epsilon"],
                           output=x, input_skip_bias_sum=sk)
    torch.cuda.synchronize()
    check(d, x.cpu(), sk.cpu())


def test_h1_gives_beta_exactly(lib):
    d = synth.sln_inputs((33, 1), None, "f32", has_beta=True, has_bias=False, seed=1)
    out, _ = run(lib, d)
    assert torch.equal(out.reshape(-1), d["beta"].expand(33))


def test_epsilon_zero_constant_row_is_nan(lib):
    # var = 0 and eps = 0: 0/0 -> NaN, as in the oracle
    x = torch.full((2, 8), 0.5)
    d = dict(input=x, skip=torch.zeros(2, 8), gamma=torch.ones(8), beta=None, bias=None, epsilon=0.0)
    out, _ = run(lib, d)
    assert torch.isnan(out).all()


def test_skip_broadcast_rows_bit_exact(lib):
    # skip row j is a spike of 1000 at column j; input 0.  Each output row is
    # one-hot-like and its residual equals its skip row exactly: a wrong skip
    # row would move the spike.
    S, H = 16, 64
    skip = torch.zeros(1, S, H)
    skip[0, torch.arange(S), torch.arange(S)] = 1000.0
    x = torch.zeros(4, S, H)
    d = dict(input=x, skip=skip, gamma=torch.ones(H), beta=torch.zeros(H), bias=None, epsilon=1e-12)
    out, s = run(lib, d, residual=True)
    want = skip.expand(4, S, H).numpy()
    assert_bit_exact(s, want.astype(np.float32))
    assert (out.argmax(dim=-1) == torch.arange(S).expand(4, S)).all()
    check(d, out, s)


def test_empty_rows_launch_nothing(lib):
    n0 = lib.kernel_launch_count()
    x = torch.empty(0, 7, 64, device="cuda")
    sk = torch.empty(0, 7, 64, device="cuda")
    g = torch.ones(64, device="cuda")
    out, _ = lib.ep_skip_layer_norm(x, sk, g, None, None)
    assert out.shape == x.shape and lib.kernel_launch_count() == n0


def test_launch_count_one_per_call(lib):
    d = synth.sln_inputs((8, 256), None, "f32", seed=0)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    n0 = lib.kernel_launch_count()
    lib.ep_skip_layer_norm(dev["input"], dev["skip"], dev["gamma"], dev["beta"], dev["bias"])
    assert lib.kernel_launch_count() == n0 + 1


def test_nondefault_stream(lib):
    d = synth.sln_inputs((64, 512), None, "f16", has_beta=True, has_bias=True, seed=2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        out, res = lib.ep_skip_layer_norm(dev["input"], dev["skip"], dev["gamma"], dev["beta"], dev["bias"],
                                          input_skip_bias_sum=True)
    s.synchronize()
    check(d, out.cpu(), res.cpu())


# ---------------------------------------------------------------------------
# the measured workloads
# ---------------------------------------------------------------------------

def test_workload_sln_f32_2x128x768(lib):
    d = synth.workload("sln_f32_2x128x768")
    out, _ = run(lib, d)
    check(d, out, None)   # every element


@pytest.mark.slow
@pytest.mark.parametrize("name", ["sln_f16_16384x4096_bias_residual", "sln_f32_32x2048x1024_bcast_skip"])
def test_workload_full_size_every_element(lib, name):
    # the whole output and residual against the oracle, in blocks of 2^22
    # elements to bound host memory
    d = synth.workload(name)
    out, s = run(lib, d, residual=d["residual"], guard=True)
    H = d["input"].shape[-1]
    R = d["input"].numel() // H
    y = out.reshape(R, H)
    res = s.reshape(R, H) if s is not None else None
    step = max(1, (1 << 22) // H)
    for r0 in range(0, R, step):
        rows = np.arange(r0, min(R, r0 + step))
        o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                                   rows=rows)["output"]
        assert_norm_close(y[r0:r0 + rows.size], o, d["input"].dtype)
        if res is not None:
            assert_bit_exact(res[r0:r0 + rows.size], oracle.skip_bias_sum(d["input"], d["skip"], d["bias"], rows=rows))


# ---------------------------------------------------------------------------
# many tiles per CTA: the shared-memory stage ring wraps many times; ragged
# last tile; a broadcast skip whose rows wrap inside a tile
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H,rows,skip_rows", [
    ("f32", 1024, 20001, None), ("f16", 4096, 6003, None), ("f32", 1024, 20000, 2000),
    ("f32", 768, 12007, 12007), ("f16", 2048, 9000, 3), ("f16", 512, 30001, 30001),
    ("f16", 32, 21000, 7), ("f32", 64, 9001, 9001), ("bf16", 128, 40000, 5),   # 64-row tiles
    ("f16", 12288, 600, 3), ("f32", 12288, 401, 401), ("f32", 16384, 300, 4),   # 1-row tiles; f32 in parts
])
def test_staged_many_tiles(lib, dtype, H, rows, skip_rows):
    if skip_rows is None or skip_rows == rows:
        d = synth.sln_inputs((rows, H), None, dtype, has_beta=True, has_bias=True, seed=rows)
    else:
        d = synth.sln_inputs((rows // skip_rows, skip_rows, H), (1, skip_rows, H), dtype, has_beta=True,
                             has_bias=False, seed=rows)
    out, s = run(lib, d, residual=True)
    sample = sorted(set(synth.sample_rows(rows, 1500)) | set(range(rows - 9, rows)))
    check(d, out, s, rows=sample)


# ---------------------------------------------------------------------------
# every row shape of the staged kernel: a group of TPR threads holds NV
# 16-byte fragments of a row.  Exact shapes (H = TPR*NV*VW) and ragged ones
# (the last fragment column partly idle), each over several tiles of 256/TPR
# rows with a partial last tile; and the sub-warp register shapes (a row of
# 1 to 16 fragments held by 4 to 16 threads, for rows that are not 16-byte
# aligned) over several CTAs.
# ---------------------------------------------------------------------------

_EXACT_SHAPES = ([(t, nv) for nv in (3, 4, 5, 7) for t in (4, 8, 16, 32, 64, 128, 256)]
                 + [(256, 6), (256, 8), (4, 2), (4, 1)])
_F32_PART_SHAPES = [(256, 12), (256, 16)]   # float32 rows staged in 3 and 4 parts
_RAGGED_NFRAG = [40, 100, 200, 300, 700, 1500]   # 16x4, 32x4, 64x4, 128x4, 256x4, 256x8 with idle lanes


def _shape_cases():
    out = []
    for dt, vw in (("f32", 4), ("f16", 8), ("bf16", 8)):
        out += [(dt, t * nv * vw) for t, nv in _EXACT_SHAPES]
        out += [(dt, nf * vw) for nf in _RAGGED_NFRAG]
    out += [("f32", t * nv * 4) for t, nv in _F32_PART_SHAPES]
    return out


@pytest.mark.parametrize("dtype,H", _shape_cases())
def test_staged_row_shapes(lib, dtype, H):
    rows = 451 if H <= 1024 else 115 if H <= 4096 else 37   # >= 7 tiles of up to 64, 16 or 2 rows
    d = synth.sln_inputs((rows, H), None, dtype, has_beta=True, has_bias=True, seed=H + rows)
    out, s = run(lib, d, residual=True)
    check(d, out, s)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("nfrag", [1, 2, 3, 4, 5, 8, 9, 16])
def test_subwarp_register_shapes(lib, dtype, nfrag):
    H = nfrag * (4 if dtype == "f32" else 8)
    rows = 64 * 5 + 17                             # several CTAs of 64, 32 or 16 rows
    d = synth.sln_inputs((rows, H), None, dtype, has_beta=True, has_bias=True, seed=nfrag)
    out, s = run(lib, d, residual=True)
    check(d, out, s)


# ---------------------------------------------------------------------------
# ep_skip_layer_norm_ex: the RMS (simplified) form and the per-row statistics
# ---------------------------------------------------------------------------

def run_ex(lib, d, simplified, residual=True):
    dev = {k: (d[k].cuda() if d[k] is not None else None) for k in ("input", "skip", "gamma", "beta", "bias")}
    x = d["input"]
    rows = x.numel() // x.shape[-1]
    go = Guarded(x.shape, x.dtype)
    gs = Guarded(x.shape, x.dtype) if residual else None
    gm = Guarded((rows,), torch.float32)
    gi = Guarded((rows,), torch.float32)
    lib.ep_skip_layer_norm_ex(dev["input"], dev["skip"], dev["gamma"], dev["beta"], dev["bias"], d["epsilon"],
                              simplified=simplified, output=go.tensor,
                              input_skip_bias_sum=gs.tensor if gs else None,
                              mean=gm.tensor, inv_std_dev=gi.tensor)
    torch.cuda.synchronize()
    for gd in (go, gs, gm, gi):
        if gd is not None:
            gd.check()
    return go.tensor.cpu(), (gs.tensor.cpu() if gs else None), gm.tensor.cpu(), gi.tensor.cpu()


@pytest.mark.parametrize("simplified", [False, True])
@pytest.mark.parametrize("dtype,shape,skip_shape,beta,bias", [
    ("f32", (19, 768), None, False, True),        # staged path
    ("f16", (7, 4096), None, True, True),         # staged path, exact rows
    ("f32", (5, 771), None, False, False),        # register path (H % 4 != 0)
    ("f16", (3, 20000), None, False, True),       # three-pass path
    ("f32", (4, 11, 1024), (11, 1024), True, False),  # broadcast skip
])
def test_ex_simplified_and_statistics(lib, simplified, dtype, shape, skip_shape, beta, bias):
    d = synth.sln_inputs(shape, skip_shape, dtype, has_beta=beta, has_bias=bias, seed=shape[-1])
    out, s, mean, inv = run_ex(lib, d, simplified)
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                               simplified=simplified)
    H = shape[-1]
    assert_norm_close(out.reshape(-1, H), o["output"], d["input"].dtype)
    assert_bit_exact(s.reshape(-1, H), oracle.skip_bias_sum(d["input"], d["skip"], d["bias"]))
    np.testing.assert_allclose(mean.numpy().astype(np.float64), o["mean"], rtol=2e-5, atol=2e-6)
    np.testing.assert_allclose(inv.numpy().astype(np.float64), o["inv_std_dev"], rtol=2e-5, atol=0)
    if simplified:
        assert (mean == 0).all()


@pytest.mark.parametrize("dtype,rows,H", [
    ("f32", 320000, 771),     # register kernel: two 128-thread rows per CTA, about two rounds of the grid
    ("f16", 20000, 20000),    # 1024-thread register rows, more rows than CTAs
    ("f16", 6000, 16401),     # three-pass kernel, more rows than CTAs
])
def test_ex_simplified_many_rows_per_cta(lib, dtype, rows, H):
    # the RMS form has one reduction per row; consecutive rows of a CTA must
    # not share its shared-memory buffer.  Inputs are drawn on the device.
    x = synth.device_normal((rows, H), dtype, seed=rows)
    sk = synth.device_normal((rows, H), dtype, seed=rows + 1)
    g = (synth.device_normal((H,), dtype, seed=rows + 2, std=0.1).float() + 1.0).to(x.dtype)
    bt = synth.device_normal((H,), dtype, seed=rows + 3, std=0.1)
    out = torch.empty_like(x)
    inv = torch.empty(rows, dtype=torch.float32, device="cuda")
    lib.ep_skip_layer_norm_ex(x, sk, g, bt, None, 1e-5, simplified=True, output=out, inv_std_dev=inv)
    torch.cuda.synchronize()
    sample = torch.tensor(sorted(set(synth.sample_rows(rows, 300)) | set(range(rows - 5, rows))))
    o = oracle.skip_layer_norm(x[sample.cuda()].cpu(), sk[sample.cuda()].cpu(), g.cpu(), bt.cpu(), None, 1e-5,
                               simplified=True)
    assert_norm_close(out[sample.cuda()].cpu(), o["output"], x.dtype)
    np.testing.assert_allclose(inv[sample.cuda()].cpu().numpy().astype(np.float64), o["inv_std_dev"],
                               rtol=2e-5, atol=0)
    del x, sk, out
    torch.cuda.empty_cache()


def test_ex_default_matches_plain_entry_point(lib):
    d = synth.sln_inputs((33, 1024), None, "f16", has_beta=True, has_bias=True, seed=4)
    a, s_a = run(lib, d, residual=True)
    b, s_b, _, _ = run_ex(lib, d, simplified=False)
    assert torch.equal(a, b) and torch.equal(s_a, s_b)


# ---------------------------------------------------------------------------
# rows of 16385-32768 elements on the staged kernel with more than 256
# consumer threads, the row staged in parts (16-bit rows of 18432-30720, in
# multiples of 2048, on H/32 threads of 4 fragments; 16-bit rows of 32768 and
# float32 rows of multiples of 2048 on 512 threads); many rows so that tiles
# are taken over by running CTAs and the stage ring wraps
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H", [("f16", 18432), ("f16", 20480), ("f16", 22528), ("f16", 24576),
                                     ("f16", 26624), ("f16", 28672), ("f16", 30720), ("f16", 32768),
                                     ("bf16", 20480), ("bf16", 28672), ("bf16", 32768),
                                     ("f32", 18432), ("f32", 20480), ("f32", 22528), ("f32", 24576),
                                     ("f32", 26624), ("f32", 28672), ("f32", 30720), ("f32", 32768)])
def test_wide_rows_staged(lib, dtype, H):
    rows = 331
    d = synth.sln_inputs((rows, H), None, dtype, has_beta=True, has_bias=True, seed=H)
    out, s = run(lib, d, residual=True)
    check(d, out, s)


def test_wide_rows_stage_reuse_repeated(lib):
    # float32 rows of 28672: one row fills the four 56 KB stages, so every
    # stage is refilled with the next row's part as soon as the consumers hand
    # it back.  Without a proxy fence between the consumers' reads and that
    # refill, about one call in five had a row whose last fragment held the
    # next row's data; eight calls must all match the oracle
    H, rows = 28672, 331
    d = synth.sln_inputs((rows, H), None, "f32", has_beta=True, has_bias=True, seed=H + 5)
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"])
    want_sum = oracle.skip_bias_sum(d["input"], d["skip"], d["bias"])
    for _ in range(8):
        out, s = run(lib, d, residual=True)
        assert_norm_close(out.reshape(-1, H), o["output"].reshape(-1, H), torch.float32)
        assert_bit_exact(s.reshape(-1, H), want_sum.reshape(-1, H))


@pytest.mark.parametrize("dtype,H,beta,bias,res,skip_rows", [
    ("f16", 32768, False, False, False, None), ("f32", 20480, True, False, False, 5),
    ("bf16", 24576, False, True, True, 7), ("f32", 32768, True, True, True, None),
    ("f16", 20480, False, True, False, 7), ("bf16", 30720, True, False, True, None),
])
def test_wide_rows_optional_inputs_and_broadcast_skip(lib, dtype, H, beta, bias, res, skip_rows):
    rows = 161
    if skip_rows is None:
        d = synth.sln_inputs((rows, H), None, dtype, has_beta=beta, has_bias=bias, seed=H + 1)
    else:
        d = synth.sln_inputs((rows // skip_rows, skip_rows, H), (1, skip_rows, H), dtype, has_beta=beta,
                             has_bias=bias, seed=H + 1)
    out, s = run(lib, d, residual=res)
    check(d, out, s)


@pytest.mark.parametrize("simplified", [False, True])
@pytest.mark.parametrize("dtype,H", [("f16", 28672), ("f32", 26624)])
def test_wide_rows_ex_statistics(lib, simplified, dtype, H):
    d = synth.sln_inputs((97, H), None, dtype, has_beta=not simplified, has_bias=True, seed=H + 2)
    out, s, mean, inv = run_ex(lib, d, simplified)
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                               simplified=simplified)
    assert_norm_close(out.reshape(-1, H), o["output"], d["input"].dtype)
    assert_bit_exact(s.reshape(-1, H), oracle.skip_bias_sum(d["input"], d["skip"], d["bias"]))
    np.testing.assert_allclose(mean.numpy().astype(np.float64), o["mean"], rtol=2e-5, atol=2e-6)
    np.testing.assert_allclose(inv.numpy().astype(np.float64), o["inv_std_dev"], rtol=2e-5, atol=0)
