"""BiasSoftmax: CUDA path (through the C ABI) vs the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gen import synth
from tests._helpers import Guarded, assert_norm_close, offset_copy, to_np64

pytestmark = pytest.mark.gpu


def run(lib, data, bias, axis, inner, offsets=None, guard=True, workspace=None):
    offsets = offsets or {}
    keep = []

    def dev(name, t):
        if name in offsets:
            raw, v = offset_copy(t, offsets[name])
            keep.append(raw)
            return v
        return t.cuda()

    g = Guarded(data.shape, data.dtype, offset_bytes=offsets.get("output", 0))
    lib.ep_bias_softmax(dev("data", data), dev("bias", bias), axis=axis, is_inner_broadcast=inner,
                        output=g.tensor, workspace=workspace)
    torch.cuda.synchronize()
    if guard:
        g.check()
    return g.tensor.cpu()


def check(data, bias, axis, inner, out, rows=None):
    o = oracle.bias_softmax(data, bias, axis=axis, is_inner_broadcast=inner, rows=rows)
    dims = oracle.bias_softmax_dims(tuple(data.shape), bias.numel(), axis)
    got = out.reshape(dims["batch"], dims["block"])
    if rows is not None:
        got = got[rows]
    return assert_norm_close(got, o, data.dtype)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("cols", [1, 2, 3, 7, 8, 9, 31, 32, 33, 64, 100, 255, 256, 257, 512, 513, 1000, 1024,
                                  2047, 4096, 4100, 8192, 16384])
def test_row_path_sizes(lib, dtype, cols):
    rows = 24 if cols <= 4096 else 6
    d = synth.bias_softmax_inputs((rows, cols), (3, cols), dtype, data_std=3.0, seed=cols)
    for inner in (0, 1):
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("cols", [16385, 20000, 65536, 65537, 100003, 262144])
def test_split_path_sizes(lib, dtype, cols):
    rows = 4
    d = synth.bias_softmax_inputs((rows, cols), (2, cols), dtype, data_std=2.0, seed=cols)
    assert lib.ep_bias_softmax_workspace_size(d["data"].dtype, d["data"].shape, 1) > 0
    for inner in (0, 1):
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)
        np.testing.assert_allclose(to_np64(out).sum(axis=1), 1.0, atol=5e-3 if dtype == "f16" else 1e-4)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("axis,bias_shape,inner", [
    (3, (2, 1, 1, 40), 1), (3, (1, 3, 4, 40), 0), (2, (2, 1, 4, 40), 1), (2, (1, 1, 4, 40), 0),
    (1, (1, 3, 4, 40), 0), (-1, (1, 1, 1, 40), 1), (-3, (2, 3, 4, 40), 0), (0, (2, 3, 4, 40), 1),
])
def test_axes_and_bias_forms(lib, dtype, axis, bias_shape, inner):
    d = synth.bias_softmax_inputs((2, 3, 4, 40), bias_shape, dtype, data_std=2.0, seed=11)
    out = run(lib, d["data"], d["bias"], axis, inner)
    check(d["data"], d["bias"], axis, inner, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("inner", [0, 1])
@pytest.mark.parametrize("rows,cols,bias_rows", [(48, 64, 8), (48, 64, 48), (64, 512, 16), (12, 20000, 4)])
def test_bias_row_map_bit_exact(lib, dtype, inner, rows, cols, bias_rows):
    # data = 0; bias row k is MASKED except 0 at column k.  The output row is
    # then exactly one-hot at its bias row's column (exp(0)=1, exp(-10000)=0).
    data = torch.zeros(rows, cols, dtype=dtype)
    bias = torch.full((bias_rows, cols), synth.MASKED, dtype=dtype)
    bias[torch.arange(bias_rows), torch.arange(bias_rows)] = 0.0
    out = run(lib, data, bias, 1, inner)
    br = oracle.bias_row_of(np.arange(rows), bias_rows, rows // bias_rows, inner)
    want = torch.zeros(rows, cols, dtype=dtype)
    want[torch.arange(rows), torch.from_numpy(br)] = 1.0
    assert torch.equal(out, want)


def test_causal_mask_rows(lib):
    d = synth.bias_softmax_inputs((2, 4, 64, 64), (2, 64, 64), "f16", data_std=4.0, seed=1, causal=True)
    out = run(lib, d["data"], d["bias"], 3, 1)
    check(d["data"], d["bias"], 3, 1, out)
    # masked keys get exactly 0 (exp(-10000 - m) underflows)
    o = out.reshape(-1, 64)
    br = oracle.bias_row_of(np.arange(o.shape[0]), 128, 4, 1)  # 512 rows, 128 bias rows
    for r in range(0, o.shape[0], 37):
        q = br[r] % 64
        assert (o[r, q + 1:] == 0).all()


@pytest.mark.parametrize("dtype,offs", [("f16", {"data": 2}), ("f16", {"output": 2, "bias": 4}),
                                        ("f32", {"data": 4, "output": 4}), ("f32", {"bias": 8})])
@pytest.mark.parametrize("cols", [512, 30000])
def test_misaligned_pointers(lib, dtype, offs, cols):
    d = synth.bias_softmax_inputs((6, cols), (3, cols), dtype, data_std=2.0, seed=4)
    out = run(lib, d["data"], d["bias"], 1, 1, offsets=offs)
    check(d["data"], d["bias"], 1, 1, out)


@pytest.mark.parametrize("cols", [512, 70000])
def test_in_place(lib, cols):
    d = synth.bias_softmax_inputs((8, cols), (2, cols), "f32", data_std=2.0, seed=8)
    x = d["data"].cuda()
    lib.ep_bias_softmax(x, d["bias"].cuda(), axis=1, is_inner_broadcast=0, output=x)
    torch.cuda.synchronize()
    check(d["data"], d["bias"], 1, 0, x.cpu())


def test_large_equal_logits_and_neg_inf(lib):
    data = torch.tensor([[60000.0, 60000.0, -float("inf"), 0.0]], dtype=torch.float16)
    bias = torch.zeros(1, 4, dtype=torch.float16)
    out = run(lib, data, bias, 1, 0)
    assert out.tolist() == [[0.5, 0.5, 0.0, 0.0]]


def test_all_masked_row_is_nan(lib):
    data = torch.full((2, 40000), -float("inf"))
    bias = torch.zeros(1, 40000)
    out = run(lib, data, bias, 1, 0)
    assert torch.isnan(out).all()
    data = torch.full((2, 100), -float("inf"))
    out = run(lib, data, torch.zeros(1, 100), 1, 0)
    assert torch.isnan(out).all()


def test_empty_launches_nothing(lib):
    n0 = lib.kernel_launch_count()
    x = torch.empty(0, 16, device="cuda")
    b = torch.empty(0, device="cuda")
    lib.ep_bias_softmax(x, b, axis=1, is_inner_broadcast=1)
    assert lib.kernel_launch_count() == n0


def test_workspace_too_small_is_rejected(lib):
    x = torch.zeros(2, 70000, device="cuda")
    b = torch.zeros(70000, device="cuda")
    need = lib.ep_bias_softmax_workspace_size(torch.float32, (2, 70000), 1)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.EpError) as e:
        lib.ep_bias_softmax(x, b, axis=1, is_inner_broadcast=0, workspace=ws)
    assert e.value.status == lib.EP_ERR_WORKSPACE


# ---------------------------------------------------------------------------
# the measured workloads
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_workload_attention_f16_every_element(lib):
    # all 262,144 rows against the oracle, in blocks of 2^22 elements
    d = synth.workload("bias_softmax_f16_32x16x512x512_causal")
    out = run(lib, d["data"], d["bias"], d["axis"], d["is_inner_broadcast"])
    y = out.reshape(-1, 512)
    R = y.shape[0]
    step = (1 << 22) // 512
    for r0 in range(0, R, step):
        rows = np.arange(r0, min(R, r0 + step))
        o = oracle.bias_softmax(d["data"], d["bias"], axis=d["axis"], is_inner_broadcast=d["is_inner_broadcast"],
                                rows=rows)
        assert_norm_close(y[r0:r0 + rows.size], o, torch.float16)


@pytest.mark.slow
@pytest.mark.parametrize("name,inner", [("bias_softmax_f32_64x262144_cyclic", 0),
                                        ("bias_softmax_f32_8x1048576", 0),
                                        ("bias_softmax_f32_8x1048576", 1)])
def test_workload_long_rows_full(lib, name, inner):
    d = synth.workload(name)
    out = run(lib, d["data"], d["bias"], d["axis"], inner)
    check(d["data"], d["bias"], d["axis"], inner, out)


# ---------------------------------------------------------------------------
# many tiles per CTA on the shared-memory-staged row kernel, with every way a
# tile's bias rows can be laid out (inner groups spanning tiles, outer maps
# with all bias rows in one tile, and outer maps that wrap inside a tile)
# ---------------------------------------------------------------------------

# every row shape of the staged kernel: a group of TPR threads holds NV
# 16-byte fragments of a row.  Exact shapes (cols = TPR*NV*VW) and ragged ones
# (the last fragment column partly idle), several tiles of 256/TPR rows with a
# partial last tile, bias broadcast both ways; and the sub-warp register shapes
# (rows of 1 to 16 fragments held by 4 to 16 threads) over several CTAs.
_EXACT_SHAPES = [(t, nv) for nv in (4, 5, 6, 7) for t in (4, 8, 16, 32, 64, 128, 256)] + [(256, 8), (4, 3)]
_RAGGED_NFRAG = [40, 100, 200, 300, 700, 1500]   # 16x4, 32x4, 64x4, 128x4, 256x4, 256x8 with idle lanes


def _shape_cases():
    out = []
    for dt, vw in (("f32", 4), ("f16", 8), ("bf16", 8)):
        out += [(dt, t * nv * vw) for t, nv in _EXACT_SHAPES]
        out += [(dt, nf * vw) for nf in _RAGGED_NFRAG]
    out += [("f32", 256 * 12 * 4), ("f32", 256 * 16 * 4)]   # float32 rows staged in 3 and 4 parts
    return out


@pytest.mark.parametrize("dtype,cols", _shape_cases())
def test_staged_row_shapes(lib, dtype, cols):
    rows, bias_rows = (455, 5) if cols <= 1024 else (115, 5) if cols <= 4096 else (40, 5)  # >= 7 tiles of 64, 16 or 2 rows
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=cols)
    for inner in (0, 1):
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("nfrag", [2, 3, 4, 5, 8, 9, 16])
def test_subwarp_register_shapes(lib, dtype, nfrag):
    cols = nfrag * (4 if dtype == "f32" else 8)
    rows, bias_rows = 64 * 5 + 16, 4               # several CTAs of 64, 32 or 16 rows
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=nfrag)
    for inner in (0, 1):
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)


@pytest.mark.parametrize("dtype,rows,cols,bias_rows,inner", [
    ("f16", 80003, 512, 11429, 1), ("f16", 80003, 512, 11429, 0), ("f16", 80003, 512, 7, 0),
    ("f16", 80003, 512, 7, 1), ("f32", 40000, 256, 40000, 0), ("f32", 30000, 1024, 3, 1),
    ("f16", 10000, 4096, 10, 0), ("f32", 9001, 2048, 9001, 1),
    ("f16", 40000, 128, 8, 0), ("f16", 40000, 96, 2500, 1), ("f32", 30000, 64, 30000, 0),   # 64-row tiles
])
def test_staged_many_tiles(lib, dtype, rows, cols, bias_rows, inner):
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=rows + bias_rows)
    out = run(lib, d["data"], d["bias"], 1, inner)
    sample = sorted(set(synth.sample_rows(rows, 1500)) | set(range(rows - 17, rows)))
    check(d["data"], d["bias"], 1, inner, out, rows=sample)


@pytest.mark.parametrize("dtype,rows,cols,bias_rows,inner", [
    ("f32", 160, 262144, 4, 1), ("f32", 160, 262144, 4, 0), ("f16", 96, 600000, 3, 0), ("f32", 5, 16388, 5, 1),
])
def test_split_path_several_windows(lib, dtype, rows, cols, bias_rows, inner):
    # more rows than one L2-sized window holds: the stats/normalize pair runs per
    # window; chunk statistics of every row must land in the right place
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=2.0, seed=rows)
    out = run(lib, d["data"], d["bias"], 1, inner)
    sample = sorted(set(synth.sample_rows(rows, 12)) | {rows - 1})
    check(d["data"], d["bias"], 1, inner, out, rows=sample)
    np.testing.assert_allclose(to_np64(out).sum(axis=1), 1.0, atol=5e-3 if dtype == "f16" else 1e-4)


# Split rows whose chunk ranges cross rows at odd places, and rows of 2.5 M
# and 4 M elements (over a thousand chunks each, spread over every CTA).
@pytest.mark.parametrize("dtype,rows,cols,bias_rows,inner", [
    ("f32", 37, 300000, 37, 0), ("f16", 29, 600000, 1, 1), ("bf16", 23, 333336, 23, 1),
    ("f32", 2, (1 << 22) + 8, 1, 0), ("f16", 2, (1 << 22) + 8, 2, 1), ("f32", 1, 2490368, 1, 0),
])
def test_split_odd_ranges_and_very_long_rows(lib, dtype, rows, cols, bias_rows, inner):
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=2.0, seed=rows + cols)
    out = run(lib, d["data"], d["bias"], 1, inner)
    sample = sorted(set(synth.sample_rows(rows, 6)) | {0, rows - 1})
    check(d["data"], d["bias"], 1, inner, out, rows=sample)
    # row sums: float16 outputs near 1/cols are subnormal (step 2^-24), so each
    # may be off by 2^-25 in absolute terms
    atol = 1e-4 if dtype == "f32" else 5e-3 + (cols * 2.0 ** -25 if dtype == "f16" else 0.0)
    np.testing.assert_allclose(to_np64(out).sum(axis=1), 1.0, atol=atol)


@pytest.mark.parametrize("dtype,cols", [("f32", 40000), ("f16", 70000), ("bf16", 70000)])
def test_split_ranges_cross_rows_with_masked_chunks(lib, dtype, cols):
    # more chunks than one wave of CTAs, so a CTA's range of chunks runs from the
    # tail of one row into the head of the next; whole chunks masked to -inf at
    # the start, the end and the middle of rows, and one fully masked row
    rows = 200
    d = synth.bias_softmax_inputs((rows, cols), (rows, cols), dtype, data_std=2.0, seed=cols)
    data = d["data"].clone()
    chunk = 4096 if dtype == "f32" else 8192
    for r in range(0, rows, 3):
        data[r, :chunk + 7] = -float("inf")
    for r in range(1, rows, 5):
        data[r, cols - chunk - 3:] = -float("inf")
    for r in range(2, rows, 7):
        data[r, chunk:2 * chunk] = -float("inf")
    data[rows // 2, :] = -float("inf")
    out = run(lib, data, d["bias"], 1, 0)
    live = [r for r in range(rows) if r != rows // 2]
    check(data, d["bias"], 1, 0, out, rows=live)
    assert torch.isnan(out[rows // 2]).all()


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("cols", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("inner", [0, 1])
@pytest.mark.parametrize("misaligned", [False, True])
def test_packed_rows(lib, dtype, cols, inner, misaligned):
    # rows of <= 8 elements: one thread per row (aligned rows of exactly 8
    # elements: the register kernel's one-thread rows; a data pointer one
    # element off sends them to the packed kernel)
    rows = 70007 if inner else 70000
    bias_rows = 7 if inner else 16
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=cols)
    offs = {"data": d["data"].element_size()} if misaligned else None
    out = run(lib, d["data"], d["bias"], 1, inner, offsets=offs)
    sample = sorted(set(synth.sample_rows(rows, 3000)) | set(range(rows - 5, rows)))
    check(d["data"], d["bias"], 1, inner, out, rows=sample)


def test_packed_rows_bias_map_bit_exact(lib):
    rows, cols, bias_rows = 4096, 8, 8
    for inner in (0, 1):
        data = torch.zeros(rows, cols)
        bias = torch.full((bias_rows, cols), synth.MASKED)
        bias[torch.arange(bias_rows), torch.arange(bias_rows)] = 0.0
        out = run(lib, data, bias, 1, inner)
        br = oracle.bias_row_of(np.arange(rows), bias_rows, rows // bias_rows, inner)
        want = torch.zeros(rows, cols)
        want[torch.arange(rows), torch.from_numpy(br)] = 1.0
        assert torch.equal(out, want)


# ---------------------------------------------------------------------------
# rows of 16385-32768 columns on the staged row kernel with more than 256
# consumer threads, the row and its bias row staged in parts: 16-bit rows of
# 18432-30720 (multiples of 2048) on nfrag/4 threads of 4 fragments, 16-bit
# rows of 32768 and float32 rows of multiples of 2048 on 512 threads
# ---------------------------------------------------------------------------

_WIDE = [("f16", 18432), ("f16", 20480), ("f16", 22528), ("f16", 24576), ("f16", 26624), ("f16", 28672),
         ("f16", 30720), ("f16", 32768), ("bf16", 20480), ("bf16", 24576), ("bf16", 30720), ("bf16", 32768),
         ("f32", 18432), ("f32", 20480), ("f32", 22528), ("f32", 24576), ("f32", 26624), ("f32", 28672),
         ("f32", 30720), ("f32", 32768)]


@pytest.mark.parametrize("dtype,cols", _WIDE)
def test_wide_rows_staged(lib, dtype, cols):
    rows, bias_rows = 301, 7
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=2.0, seed=cols)
    for inner in (0, 1):
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)


@pytest.mark.parametrize("dtype,cols", [("f32", 32768), ("f16", 20480)])
def test_wide_rows_stage_reuse_repeated(lib, dtype, cols):
    # stages refilled as soon as the consumers hand them back (see the
    # SkipLayerNorm test of the same name): eight calls must all match
    rows, bias_rows = 258, 3
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=2.0, seed=cols + 3)
    o = oracle.bias_softmax(d["data"], d["bias"], axis=1, is_inner_broadcast=0)
    for _ in range(8):
        out = run(lib, d["data"], d["bias"], 1, 0)
        assert_norm_close(out.reshape(rows, cols), o, d["data"].dtype)


@pytest.mark.parametrize("dtype,cols", [("f16", 32768), ("f16", 20480), ("bf16", 28672), ("f32", 20480)])
def test_wide_rows_masked_and_in_place(lib, dtype, cols):
    rows = 40
    d = synth.bias_softmax_inputs((rows, cols), (rows, cols), dtype, data_std=2.0, seed=cols + 1)
    data = d["data"].clone()
    for r in range(0, rows, 3):
        data[r, :cols // 3] = -float("inf")          # whole parts masked
    for r in range(1, rows, 5):
        data[r, cols - 4097:] = -float("inf")
    data[rows // 2, :] = -float("inf")               # a fully masked row: NaN
    out = run(lib, data, d["bias"], 1, 0)
    live = [r for r in range(rows) if r != rows // 2]
    check(data, d["bias"], 1, 0, out, rows=live)
    assert torch.isnan(out[rows // 2]).all()
    x = data.cuda()
    lib.ep_bias_softmax(x, d["bias"].cuda(), axis=1, is_inner_broadcast=0, output=x)
    torch.cuda.synchronize()
    assert torch.equal(x.cpu()[live], out[live])


# ---------------------------------------------------------------------------
# short rows (2 to 11 fragments, the register kernel's row groups of 4 to 16
# threads): many CTAs, every bias layout, aligned and misaligned
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("nfrag", [2, 3, 4, 5, 6, 7, 8, 9, 10, 11])
def test_short_rows_every_bias_layout(lib, dtype, nfrag):
    cols = nfrag * (4 if dtype == "f32" else 8)
    rows = 256 * 5 + 37
    for bias_rows, inner in ((3, 0), (rows, 0), (rows // 16 + 1, 1) if rows % (rows // 16 + 1) == 0 else (1, 1),
                             (1, 0)):
        if rows % bias_rows:
            continue
        d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=cols + bias_rows)
        out = run(lib, d["data"], d["bias"], 1, inner)
        check(d["data"], d["bias"], 1, inner, out)


@pytest.mark.parametrize("dtype,cols,bias_rows,inner", [("f16", 64, 1317, 0), ("f16", 32, 3, 1), ("f32", 32, 1, 0),
                                                        ("f32", 24, 1317, 1), ("bf16", 88, 1317, 1)])
def test_short_rows_bias_map_and_misaligned(lib, dtype, cols, bias_rows, inner):
    rows = 1317
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), dtype, data_std=3.0, seed=cols + 5)
    out = run(lib, d["data"], d["bias"], 1, inner)
    check(d["data"], d["bias"], 1, inner, out)
    es = 4 if dtype == "f32" else 2
    out2 = run(lib, d["data"], d["bias"], 1, inner, offsets={"data": es, "output": es})   # scalar fragments
    check(d["data"], d["bias"], 1, inner, out2)
    # one-hot bias rows: the output row is exactly one-hot at its bias row's column
    n = min(cols, bias_rows)
    data = torch.zeros(rows, cols, dtype=d["data"].dtype)
    bias = torch.full((bias_rows, cols), synth.MASKED, dtype=d["data"].dtype)
    bias[torch.arange(bias_rows), torch.arange(bias_rows) % cols] = 0.0
    got = run(lib, data, bias, 1, inner)
    br = oracle.bias_row_of(np.arange(rows), bias_rows, rows // bias_rows, inner)
    want = torch.zeros(rows, cols, dtype=data.dtype)
    want[torch.arange(rows), torch.from_numpy(br % cols)] = 1.0
    assert torch.equal(got, want), n
