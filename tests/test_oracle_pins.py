"""Pins for the CPU oracle: checks against things other than the oracle itself.

Closed forms worked by hand, invariants that hold by the mathematics, special
cases that reduce to a library routine (torch float64 layer_norm / rms_norm /
softmax), exact rational brute force on tiny inputs, and arbitrary-precision
evaluation (mpmath).  Each check is chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, sample
instead of population variance, the wrong summation order for the residual)
fails at least one of them; ``test_oracle_mutations.py`` plants such slips and
confirms it.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(7)


# ---------------------------------------------------------------------------
# attribute defaults (values the op definitions print)
# ---------------------------------------------------------------------------

def test_defaults_match_manifests():
    with open(os.path.join(GOLDEN, "op_attribute_defaults.json")) as f:
        g = json.load(f)
    assert oracle.DEFAULT_ALPHA == g["QuickGelu.alpha"]["value"]
    assert oracle.DEFAULT_EPSILON == g["SkipLayerNormalization.epsilon"]["value"]
    assert oracle.DEFAULT_AXIS == g["BiasSoftmax.axis"]["value"]
    # the printed epsilon is exactly float32(1e-12)
    assert float(np.float32(1e-12)) == g["SkipLayerNormalization.epsilon"]["value"]


# ---------------------------------------------------------------------------
# SkipLayerNormalization
# ---------------------------------------------------------------------------

def _row(vals, dtype=np.float32):
    return np.asarray([vals], dtype=dtype)


def test_sln_hand_worked_row():
    # s = [1,2,3,4]: mu = 5/2, population var = (9+1+1+9)/16 = 5/4,
    # n_i = (s_i - 5/2) / sqrt(5/4) = (2 s_i - 5) / sqrt(5).
    x = _row([1, 2, 3, 4])
    r = oracle.skip_layer_norm(x, np.zeros_like(x), np.ones(4, np.float32), None, None, epsilon=0.0)
    want = np.array([-3, -1, 1, 3]) / math.sqrt(5)
    np.testing.assert_allclose(r["output"][0], want, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["mean"], [2.5], rtol=0, atol=0)
    np.testing.assert_allclose(r["inv_std_dev"], [1 / math.sqrt(1.25)], rtol=1e-15)
    # the same row split between input and skip gives the same result
    r2 = oracle.skip_layer_norm(_row([0, 2, 1, 4]), _row([1, 0, 2, 0]), np.ones(4, np.float32), epsilon=0.0)
    np.testing.assert_allclose(r2["output"][0], want, rtol=0, atol=1e-15)


def test_sln_epsilon_closed_form():
    # eps = 1 (exact in float32): sqrt(5/4 + 1) = 3/2, n = [-1, -1/3, 1/3, 1].
    x = _row([1, 2, 3, 4])
    r = oracle.skip_layer_norm(x, np.zeros_like(x), np.ones(4, np.float32), epsilon=1.0)
    np.testing.assert_allclose(r["output"][0], [-1, -1 / 3, 1 / 3, 1], rtol=0, atol=1e-15)


def test_sln_epsilon_is_float32():
    # eps = 0.1 is read as float32(0.1), not 0.1
    x = _row([1, 2, 3, 4])
    r = oracle.skip_layer_norm(x, np.zeros_like(x), np.ones(4, np.float32), epsilon=0.1)
    e32 = float(np.float32(0.1))
    want = (np.array([1, 2, 3, 4]) - 2.5) / math.sqrt(1.25 + e32)
    np.testing.assert_allclose(r["output"][0], want, rtol=0, atol=1e-15)
    assert abs(r["output"][0][0] - (-1.5 / math.sqrt(1.35))) > 1e-10


def test_sln_affine_columns():
    # gamma and beta act per column: y_j = n_j * gamma_j + beta_j
    x = _row([1, 2, 3, 4])
    g = np.array([1, 2, 3, 4], np.float32)
    b = np.array([10, 20, 30, 40], np.float32)
    r = oracle.skip_layer_norm(x, np.zeros_like(x), g, b, epsilon=0.0)
    n = np.array([-3, -1, 1, 3]) / math.sqrt(5)
    np.testing.assert_allclose(r["output"][0], n * [1, 2, 3, 4] + [10, 20, 30, 40], rtol=0, atol=1e-13)


def test_sln_h1_gives_beta():
    x = rng.standard_normal((5, 1)).astype(np.float32)
    sk = rng.standard_normal((5, 1)).astype(np.float32)
    beta = np.array([0.375], np.float32)
    r = oracle.skip_layer_norm(x, sk, np.array([1.7], np.float32), beta)
    assert np.all(r["output"] == 0.375)


def test_sln_invariants_before_affine():
    # gamma = 1, no beta: sum(n) = 0 and mean(n^2) = var / (var + eps)
    H = 257
    x = rng.standard_normal((16, H)).astype(np.float32)
    sk = rng.standard_normal((16, H)).astype(np.float32)
    eps = 1e-3
    r = oracle.skip_layer_norm(x, sk, np.ones(H, np.float32), None, epsilon=eps)
    n = r["output"]
    s = x.astype(np.float64) + sk.astype(np.float64)
    var = np.var(s, axis=1)
    e32 = float(np.float32(eps))
    np.testing.assert_allclose(n.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((n * n).mean(axis=1), var / (var + e32), rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_sln_matches_torch_layer_norm(dtype):
    H = 96
    x = rng.standard_normal((7, H)).astype(dtype)
    sk = rng.standard_normal((7, H)).astype(dtype)
    g = rng.uniform(0.5, 1.5, H).astype(dtype)
    b = (0.1 * rng.standard_normal(H)).astype(dtype)
    bias = (0.1 * rng.standard_normal(H)).astype(dtype)
    eps = 1e-5
    r = oracle.skip_layer_norm(x, sk, g, b, bias, epsilon=eps)
    s = torch.from_numpy(x).double() + torch.from_numpy(sk).double() + torch.from_numpy(bias).double()
    ref = torch.nn.functional.layer_norm(s, (H,), torch.from_numpy(g).double(),
                                         torch.from_numpy(b).double(), float(np.float32(eps)))
    np.testing.assert_allclose(r["output"], ref.numpy(), rtol=0, atol=1e-13)


def test_sln_simplified_matches_torch_rms_norm():
    H = 64
    x = rng.standard_normal((5, H)).astype(np.float32)
    sk = rng.standard_normal((5, H)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    eps = 1e-6
    r = oracle.skip_layer_norm(x, sk, g, None, None, epsilon=eps, simplified=True)
    s = torch.from_numpy(x).double() + torch.from_numpy(sk).double()
    ref = torch.nn.functional.rms_norm(s, (H,), torch.from_numpy(g).double(), float(np.float32(eps)))
    np.testing.assert_allclose(r["output"], ref.numpy(), rtol=0, atol=1e-13)
    # hand-worked: [1,2,3,4] -> mean square 30/4, n = s / sqrt(7.5)
    x1 = _row([1, 2, 3, 4])
    r1 = oracle.skip_layer_norm(x1, np.zeros_like(x1), np.ones(4, np.float32), epsilon=0.0, simplified=True)
    np.testing.assert_allclose(r1["output"][0], np.array([1, 2, 3, 4]) / math.sqrt(7.5), atol=1e-15)
    np.testing.assert_allclose(r1["inv_std_dev"], [1 / math.sqrt(7.5)], rtol=1e-15)


@pytest.mark.parametrize("skip_shape", [(2, 3, 4), (1, 3, 4), (3, 4)])
def test_sln_skip_broadcast_brute_force(skip_shape):
    # the r mod skipRows map against NumPy's own broadcasting of skip over input
    x = rng.standard_normal((2, 3, 4)).astype(np.float32)
    sk = rng.standard_normal(skip_shape).astype(np.float32)
    g = rng.uniform(0.5, 1.5, 4).astype(np.float32)
    b = rng.standard_normal(4).astype(np.float32)
    got = oracle.skip_layer_norm(x, sk, g, b)["output"]
    full = np.ascontiguousarray(np.broadcast_to(sk, x.shape))
    want = oracle.skip_layer_norm(x, full, g, b)["output"]
    assert np.array_equal(got, want)
    # and against torch's layer_norm of the explicitly broadcast sum
    s = torch.from_numpy(x).double() + torch.from_numpy(sk).double()
    ref = torch.nn.functional.layer_norm(s, (4,), torch.from_numpy(g).double(), torch.from_numpy(b).double(),
                                         float(np.float32(oracle.DEFAULT_EPSILON)))
    np.testing.assert_allclose(got, ref.reshape(6, 4).numpy(), atol=1e-12)


def test_sln_rows_subset_matches_full():
    x = rng.standard_normal((40, 33)).astype(np.float16)
    sk = rng.standard_normal((8, 33)).astype(np.float16)  # 8 skip rows, cyclic
    g = rng.uniform(0.5, 1.5, 33).astype(np.float16)
    full = oracle.skip_layer_norm(x, sk, g)["output"]
    rows = [0, 9, 17, 39]
    sub = oracle.skip_layer_norm(x, sk, g, rows=rows)["output"]
    assert np.array_equal(sub, full[rows])


def test_skip_bias_sum_order_and_rounding_f32():
    # ((1 + 2^-24) + 2^-24) in float32: the first sum is a tie that rounds to 1,
    # so the result is 1.0.  Adding in any other order gives 1 + 2^-23.
    x = np.array([[1.0]], np.float32)
    sk = np.array([[2.0 ** -24]], np.float32)
    b = np.array([2.0 ** -24], np.float32)
    out = oracle.skip_bias_sum(x, sk, b)
    assert out.dtype == np.float32 and out[0, 0] == np.float32(1.0)
    # without bias it is the plain float32 sum
    assert oracle.skip_bias_sum(x, sk)[0, 0] == np.float32(1.0)


def test_skip_bias_sum_f16_rounds_once_from_float32():
    # 2048 + 1 = 2049 exactly in float32; + 2^-14 is below half a float32 ulp
    # at 2049, so the float32 sum is 2049, a tie between the float16 neighbours
    # 2048 and 2050 that rounds to even (2048).  Rounding the exact sum
    # 2049.00006 to float16 directly would give 2050.
    x = np.array([[2048.0]], np.float16)
    sk = np.array([[1.0]], np.float16)
    b = np.array([2.0 ** -14], np.float16)
    out = oracle.skip_bias_sum(x, sk, b)
    assert out.dtype == np.float16 and float(out[0, 0]) == 2048.0


def test_skip_bias_sum_broadcast_and_rows():
    x = rng.standard_normal((6, 5)).astype(np.float16)
    sk = rng.standard_normal((3, 5)).astype(np.float16)
    full = oracle.skip_bias_sum(x, sk)
    for r in range(6):
        for j in range(5):
            want = np.float16(np.float32(x[r, j]) + np.float32(sk[r % 3, j]))
            assert full[r, j] == want
    assert np.array_equal(oracle.skip_bias_sum(x, sk, rows=[5, 1]), full[[5, 1]])


# ---------------------------------------------------------------------------
# BiasSoftmax
# ---------------------------------------------------------------------------

def test_softmax_closed_forms():
    # [0, ln 3] -> [1/4, 3/4]
    d = np.array([[0.0, math.log(3.0)]], np.float64).astype(np.float32)
    out = oracle.bias_softmax(d, np.zeros((1, 2), np.float32), axis=1, is_inner_broadcast=0)
    np.testing.assert_allclose(out[0], [0.25, 0.75], atol=1e-7)  # ln 3 rounded to float32
    # a uniform row -> 1/n
    d = np.full((3, 7), 0.625, np.float32)
    out = oracle.bias_softmax(d, np.zeros((1, 7), np.float32), axis=1, is_inner_broadcast=1)
    assert np.allclose(out, 1 / 7, rtol=0, atol=1e-16)
    # blockSize = 1 -> 1
    d = rng.standard_normal((5, 1)).astype(np.float32)
    out = oracle.bias_softmax(d, rng.standard_normal((5, 1)).astype(np.float32), axis=1, is_inner_broadcast=0)
    assert np.all(out == 1.0)
    # huge equal logits do not overflow
    d = np.array([[60000.0, 60000.0]], np.float16)
    out = oracle.bias_softmax(d, np.zeros((1, 2), np.float16), axis=1, is_inner_broadcast=0)
    assert np.all(out == 0.5)


def test_softmax_rows_sum_to_one():
    d = (4 * rng.standard_normal((9, 300))).astype(np.float16)
    b = rng.standard_normal((3, 300)).astype(np.float16)
    out = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=1)
    np.testing.assert_allclose(out.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(out >= 0)


def test_softmax_shift_invariance_exact():
    # data on a 2^-8 grid; adding 2 is exact in float32, and exp(z - max z)
    # sees identical arguments, so the outputs are identical
    d = (np.round(rng.standard_normal((4, 50)) * 256) / 256).astype(np.float32)
    b = (np.round(rng.standard_normal((1, 50)) * 256) / 256).astype(np.float32)
    o1 = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=0)
    o2 = oracle.bias_softmax(d + np.float32(2.0), b, axis=1, is_inner_broadcast=0)
    assert np.array_equal(o1, o2)


def test_softmax_zero_bias_is_torch_softmax():
    d = rng.standard_normal((2, 3, 4, 5)).astype(np.float32)
    out = oracle.bias_softmax(d, np.zeros((2, 3, 4, 5), np.float32), axis=2, is_inner_broadcast=1)
    ref = torch.softmax(torch.from_numpy(d).double().reshape(6, 20), dim=1)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-15)


@pytest.mark.parametrize("bias_shape,inner", [((2, 1, 1, 5), 1), ((1, 3, 4, 5), 0), ((1, 1, 1, 5), 1),
                                               ((1, 1, 1, 5), 0), ((2, 3, 4, 5), 0), ((2, 3, 4, 5), 1)])
def test_softmax_bias_map_brute_force(bias_shape, inner):
    # The manifest only derives biasBlockCount and innerRepeat; its description
    # says inner broadcast reuses a bias row for consecutive groups and outer
    # broadcast reuses the bias rows cyclically.  Those maps equal NumPy/torch
    # broadcasting when the bias covers the leading (inner) or trailing (outer)
    # batch dims, which checks them by an independent mechanism.
    d = rng.standard_normal((2, 3, 4, 5)).astype(np.float32)
    b = rng.standard_normal(bias_shape).astype(np.float32)
    out = oracle.bias_softmax(d, b, axis=3, is_inner_broadcast=inner)
    z = torch.from_numpy(d).double() + torch.from_numpy(b).double()
    ref = torch.softmax(z, dim=3).reshape(24, 5)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-15)


def test_softmax_inner_and_outer_differ():
    # the two maps are distinguishable: bias (2,...) over 4 batch rows
    d = np.zeros((4, 3), np.float32)
    b = np.array([[0, -50, -50], [-50, 0, -50]], np.float32)
    inner = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=1)
    outer = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=0)
    assert list(np.argmax(inner, axis=1)) == [0, 0, 1, 1]
    assert list(np.argmax(outer, axis=1)) == [0, 1, 0, 1]


def test_softmax_flattened_suffix_and_negative_axis():
    d = rng.standard_normal((2, 3, 4, 5)).astype(np.float32)
    b = rng.standard_normal((1, 3, 4, 5)).astype(np.float32)
    out = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=0)
    ref = torch.softmax(torch.from_numpy(d).double().reshape(2, 60) + torch.from_numpy(b).double().reshape(1, 60), dim=1)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-15)
    b3 = rng.standard_normal((1, 1, 1, 5)).astype(np.float32)
    assert np.array_equal(oracle.bias_softmax(d, b3, axis=-1, is_inner_broadcast=0),
                          oracle.bias_softmax(d, b3, axis=3, is_inner_broadcast=0))


def test_softmax_masked_columns_are_zero():
    d = (4 * rng.standard_normal((8, 16))).astype(np.float16)
    mask = np.where(np.arange(16)[None, :] <= np.arange(8)[:, None], 0.0, -10000.0).astype(np.float16)
    out = oracle.bias_softmax(d, mask, axis=1, is_inner_broadcast=1)
    for r in range(8):
        assert np.all(out[r, r + 1:] == 0.0)
        assert out[r, : r + 1].sum() == pytest.approx(1.0, abs=1e-12)


@pytest.mark.parametrize("shape,bias_numel,axis,ok", [
    ((4, 6), 6, 1, True),        # one bias row shared by 4 data rows
    ((4, 6), 12, 1, True),       # 2 bias rows, 4 % 2 == 0
    ((4, 6), 24, 1, True),       # one bias row per data row
    ((4, 6), 18, 1, False),      # 3 bias rows do not divide 4
    ((4, 6), 48, 1, False),      # more bias rows than data rows
    ((4, 6), 7, 1, False),       # not a whole number of rows
    ((4, 6), 0, 1, False),       # empty bias with non-empty data
    ((0, 6), 0, 1, True),        # both empty
    ((2, 3, 4), 12, 1, True),    # blockSize = 3*4 = 12
    ((2, 3, 4), 4, -1, True),    # negative axis
])
def test_bias_contract_table(shape, bias_numel, axis, ok):
    # com.microsoft.BiasSoftmax manifest, derive.biasContract
    assert oracle.bias_softmax_dims(shape, bias_numel, axis)["contract_ok"] is ok


def test_bias_softmax_rows_subset():
    d = rng.standard_normal((12, 10)).astype(np.float32)
    b = rng.standard_normal((4, 10)).astype(np.float32)
    for inner in (0, 1):
        full = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=inner)
        sub = oracle.bias_softmax(d, b, axis=1, is_inner_broadcast=inner, rows=[11, 0, 5])
        assert np.array_equal(sub, full[[11, 0, 5]])


# ---------------------------------------------------------------------------
# BiasAdd
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_bias_add_exact_rational_brute_force(dtype):
    x = rng.standard_normal((2, 3, 4)).astype(dtype)
    b = rng.standard_normal(4).astype(dtype)
    s = rng.standard_normal((2, 3, 4)).astype(dtype)
    out = oracle.bias_add(x, b, s)
    for n in range(2):
        for t in range(3):
            for c in range(4):
                exact = Fraction(float(x[n, t, c])) + Fraction(float(b[c])) + Fraction(float(s[n, t, c]))
                got = Fraction(float(out[n, t, c]))
                if dtype == np.float16:
                    assert got == exact          # fp16 terms: float64 sum is exact
                else:
                    assert abs(got - exact) <= abs(exact) * Fraction(1, 2 ** 52) + Fraction(1, 2 ** 200)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["skip_is_minus_x", "skip_is_minus_bias", "random"])
def test_bias_add_exact_with_wide_exponents(dtype, mode):
    # terms whose exponents differ by more than float64's 53 bits, with a skip
    # that cancels one of them: the result is still the exact sum to within
    # two float64 roundings (a plain float64 sum would keep only the rounding
    # error of x + bias)
    g = np.random.default_rng(17)

    def wide(*shape):
        v = (g.random(shape) + 1.0) * np.exp2(g.integers(-60, 61, shape)) * np.where(g.random(shape) < 0.5, -1, 1)
        t = torch.from_numpy(v.astype(np.float32))
        return t.to(torch.bfloat16) if dtype == "bf16" else t

    x = wide(2, 3, 8)
    b = wide(8)
    if mode == "skip_is_minus_x":
        s = -x
    elif mode == "skip_is_minus_bias":
        s = (-b).expand(2, 3, 8).contiguous()
    else:
        s = wide(2, 3, 8)
    out = oracle.bias_add(x, b, s)
    xf, bf, sf = (t.double().numpy() for t in (x, b, s))
    for n in range(2):
        for t in range(3):
            for c in range(8):
                exact = Fraction(float(xf[n, t, c])) + Fraction(float(bf[c])) + Fraction(float(sf[n, t, c]))
                got = Fraction(float(out[n, t, c]))
                assert abs(got - exact) <= abs(exact) * Fraction(1, 2 ** 51), (n, t, c, float(got), float(exact))


# ---------------------------------------------------------------------------
# QuickGelu
# ---------------------------------------------------------------------------

def test_quick_gelu_zero_and_symmetry():
    x = (3 * rng.standard_normal(4096)).astype(np.float32)
    f = oracle.quick_gelu(x)
    fm = oracle.quick_gelu(-x)
    # sigmoid(t) + sigmoid(-t) = 1  =>  f(x) - f(-x) = x
    np.testing.assert_allclose(f - fm, x.astype(np.float64), rtol=0, atol=4e-15 * np.abs(x).max())
    assert oracle.quick_gelu(np.zeros(3, np.float32)).tolist() == [0.0, 0.0, 0.0]


def test_quick_gelu_alpha_zero_is_half():
    x = rng.standard_normal(100).astype(np.float32)
    assert np.array_equal(oracle.quick_gelu(x, alpha=0.0), x.astype(np.float64) / 2)


def test_quick_gelu_mpmath_values():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    a = mp.mpf(float(np.float32(1.702)))
    xs = [1.0, -1.0, 2.0, 0.5, -3.0, 20.0, -50.0, -200.0, 1e-30]
    x32 = np.array(xs, np.float64).astype(np.float32)
    got = oracle.quick_gelu(x32)
    for x, g in zip(x32.astype(np.float64).tolist(), got):
        want = mp.mpf(x) / (1 + mp.exp(-a * mp.mpf(x)))
        assert abs(g - float(want)) <= 4e-16 * abs(float(want)), (x, g, want)


def test_quick_gelu_worked_values_at_default_alpha():
    # x * sigmoid(1.702 x) worked at a few points (alpha as float32 shifts them
    # by < 1e-7 relative)
    got = oracle.quick_gelu(np.array([1, -1, 2, 0.5, -3], np.float32))
    want = [0.845795766, -0.154204234, 1.935658623, 0.350388437, -0.018071310]
    np.testing.assert_allclose(got, want, rtol=2e-7, atol=0)


def test_quick_gelu_ieee_specials():
    out = oracle.quick_gelu(np.array([np.inf, -np.inf, np.nan], np.float32))
    assert out[0] == np.inf and np.isnan(out[1]) and np.isnan(out[2])


def test_skip_bias_sum_bf16_rounds_to_nearest_even():
    # bfloat16 spacing at 1 is 2^-7.  1 + 2^-8 is a tie that goes to the even
    # neighbour 1; 1 + 2^-7 + 2^-8 is a tie between 1 + 2^-7 (odd) and
    # 1 + 2^-6 (even).  Truncation would give 1 + 2^-7 for the second.
    x = torch.tensor([[1.0, 1.0 + 2.0 ** -7]], dtype=torch.bfloat16)
    sk = torch.tensor([[2.0 ** -8, 2.0 ** -8]], dtype=torch.bfloat16)
    out = oracle.skip_bias_sum(x, sk)
    assert out.dtype == torch.bfloat16
    assert out.float().tolist() == [[1.0, 1.0 + 2.0 ** -6]]


def test_bf16_inputs_enter_exactly():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(5, 64, generator=g).to(torch.bfloat16)
    sk = torch.randn(5, 64, generator=g).to(torch.bfloat16)
    gm = torch.rand(64, generator=g).to(torch.bfloat16)
    a = oracle.skip_layer_norm(x, sk, gm)["output"]
    b = oracle.skip_layer_norm(x.float(), sk.float(), gm.float())["output"]
    assert np.array_equal(a, b)
    assert np.array_equal(oracle.quick_gelu(x), oracle.quick_gelu(x.float()))
