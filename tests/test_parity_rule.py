"""The float16 / bfloat16 comparison rule itself (no GPU): it accepts the
correctly rounded value of any float32 result within the op's float32 error
bound, and rejects the wrong neighbour wherever correct rounding can meet the
stated bound."""
import numpy as np
import pytest
import torch

from tests import _helpers as h


def _grid(lo, hi, n=20001):
    return np.linspace(lo, hi, n)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("lo,hi", [(-9.0, 9.0), (3.5, 8.5), (15.0, 17.0), (1e-4, 3e-3)])
def test_correct_rounding_of_a_perturbed_float32_passes(dtype, lo, hi):
    o = _grid(lo, hi)
    rng = np.random.default_rng(0)
    for scale in (0.0, 0.5, 1.0):   # float32 errors up to the bound delta = 1e-5
        g32 = o + scale * h.F32_ABS * rng.uniform(-1, 1, o.shape)
        got = torch.from_numpy(g32.astype(np.float32)).to(dtype)
        h.assert_norm_close(got, o, dtype)


def test_float16_wrong_neighbour_fails_below_8():
    # for 4 <= |o| < 8, half a float16 spacing is 2^-9 < 2e-3, so the rule is
    # the literal 2e-3 and the far neighbour (3 half-spacings away) fails
    o = np.array([4.0 + 2.0 ** -9 * 0.9, 5.5 + 2.0 ** -10, 7.9 + 2.0 ** -9 * 0.6, 6.2])
    right = torch.from_numpy(o.astype(np.float32)).to(torch.float16)
    h.assert_norm_close(right, o, torch.float16)
    step = torch.from_numpy(h.ulp16(o).astype(np.float32))
    # the neighbour on the other side of o from the correctly rounded value
    wrong = torch.where(right.double() >= torch.from_numpy(o), right.float() - step, right.float() + step)
    with pytest.raises(AssertionError):
        h.assert_norm_close(wrong.to(torch.float16), o, torch.float16)
    for i in range(o.size):
        with pytest.raises(AssertionError):
            h.assert_elementwise_close(wrong[i:i + 1].to(torch.float16), o[i:i + 1], torch.float16)


def test_float16_literal_bound_below_8():
    o = np.linspace(-8 + 2e-5, 8 - 2e-5, 10001)
    tol = h.low_precision_tol(o, torch.float16, h.F32_ABS)
    assert np.all(tol == h.F16_ABS)
    o = np.array([8.0, 9.0, 15.9])
    tol = h.low_precision_tol(o, torch.float16, h.F32_ABS)
    assert np.all(tol <= 2.0 ** -8 + h.F32_ABS) and np.all(tol > h.F16_ABS)


def test_bfloat16_wrong_neighbour_fails():
    o = np.array([1.0 + 2.0 ** -8 * 0.7, 3.3, 100.2, 1e-3 * 1.37, -7.77])
    right = torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16)
    h.assert_elementwise_close(right, o, torch.bfloat16)
    step = torch.from_numpy(h.ulp_bf16(o).astype(np.float32))
    wrong = torch.where(right.double() >= torch.from_numpy(o), right.float() - step, right.float() + step)
    for i in range(o.size):
        with pytest.raises(AssertionError):
            h.assert_elementwise_close(wrong[i:i + 1].to(torch.bfloat16), o[i:i + 1], torch.bfloat16)


def test_quick_gelu_delta_is_relative_to_the_result():
    x = torch.tensor([-30.0, -5.0, 0.0, 5.0, 60.0], dtype=torch.float32)
    a = float(np.float32(1.702))
    xs = x.double().numpy()
    o = xs / (1.0 + np.exp(-a * xs))
    d = h.quick_gelu_delta(x, 1.702, o)
    # large positive x: y = x, the exponent's error is weighted by sigmoid(-alpha x) ~ 0
    assert d[4] < 1e-5 * abs(o[4]) and d[3] < 2e-6 * abs(o[3])
    # large negative x: the exponent's error reaches y in full, ~ ln2 |t| 2^-22 relative
    assert 5e-6 * abs(o[0]) < d[0] < 3e-5 * abs(o[0])
    assert d[2] == h.TINY
