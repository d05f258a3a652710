"""bfloat16 through every op and kernel path: CUDA (through the C ABI) vs the
float64 oracle, |gpu - o| <= half a bfloat16 spacing plus the float32 error
bound of each op's arithmetic (tests/_helpers.py); the residual output and
bias-row indexing bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gen import synth
from tests import test_gpu_bias_softmax as sm
from tests import test_gpu_elementwise as ew
from tests import test_gpu_skip_layer_norm as sln

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,rows,skip", [
    (7, 19, None),          # register path, scalar (H % 8 != 0)
    (768, 37, None),        # staged path, ragged row shape
    (4096, 300, None),      # staged path, exact rows, several tiles per CTA
    (4100, 9, None),        # register path (H % 8 != 0)
    (20000, 3, None),       # three-pass path
    (1024, 64, 16),         # broadcast skip
])
def test_skip_layer_norm_bf16(lib, H, rows, skip):
    if skip is None:
        d = synth.sln_inputs((rows, H), None, "bf16", has_beta=True, has_bias=True, seed=H)
    else:
        d = synth.sln_inputs((rows // skip, skip, H), (1, skip, H), "bf16", has_beta=True, has_bias=True, seed=H)
    out, s = sln.run(lib, d, residual=True)
    sln.check(d, out, s)


@pytest.mark.parametrize("simplified", [False, True])
def test_skip_layer_norm_ex_bf16(lib, simplified):
    d = synth.sln_inputs((40, 2048), None, "bf16", has_beta=not simplified, has_bias=True, seed=2)
    out, s, mean, inv = sln.run_ex(lib, d, simplified)
    o = oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                               simplified=simplified)
    sln.assert_norm_close(out, o["output"], torch.bfloat16)
    np.testing.assert_allclose(inv.numpy().astype(np.float64), o["inv_std_dev"], rtol=2e-5)


@pytest.mark.parametrize("cols,rows,bias_rows,inner", [
    (5, 4096, 8, 1),        # packed rows
    (512, 2048, 128, 1),    # staged row kernel
    (1000, 48, 3, 0),       # staged, ragged row shape
    (4100, 12, 4, 1),       # register row kernel
    (20000, 4, 2, 0),       # split rows
])
def test_bias_softmax_bf16(lib, cols, rows, bias_rows, inner):
    d = synth.bias_softmax_inputs((rows, cols), (bias_rows, cols), "bf16", data_std=3.0, seed=cols)
    out = sm.run(lib, d["data"], d["bias"], 1, inner)
    sm.check(d["data"], d["bias"], 1, inner, out)


def test_bias_softmax_bf16_causal(lib):
    d = synth.bias_softmax_inputs((2, 4, 64, 64), (2, 64, 64), "bf16", data_std=4.0, seed=1, causal=True)
    out = sm.run(lib, d["data"], d["bias"], 3, 1)
    sm.check(d["data"], d["bias"], 3, 1, out)


@pytest.mark.parametrize("shape", [(2, 3, 5), (5, 17, 4096), (8, 1000, 4096)])
def test_bias_add_bf16(lib, shape):
    d = synth.bias_add_inputs(shape, "bf16", seed=sum(shape))
    out = ew.run_bias_add(lib, d)
    ew.check_bias_add(out, d["X"], d["bias"], d["skip"])


@pytest.mark.parametrize("n,offs", [(1001, None), ((1 << 20) + 5, None), (70000, {"X": 2, "Y": 2})])
def test_quick_gelu_bf16(lib, n, offs):
    d = synth.quick_gelu_inputs(n, "bf16", seed=n)
    out = ew.run_gelu(lib, d["X"], d["alpha"], offsets=offs)
    ew.check_quick_gelu(out, d["X"], d["alpha"])


def test_quick_gelu_bf16_all_values(lib):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16)
    x = x[torch.isfinite(x)].contiguous()
    out = ew.run_gelu(lib, x, 1.702)
    ew.check_quick_gelu(out, x, 1.702)


def test_bias_add_bf16_cancellation(lib):
    # skip ~ -(x + bias): the compensated float32 sum keeps the result within a
    # bfloat16 spacing of the exact sum even when it is tiny
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(4, 8, 64, generator=g) * 100).to(torch.bfloat16)
    b = torch.randn(64, generator=g).to(torch.bfloat16)
    s = (-(x.double() + b.double()) + torch.randn(4, 8, 64, generator=g).double() * 1e-2).to(torch.bfloat16)
    out = ew.run_bias_add(lib, dict(X=x, bias=b, skip=s))
    ew.check_bias_add(out, x, b, s)


@pytest.mark.parametrize("mode", ["skip_is_minus_x", "skip_is_minus_bias", "random"])
def test_bias_add_bf16_wide_exponents(lib, mode):
    # terms whose exponents differ by far more than float32's 24 bits, so that
    # x + bias is not exact in float32, and a skip that cancels one of them:
    # the result must still be within a bfloat16 spacing of the exact sum
    g = torch.Generator().manual_seed(5)

    def wide(*shape):
        m = torch.rand(*shape, generator=g) + 1.0
        e = torch.randint(-60, 61, shape, generator=g).double()
        sign = torch.where(torch.rand(*shape, generator=g) < 0.5, -1.0, 1.0)
        return (sign * m * torch.pow(2.0, e)).to(torch.bfloat16)

    x = wide(4, 64, 64)
    b = wide(64)
    if mode == "skip_is_minus_x":
        s = -x
    elif mode == "skip_is_minus_bias":
        s = (-b).expand(4, 64, 64).contiguous()
    else:
        s = wide(4, 64, 64)
    out = ew.run_bias_add(lib, dict(X=x, bias=b, skip=s))
    ew.check_bias_add(out, x, b, s)
