"""BiasAdd and QuickGelu: CUDA path (through the C ABI) vs the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gen import synth
from tests._helpers import Guarded, assert_elementwise_close, bias_add_delta, offset_copy, quick_gelu_delta

pytestmark = pytest.mark.gpu


def check_bias_add(out, X, bias, skip):
    """out against the oracle's exact sum, with the float32 error bound of the
    kernel's arithmetic for float16 / bfloat16 results."""
    o = oracle.bias_add(X, bias, skip)
    T = torch.as_tensor(X).dtype
    return assert_elementwise_close(out, o, T, delta=bias_add_delta(X, bias, skip, o, T))


def check_quick_gelu(out, X, alpha):
    o = oracle.quick_gelu(X, alpha)
    T = torch.as_tensor(X).dtype
    return assert_elementwise_close(out, o, T, delta=quick_gelu_delta(X, alpha, o))


def run_bias_add(lib, d, offsets=None, guard=True):
    offsets = offsets or {}
    keep = []

    def dev(name):
        t = d[name]
        if name in offsets:
            raw, v = offset_copy(t, offsets[name])
            keep.append(raw)
            return v
        return t.cuda()

    g = Guarded(d["X"].shape, d["X"].dtype, offset_bytes=offsets.get("Y", 0))
    lib.ep_bias_add(dev("X"), dev("bias"), dev("skip"), Y=g.tensor)
    torch.cuda.synchronize()
    if guard:
        g.check()
    return g.tensor.cpu()


def run_gelu(lib, x, alpha, offsets=None):
    offsets = offsets or {}
    if "X" in offsets:
        raw, xd = offset_copy(x, offsets["X"])
    else:
        xd = x.cuda()
    g = Guarded(x.shape, x.dtype, offset_bytes=offsets.get("Y", 0))
    lib.ep_quick_gelu(xd, alpha, Y=g.tensor)
    torch.cuda.synchronize()
    g.check()
    return g.tensor.cpu()


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 4), (2, 3, 5), (3, 7, 8), (4, 5, 9), (2, 33, 64),
                                   (5, 17, 4096), (1, 1, 100003)])
def test_bias_add_shapes(lib, dtype, shape):
    d = synth.bias_add_inputs(shape, dtype, seed=sum(shape))
    out = run_bias_add(lib, d)
    check_bias_add(out, d["X"], d["bias"], d["skip"])


@pytest.mark.parametrize("dtype,offs", [("f16", {"X": 2}), ("f16", {"Y": 2}), ("f16", {"bias": 6}),
                                        ("f32", {"skip": 4}), ("f32", {"X": 8, "Y": 8, "skip": 8, "bias": 8})])
def test_bias_add_misaligned(lib, dtype, offs):
    d = synth.bias_add_inputs((3, 9, 64), dtype, seed=1)
    out = run_bias_add(lib, d, offsets=offs)
    check_bias_add(out, d["X"], d["bias"], d["skip"])


@pytest.mark.parametrize("dtype,offs", [
    ("f16", {"X": 2, "skip": 2, "Y": 2}), ("f16", {"X": 14, "skip": 14, "Y": 14, "bias": 6}),
    ("f16", {"bias": 2}), ("f32", {"X": 4, "skip": 4, "Y": 4}), ("f32", {"X": 8, "skip": 8, "Y": 8, "bias": 12}),
    ("bf16", {"X": 6, "skip": 6, "Y": 6}),
])
@pytest.mark.parametrize("shape", [(3, 700, 1024), (2, 999, 4104)])
def test_bias_add_same_offset_staged(lib, dtype, offs, shape):
    # X, skip and Y at the same offset within 16 bytes (the bias at any): the
    # staged kernel takes the aligned body after a scalar head, with the bias
    # staged rotated by the head; tiles, the ragged last tile and the tail
    d = synth.bias_add_inputs(shape, dtype, seed=sum(shape) + sum(offs.values()))
    out = run_bias_add(lib, d, offsets=offs)
    check_bias_add(out, d["X"], d["bias"], d["skip"])


def test_bias_add_f32_cancellation(lib):
    # skip = -(x + bias) + small: plain float32 (x + b) + s loses the small part;
    # the compensated sum keeps it to within relative 1e-6.
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4, 8, 64, generator=g) * 1000
    b = torch.randn(64, generator=g)
    small = torch.randn(4, 8, 64, generator=g) * 1e-3
    s = (-(x.double() + b.double()) + small.double()).float()
    d = dict(X=x, bias=b, skip=s)
    out = run_bias_add(lib, d)
    check_bias_add(out, x, b, s)


def test_bias_add_in_place(lib):
    d = synth.bias_add_inputs((2, 16, 128), "f16", seed=2)
    x = d["X"].cuda()
    lib.ep_bias_add(x, d["bias"].cuda(), d["skip"].cuda(), Y=x)
    torch.cuda.synchronize()
    check_bias_add(x.cpu(), d["X"], d["bias"], d["skip"])


@pytest.mark.parametrize("mode", ["skip_is_minus_x", "skip_is_minus_bias", "random"])
def test_bias_add_f32_wide_exponents(lib, mode):
    # terms whose exponents differ by far more than float32's 24 bits, with a
    # skip that cancels one of them: the result must be within the float32
    # tolerance of the exact sum
    g = torch.Generator().manual_seed(9)

    def wide(*shape):
        m = torch.rand(*shape, generator=g) + 1.0
        e = torch.randint(-60, 61, shape, generator=g).float()
        sign = torch.where(torch.rand(*shape, generator=g) < 0.5, -1.0, 1.0)
        return sign * m * torch.pow(2.0, e)

    x = wide(4, 64, 64)
    b = wide(64)
    if mode == "skip_is_minus_x":
        s = -x
    elif mode == "skip_is_minus_bias":
        s = (-b).expand(4, 64, 64).contiguous()
    else:
        s = wide(4, 64, 64)
    out = run_bias_add(lib, dict(X=x, bias=b, skip=s))
    check_bias_add(out, x, b, s)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 9, 15, 16, 17, 1000, 4099, 1 << 20, (1 << 20) + 5])
def test_quick_gelu_sizes(lib, dtype, n):
    d = synth.quick_gelu_inputs(n, dtype, seed=n)
    out = run_gelu(lib, d["X"], d["alpha"])
    check_quick_gelu(out, d["X"], d["alpha"])


@pytest.mark.parametrize("dtype,offs", [("f16", {"X": 2, "Y": 2}), ("f16", {"X": 2, "Y": 4}), ("f16", {"Y": 14}),
                                        ("f32", {"X": 4, "Y": 4}), ("f32", {"X": 8}), ("f32", {"Y": 12})])
@pytest.mark.parametrize("n", [5, 1001, 70000])
def test_quick_gelu_misaligned(lib, dtype, offs, n):
    d = synth.quick_gelu_inputs(n, dtype, seed=7)
    out = run_gelu(lib, d["X"], d["alpha"], offsets=offs)
    check_quick_gelu(out, d["X"], d["alpha"])


@pytest.mark.parametrize("alpha", [1.702, 0.0, -1.0, 1.0, 3.5])
def test_quick_gelu_f32_wide_range(lib, alpha):
    # a dense grid over [-120, 120] exercises every branch of the float32 kernel,
    # including the products that fall into the subnormal range
    x = torch.linspace(-120, 120, 200001, dtype=torch.float32)
    out = run_gelu(lib, x, alpha)
    check_quick_gelu(out, x, alpha)


@pytest.mark.parametrize("alpha", [1.702, -0.5])
def test_quick_gelu_f32_random_bits(lib, alpha):
    # random float32 bit patterns: every exponent, subnormal inputs, products
    # alpha*x that overflow, results that underflow
    x = synth.float32_bit_patterns(1 << 21, seed=11)
    out = run_gelu(lib, x, alpha)
    check_quick_gelu(out, x, alpha)


def test_quick_gelu_f16_all_values(lib):
    # every finite float16 value
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.float16)
    x = x[torch.isfinite(x)].contiguous()
    out = run_gelu(lib, x, 1.702)
    check_quick_gelu(out, x, 1.702)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_quick_gelu_specials(lib, dtype):
    x = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"), 1.0], dtype=dtype)
    out = run_gelu(lib, x, 1.702).float()
    assert out[0] == 0 and out[1] == 0 and out[2] == float("inf")
    assert torch.isnan(out[3]) and torch.isnan(out[4])


def test_quick_gelu_in_place(lib):
    d = synth.quick_gelu_inputs(12345, "f16", seed=3)
    x = d["X"].cuda()
    lib.ep_quick_gelu(x, d["alpha"], Y=x)
    torch.cuda.synchronize()
    check_quick_gelu(x.cpu(), d["X"], d["alpha"])


def test_empty_launches_nothing(lib):
    n0 = lib.kernel_launch_count()
    lib.ep_quick_gelu(torch.empty(0, device="cuda"))
    lib.ep_bias_add(torch.empty(0, 3, 4, device="cuda"), torch.zeros(4, device="cuda"),
                    torch.empty(0, 3, 4, device="cuda"))
    assert lib.kernel_launch_count() == n0


# ---------------------------------------------------------------------------
# the measured workloads
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_workload_bias_add_f16_full(lib):
    d = synth.workload("bias_add_f16_16x1024x4096")
    out = run_bias_add(lib, d)
    # every element (the float64 sum of float16 terms is exact)
    check_bias_add(out, d["X"], d["bias"], d["skip"])


@pytest.mark.slow
def test_workload_quick_gelu_f16_full(lib):
    d = synth.workload("quick_gelu_f16_67108867")
    out = run_gelu(lib, d["X"], d["alpha"])
    # every element, including the 3-element tail after the 8-wide vectors
    check_quick_gelu(out, d["X"], d["alpha"])


# ---------------------------------------------------------------------------
# many tiles per CTA on the shared-memory-staged kernels, ragged last tile and
# a scalar tail
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,n", [("f16", (1 << 24) + 5), ("f32", (1 << 23) + 3), ("f16", 8192 * 3001 + 8)])
def test_quick_gelu_staged_many_tiles(lib, dtype, n):
    d = synth.quick_gelu_inputs(n, dtype, seed=n)
    out = run_gelu(lib, d["X"], d["alpha"])
    check_quick_gelu(out, d["X"], d["alpha"])


@pytest.mark.parametrize("dtype,shape", [("f16", (8, 1000, 4096)), ("f32", (3, 777, 1000)), ("f16", (5, 999, 7000))])
def test_bias_add_staged_many_tiles(lib, dtype, shape):
    d = synth.bias_add_inputs(shape, dtype, seed=shape[1])
    out = run_bias_add(lib, d)
    check_bias_add(out, d["X"], d["bias"], d["skip"])
