"""Comparison rules and guard-band canaries shared by the GPU parity tests.

Tolerances (written out here, applied element by element; ``o`` is always the
oracle's unrounded float64 value):
  * float32 SkipLayerNormalization / BiasSoftmax: |gpu - o| <= 1e-5.
  * float32 BiasAdd / QuickGelu: |gpu - o| <= 1e-6 * |o| + 2**-149.
  * float16 and bfloat16: the kernels compute in float32 and round once to T.
    If the float32 value g is within delta of o, the rounded result is within
    half a T spacing of g, so

        |gpu - o| <= half_spacing_T(|o| + delta) + delta,

    where half_spacing_T(a) is half the distance between the T values around a
    (taken at |o| + delta, so that a g just across a power of two is covered).
    float16 additionally keeps the stated absolute bound:
    |gpu - o| <= max(2e-3, the above).  Below |o| = 8 - delta the float16 rule
    is the literal 2e-3 (half a spacing is at most 2**-9 = 1.953e-3 there);
    from 8 up, correct rounding alone can err by 2**-8 = 3.9e-3.
    delta, the float32 error before the final rounding, per op:
      - LayerNorm / softmax: 1e-5, the float32 criterion the same float32
        arithmetic is held to by the float32 tests (the kernels are the same
        templates, computing in float32 for every T);
      - BiasAdd float16: the plain float32 sum (x + b) + s, two roundings:
        2**-24 (|x + b| + |o|) (1 + 2**-23);
      - BiasAdd bfloat16: the first addition compensated (TwoSum), so the sum
        is within two float32 ulps: 2**-22 |o|;
      - QuickGelu (float16 and bfloat16): y = x / (1 + u), u = 2^t,
        t = -alpha x log2(e) rounded twice (|dt| <= 2**-23 |t|, twice that on
        the bfloat16 underflow branch), so 2^t is off by ln2 |dt| relatively,
        which reaches y weighted by w = u / (1 + u) = 1 - sigmoid(alpha x);
        plus 8 float32 ulps for the approximate 2^x and reciprocal and the
        roundings of 1 + u and of the product:
        (ln2 |t| w 2**-22 + 8 * 2**-23) |o|;
      - every delta also has 2**-149 added (float32 subnormal results).
  * the input_skip_bias_sum output and broadcast row indexing: bit-exact.

Every comparison records its literal max |gpu - o| and its largest ratio
|gpu - o| / tolerance under the running test's name (``RECORDS``); the
test session prints them in its summary.
"""
import math

import numpy as np
import torch

F32_ABS = 1e-5
F32_REL = 1e-6
F16_ABS = 2e-3
TINY = 2.0 ** -149
U32 = 2.0 ** -24          # float32 unit roundoff
LN2 = math.log(2.0)
LOG2E = 1.0 / LN2

# (test node id, kind, dtype, elements compared, max |gpu - o|, max ratio to the tolerance)
RECORDS = []
CURRENT_TEST = ["(outside a test)"]


def _record(kind, dtype, g, o, tol, ok_mask):
    d = np.abs(g - o)
    fin = np.isfinite(d) & ok_mask
    max_abs = float(np.max(d[fin])) if fin.any() else 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(fin & (tol > 0), d / np.where(tol > 0, tol, 1.0), 0.0)
    max_ratio = float(np.max(r)) if r.size else 0.0
    RECORDS.append((CURRENT_TEST[0], kind, str(dtype).replace("torch.", ""), int(o.size), max_abs, max_ratio))
    return max_abs


def _exp2_floor(a):
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.floor(np.log2(np.where(a > 0, a, 1.0)))


def ulp16(o):
    """float16 spacing at |o| (2**(floor(log2|o|) - 10), at least 2**-24)."""
    return np.maximum(2.0 ** (_exp2_floor(np.abs(o)) - 10), 2.0 ** -24)


def ulp_bf16(o):
    """bfloat16 spacing at |o| (2**(floor(log2|o|) - 7), at least 2**-133)."""
    return np.maximum(2.0 ** (_exp2_floor(np.abs(o)) - 7), 2.0 ** -133)


def low_precision_tol(o, dtype, delta):
    """Half a T spacing at |o| + delta, plus delta; float16 at least 2e-3."""
    with np.errstate(invalid="ignore", over="ignore"):
        a = np.abs(o) + delta
        if dtype == torch.bfloat16:
            return 0.5 * ulp_bf16(a) + delta
        return np.maximum(F16_ABS, 0.5 * ulp16(a) + delta)


def to_np64(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def _report(bad, gpu, o, tol, what):
    idx = np.argwhere(bad)[:5]
    rows = [(tuple(int(j) for j in i), float(gpu[tuple(i)]), float(o[tuple(i)]), float(tol[tuple(i)]))
            for i in idx]
    return f"{what}: {int(bad.sum())} elements out of tolerance, first (index, gpu, oracle, tol): {rows}"


def assert_norm_close(gpu: torch.Tensor, o: np.ndarray, dtype):
    """LayerNorm / softmax outputs; returns the literal max |gpu - o|."""
    g = to_np64(gpu).reshape(o.shape)
    both_nan = np.isnan(g) & np.isnan(o)
    if dtype == torch.float32:
        tol = np.full(o.shape, F32_ABS)
    else:
        tol = low_precision_tol(o, dtype, F32_ABS + TINY)
    bad = ~both_nan & ~(np.abs(g - o) <= tol)
    assert not bad.any(), _report(bad, g, o, tol, "norm/softmax")
    return _record("norm", dtype, g, o, tol, ~both_nan)


def assert_elementwise_close(gpu: torch.Tensor, o: np.ndarray, dtype, delta=None):
    """BiasAdd / QuickGelu outputs; returns the literal max |gpu - o| over the
    finite oracle values.  ``delta`` is the float32 error bound before the
    final rounding for float16 / bfloat16 (``bias_add_delta``,
    ``quick_gelu_delta``); it defaults to the float32 criterion."""
    g = to_np64(gpu).reshape(o.shape)
    both_nan = np.isnan(g) & np.isnan(o)
    same_inf = np.isinf(o) & (g == o)
    with np.errstate(invalid="ignore", over="ignore"):
        if dtype == torch.float32:
            tol = F32_REL * np.abs(o) + TINY
        else:
            dl = F32_REL * np.abs(o) + TINY if delta is None else np.asarray(delta, dtype=np.float64).reshape(o.shape)
            tol = low_precision_tol(o, dtype, dl)
        bad = ~both_nan & ~same_inf & ~(np.abs(g - o) <= tol)
    assert not bad.any(), _report(bad, g, o, tol, "elementwise")
    return _record("elementwise", dtype, g, o, tol, np.isfinite(o))


def bias_add_delta(X, bias, skip, o, dtype):
    """float32 error bound of the kernel's BiasAdd sum before the rounding to T
    (see the module docstring); X, bias, skip as given to the op, o the oracle."""
    o = np.asarray(o, dtype=np.float64)
    if dtype == torch.bfloat16:
        return 2.0 ** -22 * np.abs(o) + TINY
    x = to_np64(torch.as_tensor(X)).reshape(o.shape)
    C = o.shape[-1]
    b = to_np64(torch.as_tensor(bias)).reshape((1,) * (o.ndim - 1) + (C,))
    with np.errstate(invalid="ignore", over="ignore"):
        return U32 * (np.abs(x + b) * (1 + 2.0 ** -23) + np.abs(o)) + TINY


def quick_gelu_delta(X, alpha, o):
    """float32 error bound of the kernels' float16 / bfloat16 QuickGelu before
    the rounding to T (see the module docstring)."""
    o = np.asarray(o, dtype=np.float64)
    x = to_np64(torch.as_tensor(X)).reshape(o.shape)
    a = float(np.float32(alpha))
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        t = np.abs(a * x * LOG2E)
        sig = np.where(x != 0, o / np.where(x != 0, x, 1.0), 0.5)   # sigmoid(alpha x) = o / x
        w = np.clip(1.0 - sig, 0.0, 1.0)
        rel = LN2 * t * w * 2.0 ** -22 + 8 * 2.0 ** -23
        return np.where(np.isfinite(rel), rel, np.inf) * np.abs(o) + TINY


def assert_bit_exact(gpu: torch.Tensor, want):
    if gpu.dtype == torch.bfloat16:
        g16 = gpu.detach().cpu().reshape(-1).view(torch.int16)
        w16 = torch.as_tensor(want).reshape(-1).view(torch.int16)
        bad = (g16 != w16).numpy()
        assert not bad.any(), f"{int(bad.sum())} bfloat16 elements differ bitwise, first at {np.argwhere(bad)[:5].tolist()}"
        return
    g = gpu.detach().cpu().numpy()
    w = np.asarray(want).reshape(g.shape)
    assert g.dtype == w.dtype
    gi = g.view(np.uint16 if g.dtype == np.float16 else np.uint32)
    wi = w.view(np.uint16 if w.dtype == np.float16 else np.uint32)
    bad = gi != wi
    assert not bad.any(), f"{int(bad.sum())} elements differ bitwise, first at {np.argwhere(bad)[:5].tolist()}"


# ---------------------------------------------------------------------------
# guard bands: outputs are views into a larger buffer whose padding holds a
# sentinel byte pattern; any write outside the view changes the padding.
# ---------------------------------------------------------------------------

GUARD_BYTES = 4096
SENTINEL = 0x5A


class Guarded:
    def __init__(self, shape, dtype, device="cuda", offset_bytes=0):
        es = torch.empty((), dtype=dtype).element_size()
        assert offset_bytes % es == 0
        n = int(np.prod(shape)) if len(shape) else 1
        total = GUARD_BYTES * 2 + n * es + offset_bytes
        total += (-total) % es
        self.raw = torch.full((total,), SENTINEL, dtype=torch.uint8, device=device)
        start = GUARD_BYTES + offset_bytes
        self.lo, self.hi = start, start + n * es
        self.tensor = self.raw[self.lo:self.hi].view(dtype).view(shape)

    def check(self):
        r = self.raw.cpu()
        assert bool((r[: self.lo] == SENTINEL).all()), "write below the output buffer"
        assert bool((r[self.hi:] == SENTINEL).all()), "write above the output buffer"


def offset_copy(t: torch.Tensor, offset_bytes: int, device="cuda"):
    """A device copy of t whose data pointer is offset by offset_bytes from a
    256-byte-aligned allocation (offset a multiple of the element size)."""
    es = t.element_size()
    assert offset_bytes % es == 0
    n = t.numel()
    raw = torch.empty(n * es + offset_bytes + 256, dtype=torch.uint8, device=device)
    v = raw[offset_bytes: offset_bytes + n * es].view(t.dtype).view(t.shape)
    v.copy_(t.to(device))
    return raw, v
