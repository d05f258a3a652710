"""Comparison rules and guard-band canaries shared by the GPU parity tests.

Tolerances (written out here, applied element by element):
  * float32 SkipLayerNormalization / BiasSoftmax: |gpu - o| <= 1e-5.
  * float32 BiasAdd / QuickGelu: |gpu - o| <= 1e-6 * |o| + 2**-149.
  * float16, every op: |gpu - o| <= max(2e-3, ulp16(o)), where ulp16(o) is the
    float16 spacing at |o| (2**(floor(log2|o|) - 10), at least 2**-24).  For
    |o| < 4 this is the literal 2e-3; above it, correct rounding alone can err
    by half a float16 spacing, which exceeds 2e-3 once |o| >= 8.
  * bfloat16: |gpu - o| <= ulp_bf16(o), the bfloat16 spacing at |o|
    (2**(floor(log2|o|) - 7), at least 2**-133): correct rounding (half a
    spacing) plus the float32 arithmetic's error; for LayerNorm / softmax
    outputs at least the float32 bound 1e-5, because where gamma*n cancels beta
    the float32 arithmetic's own error (a few float32 ulps of the terms) is
    larger than a bfloat16 spacing at the near-zero result.
  * the input_skip_bias_sum output and broadcast row indexing: bit-exact.
``o`` is always the oracle's unrounded float64 value.
"""
import numpy as np
import torch

F32_ABS = 1e-5
F32_REL = 1e-6
F16_ABS = 2e-3
TINY = 2.0 ** -149


def ulp16(o):
    a = np.abs(o)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(2.0 ** (e - 10), 2.0 ** -24)


def ulp_bf16(o):
    a = np.abs(o)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(2.0 ** (e - 7), 2.0 ** -133)


def to_np64(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def _low_tol(o, dtype, norm):
    if dtype == torch.bfloat16:
        return np.maximum(ulp_bf16(o), F32_ABS) if norm else ulp_bf16(o)
    return np.maximum(F16_ABS, ulp16(o))


def _report(bad, gpu, o, what):
    idx = np.argwhere(bad)[:5]
    rows = [(tuple(int(j) for j in i), float(gpu[tuple(i)]), float(o[tuple(i)])) for i in idx]
    return f"{what}: {int(bad.sum())} elements out of tolerance, first: {rows}"


def assert_norm_close(gpu: torch.Tensor, o: np.ndarray, dtype):
    """LayerNorm / softmax outputs."""
    g = to_np64(gpu).reshape(o.shape)
    both_nan = np.isnan(g) & np.isnan(o)
    if dtype == torch.float32:
        tol = np.full(o.shape, F32_ABS)
    else:
        tol = _low_tol(o, dtype, norm=True)
    bad = ~both_nan & ~(np.abs(g - o) <= tol)
    assert not bad.any(), _report(bad, g, o, "norm/softmax")
    return float(np.nanmax(np.abs(g - o))) if o.size else 0.0


def assert_elementwise_close(gpu: torch.Tensor, o: np.ndarray, dtype):
    """BiasAdd / QuickGelu outputs."""
    g = to_np64(gpu).reshape(o.shape)
    both_nan = np.isnan(g) & np.isnan(o)
    same_inf = np.isinf(o) & (g == o)
    if dtype == torch.float32:
        with np.errstate(invalid="ignore"):
            tol = F32_REL * np.abs(o) + TINY
    else:
        tol = _low_tol(o, dtype, norm=False)
    with np.errstate(invalid="ignore"):
        bad = ~both_nan & ~same_inf & ~(np.abs(g - o) <= tol)
    assert not bad.any(), _report(bad, g, o, "elementwise")
    fin = np.isfinite(o)
    return float(np.max(np.abs(g[fin] - o[fin]))) if fin.any() else 0.0


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
