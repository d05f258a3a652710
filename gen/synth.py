"""Seeded synthetic inputs for the four epilogue ops.

This module is the one thing the CUDA path's tests/bench and the CPU oracle
share: it draws tensors and nothing else.  It holds none of the ops'
arithmetic (no sums, no normalisation, no exponentials); it only produces the
values that are fed to both sides.

Recipe (the same for every workload):
  * a fresh ``torch.Generator('cpu')`` seeded with ``seed`` (0 by default) at
    the start of each workload;
  * float32 draws on the CPU, in the op's argument order
    (SkipLayerNormalization: input, skip, gamma, beta, bias;
    BiasSoftmax: data, bias; BiasAdd: X, bias, skip; QuickGelu: X);
  * then a single cast to the op's element type T.  The T-typed CPU tensor is
    the single source of truth: the oracle reads it as float64, the GPU gets a
    byte copy of it.

N(m, s) below means mean m and standard deviation s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Attribute defaults printed by the op definitions:
#   com.microsoft.QuickGelu manifest, `attributes.alpha`            -> 1.702
#   com.microsoft.SkipLayerNormalization manifest, `attributes.epsilon`
#                                                                    -> 9.999999960041972e-13 (= float32(1e-12))
#   com.microsoft.BiasSoftmax manifest, `attributes.axis`            -> 1
DEFAULT_ALPHA = 1.702
DEFAULT_EPSILON = 9.999999960041972e-13
DEFAULT_AXIS = 1

# The additive-mask value of a masked attention position (exact in fp16).
MASKED = -10000.0


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(g: torch.Generator, shape, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def uniform(g: torch.Generator, shape, lo: float, hi: float) -> torch.Tensor:
    t = torch.rand(tuple(shape), generator=g, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def causal_mask(batch: int, q: int, k: int, dtype=torch.float32) -> torch.Tensor:
    """(batch, q, k) additive mask: 0 where key index <= query index, MASKED elsewhere."""
    keep = torch.ones(q, k, dtype=torch.bool).tril_()
    m = torch.full((q, k), MASKED, dtype=dtype)
    m.masked_fill_(keep, 0.0)
    return m.unsqueeze(0).expand(batch, q, k).contiguous()


# --------------------------------------------------------------------------
# per-op input builders (arbitrary shapes; used by tests at small sizes)
# --------------------------------------------------------------------------

def sln_inputs(in_shape, skip_shape=None, dtype="f32", has_beta=True, has_bias=False,
               seed=0, std=1.0, mean=0.0):
    """input, skip ~N(mean, std); gamma ~U(0.5, 1.5); beta, bias ~N(0, 0.1)."""
    T = DTYPES[dtype]
    g = _gen(seed)
    H = int(in_shape[-1])
    skip_shape = tuple(in_shape) if skip_shape is None else tuple(skip_shape)
    x = normal(g, in_shape, std, mean)
    sk = normal(g, skip_shape, std, mean)
    gamma = uniform(g, (H,), 0.5, 1.5)
    beta = normal(g, (H,), 0.1) if has_beta else None
    bias = normal(g, (H,), 0.1) if has_bias else None
    cast = lambda t: None if t is None else t.to(T)
    return dict(input=cast(x), skip=cast(sk), gamma=cast(gamma), beta=cast(beta),
                bias=cast(bias), epsilon=DEFAULT_EPSILON)


def bias_softmax_inputs(data_shape, bias_shape, dtype="f32", data_std=1.0, bias_std=1.0,
                        seed=0, causal=False):
    """data ~N(0, data_std); bias ~N(0, bias_std), or a causal 0/MASKED mask of
    shape (b, q, k) when ``causal``."""
    T = DTYPES[dtype]
    g = _gen(seed)
    data = normal(g, data_shape, data_std)
    if causal:
        b, q, k = bias_shape
        bias = causal_mask(b, q, k)
    else:
        bias = normal(g, bias_shape, bias_std)
    return dict(data=data.to(T), bias=bias.to(T))


def bias_add_inputs(shape, dtype="f32", seed=0, std=1.0, bias_std=0.1):
    T = DTYPES[dtype]
    g = _gen(seed)
    x = normal(g, shape, std)
    bias = normal(g, (shape[-1],), bias_std)
    skip = normal(g, shape, std)
    return dict(X=x.to(T), bias=bias.to(T), skip=skip.to(T))


def quick_gelu_inputs(numel, dtype="f32", seed=0, std=3.0):
    T = DTYPES[dtype]
    g = _gen(seed)
    return dict(X=normal(g, (int(numel),), std).to(T), alpha=DEFAULT_ALPHA)


def float32_bit_patterns(n: int, seed: int = 0) -> torch.Tensor:
    """n float32 values with uniformly random bit patterns, the non-finite ones
    dropped: every exponent (subnormals included) and both signs."""
    g = _gen(seed)
    bits = torch.randint(-(1 << 31), 1 << 31, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    x = bits.view(torch.float32)
    return x[torch.isfinite(x)].contiguous()


# --------------------------------------------------------------------------
# named workloads: the transformer-activation shapes the ops are measured on
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str          # what it is, with its sizes
    op: str            # skip_layer_norm | bias_softmax | bias_add | quick_gelu
    dtype: str         # f32 | f16
    build: object = field(repr=False, compare=False)
    attrs: dict = field(default_factory=dict, compare=False)


def _sln_small():
    return sln_inputs((2, 128, 768), None, "f32", has_beta=True, has_bias=False, seed=0)


def _sln_f16_residual():
    return sln_inputs((16384, 4096), None, "f16", has_beta=True, has_bias=True, seed=0)


def _sln_f32_broadcast():
    return sln_inputs((32, 2048, 1024), (1, 2048, 1024), "f32", has_beta=True,
                      has_bias=False, seed=0)


def _bias_add_f16():
    return bias_add_inputs((16, 1024, 4096), "f16", seed=0)


def _quick_gelu_f16():
    return quick_gelu_inputs(67_108_867, "f16", seed=0)


def _softmax_attention_f16():
    d = bias_softmax_inputs((32, 16, 512, 512), (32, 512, 512), "f16", data_std=4.0,
                            seed=0, causal=True)
    return d


def _softmax_long_cyclic():
    return bias_softmax_inputs((64, 1, 262144), (2, 1, 262144), "f32", data_std=2.0,
                               bias_std=1.0, seed=0)


def _softmax_long_single():
    return bias_softmax_inputs((8, 1048576), (1, 1048576), "f32", data_std=2.0,
                               bias_std=1.0, seed=0)


WORKLOADS = {
    w.name: w for w in [
        Workload("sln_f32_2x128x768", "skip_layer_norm", "f32", _sln_small,
                 dict(residual=False)),
        Workload("bias_add_f16_16x1024x4096", "bias_add", "f16", _bias_add_f16),
        Workload("quick_gelu_f16_67108867", "quick_gelu", "f16", _quick_gelu_f16),
        Workload("bias_softmax_f16_32x16x512x512_causal", "bias_softmax", "f16",
                 _softmax_attention_f16, dict(axis=3, is_inner_broadcast=1)),
        Workload("sln_f16_16384x4096_bias_residual", "skip_layer_norm", "f16",
                 _sln_f16_residual, dict(residual=True)),
        Workload("sln_f32_32x2048x1024_bcast_skip", "skip_layer_norm", "f32",
                 _sln_f32_broadcast, dict(residual=False)),
        Workload("bias_softmax_f32_64x262144_cyclic", "bias_softmax", "f32",
                 _softmax_long_cyclic, dict(axis=1, is_inner_broadcast=0)),
        Workload("bias_softmax_f32_8x1048576", "bias_softmax", "f32",
                 _softmax_long_single, dict(axis=1, is_inner_broadcast=0)),
    ]
}


def workload(name: str) -> dict:
    """Build a named workload's inputs (CPU, T-typed) plus its attributes."""
    w = WORKLOADS[name]
    d = w.build()
    d.update(w.attrs)
    return d


def device_normal(shape, dtype="f16", seed=0, std=1.0, device="cuda") -> torch.Tensor:
    """N(0, std) draws made on the device with a seeded generator, 2^26 at a
    time, then cast to T: for tensors too large to build on the host."""
    T = DTYPES[dtype]
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(tuple(shape), dtype=T, device=device)
    flat = out.view(-1)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = (torch.randn(n, generator=g, device=device, dtype=torch.float32) * std).to(T)
    return out


def sample_indices(n: int, k: int, seed: int = 1234) -> set:
    """About k distinct indices in [0, n), drawn without materialising a
    permutation (n may be in the billions)."""
    g = _gen(seed)
    return set(torch.randint(0, n, (k,), generator=g, dtype=torch.int64).tolist())


def sample_rows(n_rows: int, k: int, seed: int = 1234) -> list:
    """k distinct row indices in [0, n_rows), always including the first and last
    rows; used to check full-size outputs row by row against the oracle."""
    g = _gen(seed)
    k = min(k, n_rows)
    picks = set([0, n_rows - 1])
    if k > 2:
        extra = torch.randperm(n_rows, generator=g)[: k].tolist()
        for r in extra:
            if len(picks) >= k:
                break
            picks.add(int(r))
    return sorted(picks)


def numel(shape) -> int:
    return int(math.prod(int(s) for s in shape))
