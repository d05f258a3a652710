"""Plain CPU oracle for the four fused transformer-block epilogue ops.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference legs may import this module.  The library's
product path never calls it, and this module never imports the library.

Every function reads its T-typed inputs (float16 or float32 NumPy arrays),
converts them to float64 exactly, and evaluates the op's definition in
float64, one row chunk at a time (at most 2**20 elements per chunk) so that
memory stays bounded.  There is no blocking, fusion or reordering beyond what
the definitions state.  Each function cites the passage it follows, by the
manifest page's title and the manifest section.

Readings taken where the op definitions are silent (each is listed in the
repository's design notes as well):
  * LayerNorm variance is the population variance (divide by H).
  * epsilon is a float32 attribute: the oracle uses float64(float32(eps)).
  * alpha is a float32 attribute: the oracle uses float64(float32(alpha)).
  * The ``input_skip_bias_sum`` output is the sum evaluated in float32 in the
    op's stated order, ((input + skip) + bias), rounded once to T at the end.
  * BiasSoftmax adds data and bias exactly (no rounding to T in between).
  * BiasSoftmax bias rows: row r of the data uses bias row r // innerRepeat
    when is_inner_broadcast != 0 and r % biasBlockCount otherwise.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, hand-worked rows, invariants and
library special cases); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

CHUNK_ELEMS = 1 << 20

DEFAULT_EPSILON = 9.999999960041972e-13   # SkipLayerNormalization `attributes.epsilon`
DEFAULT_ALPHA = 1.702                     # QuickGelu `attributes.alpha`
DEFAULT_AXIS = 1                          # BiasSoftmax `attributes.axis`


def _is_bf16(a):
    return hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16"


def _np(a):
    """Accept NumPy arrays or CPU torch tensors; return a NumPy array.  A
    bfloat16 tensor (which NumPy has no type for) becomes float32, exactly."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if _is_bf16(a):
            a = a.float()
        a = a.numpy()
    return np.asarray(a)


def _rows_iter(n_rows, H, rows):
    """Yield (positions, row indices) chunks of at most CHUNK_ELEMS elements."""
    idx = np.arange(n_rows, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    step = max(1, CHUNK_ELEMS // max(1, H))
    for p in range(0, idx.size, step):
        yield slice(p, min(p + step, idx.size)), idx[p:p + step]


# ---------------------------------------------------------------------------
# SkipLayerNormalization
# ---------------------------------------------------------------------------

def skip_layer_norm(input, skip, gamma, beta=None, bias=None, epsilon=DEFAULT_EPSILON,
                    rows=None, simplified=False):
    """SkipLayerNormalization in float64.

    com.microsoft.SkipLayerNormalization manifest, `description`, `inputs`
    (skip shapes, optional beta/bias), `outputs` (input_skip_bias_sum) and
    `attributes.epsilon`:
      1. H = last dim; R = numel(input)/H rows; skipRows = numel(skip)/H; row r
         uses skip row r mod skipRows (exact, (1,S,H) or (S,H) skip all reduce
         to this).
      2. s = input + skip (+ bias), exact in float64.
      3. mu = mean(s); var = mean((s - mu)^2) (population).
      4. n = (s - mu) / sqrt(var + eps), eps = float64(float32(epsilon)).
      5. y = n * gamma (+ beta).
    ``simplified`` selects the RMS form that the manifest's ``simplified``
    shader flag names: no mean subtraction, n = s / sqrt(mean(s^2) + eps),
    y = n * gamma (+ beta).

    Returns a dict with ``output`` (float64, shape (len(rows) or R, H)),
    ``mean`` and ``inv_std_dev`` (float64 per row; mean is 0 when simplified).
    ``rows`` restricts the computation to the given row indices.
    """
    x = _np(input)
    sk = _np(skip)
    H = int(x.shape[-1])
    R = x.size // H
    skip_rows = sk.size // H
    x2 = x.reshape(R, H)
    sk2 = sk.reshape(skip_rows, H)
    g = _np(gamma).astype(np.float64).reshape(H)
    b = None if beta is None else _np(beta).astype(np.float64).reshape(H)
    bb = None if bias is None else _np(bias).astype(np.float64).reshape(H)
    eps = float(np.float32(epsilon))

    n_out = R if rows is None else len(rows)
    out = np.empty((n_out, H), dtype=np.float64)
    mean = np.empty(n_out, dtype=np.float64)
    inv_std = np.empty(n_out, dtype=np.float64)
    for pos, r in _rows_iter(R, H, rows):
        s = x2[r].astype(np.float64) + sk2[r % skip_rows].astype(np.float64)
        if bb is not None:
            s = s + bb
        if simplified:
            mu = np.zeros(s.shape[0])
            ms = np.mean(s * s, axis=1)
            rstd = 1.0 / np.sqrt(ms + eps)
            n = s * rstd[:, None]
        else:
            mu = np.mean(s, axis=1)
            d = s - mu[:, None]
            var = np.mean(d * d, axis=1)
            rstd = 1.0 / np.sqrt(var + eps)
            n = d * rstd[:, None]
        y = n * g
        if b is not None:
            y = y + b
        out[pos] = y
        mean[pos] = mu
        inv_std[pos] = rstd
    return dict(output=out, mean=mean, inv_std_dev=inv_std)


def skip_bias_sum(input, skip, bias=None, rows=None):
    """The ``input_skip_bias_sum`` output, as a T-typed array.

    com.microsoft.SkipLayerNormalization manifest, `outputs`
    (input_skip_bias_sum) and `inputs.bias` (bias "added to input + skip").
    Reading: the sum is evaluated in float32 in that order,
    f32(f32(input + skip) + bias), each step rounded to nearest-even, and the
    result is rounded once to T.  NumPy float32 arithmetic is IEEE
    round-to-nearest-even, so it states the rounding exactly.  For bfloat16
    the final rounding is torch's float32 -> bfloat16 conversion (also
    nearest-even) and the result is a bfloat16 torch tensor.
    """
    bf16 = _is_bf16(input)
    x = _np(input)
    sk = _np(skip)
    T = x.dtype
    H = int(x.shape[-1])
    R = x.size // H
    skip_rows = sk.size // H
    x2 = x.reshape(R, H)
    sk2 = sk.reshape(skip_rows, H)
    bb = None if bias is None else _np(bias).astype(np.float32).reshape(H)
    n_out = R if rows is None else len(rows)
    out = np.empty((n_out, H), dtype=T)
    for pos, r in _rows_iter(R, H, rows):
        s = x2[r].astype(np.float32) + sk2[r % skip_rows].astype(np.float32)
        if bb is not None:
            s = s + bb
        out[pos] = s.astype(T)
    if bf16:
        import torch
        return torch.from_numpy(out).to(torch.bfloat16)
    return out


# ---------------------------------------------------------------------------
# BiasSoftmax
# ---------------------------------------------------------------------------

def bias_softmax_dims(shape, bias_numel, axis=DEFAULT_AXIS):
    """`derive` block of the com.microsoft.BiasSoftmax manifest:
    axisNorm, batchCount (product of dims before axisNorm), blockSize (product
    from axisNorm on), biasBlockCount = numel(bias)/blockSize, innerRepeat =
    batchCount / biasBlockCount, and whether `biasContract` holds."""
    rank = len(shape)
    axis_n = axis if axis >= 0 else axis + rank
    if not (0 <= axis_n < rank):
        raise ValueError("axis out of range")
    batch = int(math.prod(shape[:axis_n]))
    block = int(math.prod(shape[axis_n:]))
    numel = batch * block
    bias_rows = bias_numel // max(1, block)
    ok = (numel == 0 and bias_numel == 0) or (
        block > 0 and bias_rows > 0 and bias_numel % block == 0
        and bias_rows <= batch and batch % bias_rows == 0)
    inner_repeat = max(1, batch // max(1, bias_rows))
    return dict(axis=axis_n, batch=batch, block=block, bias_rows=bias_rows,
                inner_repeat=inner_repeat, contract_ok=bool(ok))


def bias_row_of(r, bias_rows, inner_repeat, is_inner_broadcast):
    """Bias row used by data row r (com.microsoft.BiasSoftmax manifest,
    `description` and `attributeDescriptions.is_inner_broadcast`: consecutive
    groups of innerRepeat rows share a bias row for inner broadcast; the bias
    rows repeat cyclically for outer broadcast)."""
    r = np.asarray(r, dtype=np.int64)
    if is_inner_broadcast:
        return r // inner_repeat
    return r % bias_rows


def bias_softmax(data, bias, axis=DEFAULT_AXIS, is_inner_broadcast=0, rows=None):
    """softmax(data + bias) over the flattened suffix from ``axis``, in float64.

    com.microsoft.BiasSoftmax manifest, `description`, `derive` and
    `attributeDescriptions`.  z = data[r] + bias[bias_row_of(r)] (exact),
    m = max z, y = exp(z - m) / sum(exp(z - m)).  Returns (len(rows) or
    batchCount, blockSize) float64.
    """
    d = _np(data)
    bs = _np(bias)
    dims = bias_softmax_dims(d.shape, bs.size, axis)
    if not dims["contract_ok"]:
        raise ValueError("biasContract violated")
    batch, block = dims["batch"], dims["block"]
    n_out = batch if rows is None else len(rows)
    out = np.empty((n_out, block), dtype=np.float64)
    if d.size == 0:
        return out
    d2 = d.reshape(batch, block)
    b2 = bs.reshape(dims["bias_rows"], block)
    for pos, r in _rows_iter(batch, block, rows):
        br = bias_row_of(r, dims["bias_rows"], dims["inner_repeat"], is_inner_broadcast)
        z = d2[r].astype(np.float64) + b2[br].astype(np.float64)
        m = np.max(z, axis=1)
        e = np.exp(z - m[:, None])
        out[pos] = e / np.sum(e, axis=1)[:, None]
    return out


# ---------------------------------------------------------------------------
# BiasAdd
# ---------------------------------------------------------------------------

def _two_sum(a, b):
    """Knuth's TwoSum in float64: s = fl(a + b) and its rounding error e, so
    that a + b = s + e exactly (no overflow for the operand types here)."""
    s = a + b
    bb = s - a
    e = (a - (s - bb)) + (b - bb)
    return s, e


def bias_add(X, bias, skip):
    """Y = X + bias[c] + skip over (N, S, C): the exact sum, rounded to float64.

    com.microsoft.BiasAdd manifest, `description` and `inputs`: bias is
    broadcast over the channel (last) dimension, then the residual is added.
    A plain float64 sum is exact for fp16 terms but not for fp32 or bf16 ones
    whose exponents differ by more than 53 bits, and where the skip then
    cancels a term only that rounding error is left.  So the sum is formed as
    an error-free expansion (TwoSum twice): x + b = s1 + e1 and
    s1 + skip = s2 + e2 exactly; y = s2 + (e1 + e2) is within two float64
    roundings of the exact sum, cancellation or not.  Non-finite sums are the
    plain float64 ones.
    """
    x = _np(X).astype(np.float64)
    b = _np(bias).astype(np.float64)
    s = _np(skip).astype(np.float64)
    C = x.shape[-1]
    b = np.broadcast_to(b.reshape((1,) * (x.ndim - 1) + (C,)), x.shape)
    with np.errstate(invalid="ignore"):
        s1, e1 = _two_sum(x, b)
        s2, e2 = _two_sum(s1, s)
        y = s2 + (e1 + e2)
    return np.where(np.isfinite(s2), y, s2)


# ---------------------------------------------------------------------------
# QuickGelu
# ---------------------------------------------------------------------------

def quick_gelu(X, alpha=DEFAULT_ALPHA):
    """y = x * sigmoid(alpha * x) in float64, alpha = float64(float32(alpha)).

    com.microsoft.QuickGelu manifest, `description` and `attributes.alpha`.
    sigmoid(t) = 1/(1+exp(-t)) for t >= 0 and exp(t)/(1+exp(t)) for t < 0
    (the same function; the second form avoids overflow of exp(-t)).
    """
    x = _np(X).astype(np.float64)
    a = float(np.float32(alpha))
    out = np.empty(x.shape, dtype=np.float64)
    flat_x = x.reshape(-1)
    flat_o = out.reshape(-1)
    for p in range(0, flat_x.size, CHUNK_ELEMS):
        xs = flat_x[p:p + CHUNK_ELEMS]
        t = a * xs
        sig = np.empty_like(t)
        with np.errstate(over="ignore", invalid="ignore"):
            pos = t >= 0
            sig[pos] = 1.0 / (1.0 + np.exp(-t[pos]))
            et = np.exp(t[~pos])
            sig[~pos] = et / (1.0 + et)
            flat_o[p:p + CHUNK_ELEMS] = xs * sig
    return out
