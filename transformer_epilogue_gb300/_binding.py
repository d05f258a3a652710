"""Thin ctypes binding of the C ABI declared in ``include/ep.h``.

Argument marshalling only: every function here checks that its tensors are
contiguous CUDA tensors, allocates outputs the caller did not pass (PyTorch is
the allocator), and calls the C entry point of the same name on the current
CUDA stream.  All computation happens in the library's CUDA kernels; there is
no CPU or PyTorch fallback.  A non-OK status raises ``EpError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libtransformer_epilogue.so")

EP_F32, EP_F16, EP_BF16 = 0, 1, 2
EP_OK, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_WORKSPACE, EP_ERR_CUDA = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "EP_OK", 1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_UNSUPPORTED", 3: "EP_ERR_WORKSPACE",
                4: "EP_ERR_CUDA"}

# Attribute defaults of the op definitions (manifest `attributes` sections).
DEFAULT_EPSILON = 9.999999960041972e-13   # SkipLayerNormalization
DEFAULT_ALPHA = 1.702                     # QuickGelu
DEFAULT_AXIS = 1                          # BiasSoftmax

_TORCH_TO_EP = {torch.float32: EP_F32, torch.float16: EP_F16, torch.bfloat16: EP_BF16}

_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p

# name -> (restype, argtypes)
_SIGNATURES = {
    "ep_last_error": (ctypes.c_char_p, []),
    "ep_status_name": (ctypes.c_char_p, [ctypes.c_int]),
    "ep_kernel_launch_count": (ctypes.c_uint64, []),
    "ep_abi_version": (ctypes.c_int, []),
    "ep_pipeline_timeouts": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]),
    "ep_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint64), _vp]),
    "ep_skip_layer_norm": (ctypes.c_int, [ctypes.c_int, _vp, _i64p, ctypes.c_int, _vp, _i64p, ctypes.c_int,
                                          _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp]),
    "ep_skip_layer_norm_ex": (ctypes.c_int, [ctypes.c_int, _vp, _i64p, ctypes.c_int, _vp, _i64p, ctypes.c_int,
                                             _vp, _vp, _vp, ctypes.c_float, ctypes.c_int, _vp, _vp, _vp, _vp,
                                             _vp]),
    "ep_bias_softmax": (ctypes.c_int, [ctypes.c_int, _vp, _i64p, ctypes.c_int, _vp, ctypes.c_int64,
                                       ctypes.c_int, ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp]),
    "ep_bias_softmax_workspace_size": (ctypes.c_size_t, [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int]),
    "ep_bias_softmax_noalloc": (ctypes.c_int, [ctypes.c_int, _vp, _i64p, ctypes.c_int, _vp, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_int, _vp, _vp]),
    "ep_bias_add": (ctypes.c_int, [ctypes.c_int, _vp, _i64p, _vp, _vp, _vp, _vp]),
    "ep_quick_gelu": (ctypes.c_int, [ctypes.c_int, _vp, ctypes.c_int64, ctypes.c_float, _vp, _vp]),
}


class EpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load the C-ABI library (built by ``__graft_entry__.build()`` or
    ``python -m transformer_epilogue_gb300.build``).  Raises if it is missing:
    there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} is missing "
                          "(run `python -m transformer_epilogue_gb300.build`)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def raw():
    """The loaded ctypes library (for pointer-level calls)."""
    return load_library()


def _check(status: int):
    if status != EP_OK:
        msg = load_library().ep_last_error().decode(errors="replace")
        raise EpError(status, msg)


def _shape(dims) -> ctypes.Array:
    dims = [int(d) for d in dims]
    return (ctypes.c_int64 * max(1, len(dims)))(*dims)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _TORCH_TO_EP[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _cuda(name, t, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kernel_launch_count() -> int:
    return int(load_library().ep_kernel_launch_count())


def ep_pipeline_timeouts(clear=False) -> int:
    """Bounded-wait timeouts the staged kernels counted on the current device
    (synchronises with the device)."""
    n = ctypes.c_uint64(0)
    _check(load_library().ep_pipeline_timeouts(ctypes.byref(n), int(bool(clear))))
    return int(n.value)


def ep_selftest_bounded_wait(timeout_us=5000, stream=None) -> int:
    """Run the failure-detection self-test; returns the timed-out waits counted
    meanwhile (1 when the mechanism works)."""
    n = ctypes.c_uint64(0)
    _check(load_library().ep_selftest_bounded_wait(int(timeout_us), ctypes.byref(n),
                                                   _stream(stream, torch.cuda.current_device())))
    return int(n.value)


def ep_skip_layer_norm(input, skip, gamma, beta=None, bias=None, epsilon=DEFAULT_EPSILON, output=None,
                       input_skip_bias_sum=None, stream=None):
    """SkipLayerNormalization.  ``input_skip_bias_sum``: a tensor to fill, True
    to allocate one, or None.  Returns (output, input_skip_bias_sum or None)."""
    lib = load_library()
    for n, t in (("input", input), ("skip", skip), ("gamma", gamma)):
        _cuda(n, t)
    _cuda("beta", beta, True)
    _cuda("bias", bias, True)
    if output is None:
        output = torch.empty_like(input)
    _cuda("output", output)
    if input_skip_bias_sum is True:
        input_skip_bias_sum = torch.empty_like(input)
    elif input_skip_bias_sum is False:
        input_skip_bias_sum = None
    _cuda("input_skip_bias_sum", input_skip_bias_sum, True)
    st = lib.ep_skip_layer_norm(_dtype(input), _ptr(input), _shape(input.shape), input.dim(),
                                _ptr(skip), _shape(skip.shape), skip.dim(),
                                _ptr(gamma), _ptr(beta), _ptr(bias), float(epsilon),
                                _ptr(output), _ptr(input_skip_bias_sum), _stream(stream, input.device))
    _check(st)
    return output, input_skip_bias_sum


def ep_skip_layer_norm_ex(input, skip, gamma, beta=None, bias=None, epsilon=DEFAULT_EPSILON, simplified=False,
                          output=None, input_skip_bias_sum=None, mean=None, inv_std_dev=None, stream=None):
    """SkipLayerNormalization with the RMS form (``simplified``) and the
    per-row float32 statistics.  ``mean`` / ``inv_std_dev``: tensors to fill,
    True to allocate, or None.  Returns (output, input_skip_bias_sum, mean,
    inv_std_dev), the last three None when not requested."""
    lib = load_library()
    for n, t in (("input", input), ("skip", skip), ("gamma", gamma)):
        _cuda(n, t)
    _cuda("beta", beta, True)
    _cuda("bias", bias, True)
    if output is None:
        output = torch.empty_like(input)
    _cuda("output", output)
    if input_skip_bias_sum is True:
        input_skip_bias_sum = torch.empty_like(input)
    elif input_skip_bias_sum is False:
        input_skip_bias_sum = None
    _cuda("input_skip_bias_sum", input_skip_bias_sum, True)
    rows = input.numel() // max(1, input.shape[-1])
    stat_shape = tuple(input.shape[:-1]) + (1,)
    if mean is True:
        mean = torch.empty(stat_shape, dtype=torch.float32, device=input.device)
    if inv_std_dev is True:
        inv_std_dev = torch.empty(stat_shape, dtype=torch.float32, device=input.device)
    for n, t in (("mean", mean), ("inv_std_dev", inv_std_dev)):
        _cuda(n, t, True)
        if t is not None and (t.dtype != torch.float32 or t.numel() != rows):
            raise ValueError(f"{n} must be a float32 tensor of {rows} elements")
    st = lib.ep_skip_layer_norm_ex(_dtype(input), _ptr(input), _shape(input.shape), input.dim(),
                                   _ptr(skip), _shape(skip.shape), skip.dim(),
                                   _ptr(gamma), _ptr(beta), _ptr(bias), float(epsilon), int(bool(simplified)),
                                   _ptr(output), _ptr(input_skip_bias_sum), _ptr(mean), _ptr(inv_std_dev),
                                   _stream(stream, input.device))
    _check(st)
    return output, input_skip_bias_sum, mean, inv_std_dev


def ep_bias_softmax_workspace_size(dtype, shape, axis=DEFAULT_AXIS) -> int:
    lib = load_library()
    code = _TORCH_TO_EP[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(lib.ep_bias_softmax_workspace_size(code, _shape(shape), len(shape), int(axis)))


def ep_bias_softmax(data, bias, axis=DEFAULT_AXIS, is_inner_broadcast=None, output=None, workspace=None,
                    stream=None):
    """BiasSoftmax.  ``is_inner_broadcast`` is required (the op definition has
    no default for it).  A workspace is allocated when the split-row path needs
    one and none is passed.  Returns output."""
    if is_inner_broadcast is None:
        raise ValueError("is_inner_broadcast is required")
    lib = load_library()
    _cuda("data", data)
    _cuda("bias", bias)
    if output is None:
        output = torch.empty_like(data)
    _cuda("output", output)
    need = ep_bias_softmax_workspace_size(data.dtype, data.shape, axis) if data.dtype in _TORCH_TO_EP else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=data.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.ep_bias_softmax(_dtype(data), _ptr(data), _shape(data.shape), data.dim(), _ptr(bias),
                             int(bias.numel()), int(axis), int(is_inner_broadcast), _ptr(output),
                             _ptr(workspace), wbytes, _stream(stream, data.device))
    _check(st)
    return output


def ep_bias_softmax_noalloc(data, bias, axis=DEFAULT_AXIS, is_inner_broadcast=None, output=None, stream=None):
    """BiasSoftmax for callers that cannot allocate device memory: the
    split-row scratch comes from a fixed 1 MiB array inside the library
    (rows * ceil(blockSize / chunk) <= 131072 when blockSize > 16384, chunk =
    4096 for float32, 8192 for float16/bfloat16).  Calls
    that may overlap on the GPU share that array and must be ordered by the
    caller.  Pass ``output`` to keep the call free of allocations (otherwise
    PyTorch allocates it here).  Returns output."""
    if is_inner_broadcast is None:
        raise ValueError("is_inner_broadcast is required")
    lib = load_library()
    _cuda("data", data)
    _cuda("bias", bias)
    if output is None:
        output = torch.empty_like(data)
    _cuda("output", output)
    st = lib.ep_bias_softmax_noalloc(_dtype(data), _ptr(data), _shape(data.shape), data.dim(), _ptr(bias),
                                     int(bias.numel()), int(axis), int(is_inner_broadcast), _ptr(output),
                                     _stream(stream, data.device))
    _check(st)
    return output


def ep_bias_add(X, bias, skip, Y=None, stream=None):
    """BiasAdd on (N, S, C) tensors.  Returns Y."""
    lib = load_library()
    for n, t in (("X", X), ("bias", bias), ("skip", skip)):
        _cuda(n, t)
    if X.dim() != 3:
        raise ValueError("X must have rank 3 (N, S, C)")
    if tuple(skip.shape) != tuple(X.shape) or bias.numel() != X.shape[2] or bias.dim() != 1:
        raise ValueError("skip must match X and bias must have C elements")
    if Y is None:
        Y = torch.empty_like(X)
    _cuda("Y", Y)
    if tuple(Y.shape) != tuple(X.shape):
        raise ValueError("Y must match X")
    st = lib.ep_bias_add(_dtype(X), _ptr(X), _shape(X.shape), _ptr(bias), _ptr(skip), _ptr(Y),
                         _stream(stream, X.device))
    _check(st)
    return Y


def ep_quick_gelu(X, alpha=DEFAULT_ALPHA, Y=None, stream=None):
    """QuickGelu over all elements of X.  Returns Y."""
    lib = load_library()
    _cuda("X", X)
    if Y is None:
        Y = torch.empty_like(X)
    _cuda("Y", Y)
    if Y.numel() != X.numel():
        raise ValueError("Y must have as many elements as X")
    st = lib.ep_quick_gelu(_dtype(X), _ptr(X), int(X.numel()), float(alpha), _ptr(Y), _stream(stream, X.device))
    _check(st)
    return Y
