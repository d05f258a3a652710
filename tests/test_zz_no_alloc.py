"""ep_bias_softmax_noalloc: the BiasSoftmax entry point for callers that cannot
allocate device memory (an engine or plugin whose device memory is all reserved
at start-up, code inside an allocator callback, or a loop that cannot afford
the synchronisation cudaMalloc may cause).  Its split-row scratch is a fixed
array inside the library instead of a caller-provided workspace.

Two calls in a row, on different shapes, must each match the workspace entry
point ep_bias_softmax within the usual BiasSoftmax tolerance; the second call
runs on scratch still holding the first call's statistics.  (Shapes beyond
the fixed scratch are rejected before anything is enqueued; that host-side
check is covered without a GPU in tests/abi_host_cases.py.)  This file is
collected last so that a failure here comes after every other test has run.
"""
import pytest
import torch

from gen import synth
from tests._helpers import assert_norm_close, to_np64

pytestmark = pytest.mark.gpu

CASES = [
    # (data shape, bias shape, dtype, is_inner_broadcast): both take the split-row path
    ((64, 1, 262144), (2, 1, 262144), "f32", 0),
    ((6, 40000), (3, 40000), "f16", 1),
]


def test_noalloc_matches_workspace_entry_point_twice(lib):
    for data_shape, bias_shape, dtype, inner in CASES:
        d = synth.bias_softmax_inputs(data_shape, bias_shape, dtype, data_std=2.0, seed=len(data_shape))
        assert lib.ep_bias_softmax_workspace_size(d["data"].dtype, data_shape, 1) > 0
        data, bias = d["data"].cuda(), d["bias"].cuda()
        want = lib.ep_bias_softmax(data, bias, axis=1, is_inner_broadcast=inner)
        got = torch.full_like(data, float("nan"))
        n0 = lib.kernel_launch_count()
        lib.ep_bias_softmax_noalloc(data, bias, axis=1, is_inner_broadcast=inner, output=got)
        torch.cuda.synchronize()
        assert lib.kernel_launch_count() > n0
        rows = data.numel() // data_shape[-1]
        assert_norm_close(got.reshape(rows, -1), to_np64(want.reshape(rows, -1)), data.dtype)

