"""Tensors past 2^31 elements: every offset must be computed in 64 bits.

Inputs are drawn on the device (gen/synth.device_normal); outputs are checked
against the oracle on sampled elements or rows, always including those on
both sides of element 2^31 and the last ones.
"""
import pytest
import torch

import oracle
from gen import synth
from tests import test_gpu_elementwise as ew
from tests._helpers import assert_bit_exact, assert_norm_close

pytestmark = pytest.mark.gpu

E31 = 1 << 31


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _rows_to_check(n_rows, row_len, seed):
    """Sampled rows, the first and last ones, and those holding elements near 2^31."""
    r31 = E31 // row_len
    picks = synth.sample_indices(n_rows, 24, seed)
    picks |= {0, 1, n_rows - 2, n_rows - 1} | {r for r in range(r31 - 2, r31 + 3) if 0 <= r < n_rows}
    return torch.tensor(sorted(picks), dtype=torch.int64)


def test_quick_gelu_past_2_31_elements(lib):
    n = E31 + 37
    x = synth.device_normal((n,), "f16", seed=61, std=3.0)
    y = torch.empty_like(x)
    lib.ep_quick_gelu(x, 1.702, Y=y)
    idx = synth.sample_indices(n, 1 << 16, seed=62)
    idx |= set(range(0, 1024)) | set(range(E31 - 4096, n))
    idx = torch.tensor(sorted(idx), dtype=torch.int64, device="cuda")
    ew.check_quick_gelu(y[idx].cpu(), x[idx].cpu(), 1.702)


def test_bias_add_past_2_31_elements(lib):
    N, S, C = 8, 65537, 4104                      # 2,151,710,592 elements
    x = synth.device_normal((N, S, C), "f16", seed=63)
    s = synth.device_normal((N, S, C), "f16", seed=64)
    b = synth.device_normal((C,), "f16", seed=65, std=0.1)
    y = torch.empty_like(x)
    lib.ep_bias_add(x, b, s, Y=y)
    rows = _rows_to_check(N * S, C, seed=66).cuda()
    xr, sr, yr = (t.view(-1, C)[rows].cpu() for t in (x, s, y))
    k = rows.numel()
    ew.check_bias_add(yr.view(1, k, C), xr.view(1, k, C), b.cpu(), sr.view(1, k, C))


def test_skip_layer_norm_past_2_31_elements(lib):
    R, H = E31 // 4096 + 1, 4096                  # 524,289 rows
    x = synth.device_normal((R, H), "f16", seed=67)
    sk = synth.device_normal((R, H), "f16", seed=68)
    g = (synth.device_normal((H,), "f16", seed=69, std=0.1).float() + 1.0).half()
    bt = synth.device_normal((H,), "f16", seed=70, std=0.1)
    bi = synth.device_normal((H,), "f16", seed=71, std=0.1)
    out, res = torch.empty_like(x), torch.empty_like(x)
    lib.ep_skip_layer_norm(x, sk, g, bt, bi, 1e-5, output=out, input_skip_bias_sum=res)
    rows = _rows_to_check(R, H, seed=72).cuda()
    xr, sr = x[rows].cpu(), sk[rows].cpu()
    want = oracle.skip_layer_norm(xr, sr, g.cpu(), bt.cpu(), bi.cpu(), 1e-5)["output"]
    assert_norm_close(out[rows].cpu(), want, torch.float16)
    assert_bit_exact(res[rows].cpu(), oracle.skip_bias_sum(xr, sr, bi.cpu()))


def test_bias_softmax_rows_past_2_31_elements(lib):
    R, C, BR = E31 // 4096 + 8, 4096, 8            # 524,296 rows (a multiple of BR)
    d = synth.device_normal((R, C), "f16", seed=73, std=3.0)
    b = synth.device_normal((BR, C), "f16", seed=74)
    y = torch.empty_like(d)
    lib.ep_bias_softmax(d, b, axis=1, is_inner_broadcast=0, output=y)
    rows = _rows_to_check(R, C, seed=75)
    dr = d[rows.cuda()].cpu()
    br = b.cpu()[rows % BR]                        # outer map: row r uses bias row r mod BR
    assert_norm_close(y[rows.cuda()].cpu(), oracle.bias_softmax(dr, br, axis=1, is_inner_broadcast=0), torch.float16)


def test_bias_softmax_split_rows_past_2_31_elements(lib):
    R, C = 2049, 1 << 20                           # 2,148,532,224 elements, split-row path
    d = synth.device_normal((R, C), "f16", seed=76, std=2.0)
    b = synth.device_normal((1, C), "f16", seed=77)
    y = torch.empty_like(d)
    ws = torch.empty(lib.ep_bias_softmax_workspace_size(torch.float16, (R, C), 1), dtype=torch.uint8, device="cuda")
    lib.ep_bias_softmax(d, b, axis=1, is_inner_broadcast=0, output=y, workspace=ws)
    rows = torch.tensor(sorted({0, 1, 1023, 2047, 2048} | synth.sample_indices(R, 4, seed=78)), dtype=torch.int64)
    dr = d[rows.cuda()].cpu()
    br = b.cpu().expand(rows.numel(), C)
    assert_norm_close(y[rows.cuda()].cpu(), oracle.bias_softmax(dr, br, axis=1, is_inner_broadcast=0), torch.float16)
