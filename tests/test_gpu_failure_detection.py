"""Failure detection on the GPU without faulting it: the staged kernels'
shared-memory barrier waits are bounded, a wait that runs out is counted, and
the kernel returns with nothing left in flight.  The self-test makes one such
wait run out on purpose (a barrier armed for bytes no copy delivers) with a
short limit; nothing here traps, faults or hangs the device."""
import time

import pytest
import torch

import oracle
from gen import synth
from tests._helpers import assert_norm_close

pytestmark = pytest.mark.gpu


def test_normal_calls_count_no_timeouts(lib):
    lib.ep_pipeline_timeouts(clear=True)
    d = synth.sln_inputs((512, 4096), None, "f16", has_beta=True, has_bias=True, seed=0)
    lib.ep_skip_layer_norm(d["input"].cuda(), d["skip"].cuda(), d["gamma"].cuda(), d["beta"].cuda(),
                           d["bias"].cuda(), input_skip_bias_sum=True)
    sm = synth.bias_softmax_inputs((4096, 512), (256, 512), "f16", seed=0)
    lib.ep_bias_softmax(sm["data"].cuda(), sm["bias"].cuda(), axis=1, is_inner_broadcast=1)
    lg = synth.bias_softmax_inputs((4, 100000), (1, 100000), "f32", seed=0)
    lib.ep_bias_softmax(lg["data"].cuda(), lg["bias"].cuda(), axis=1, is_inner_broadcast=0)
    x = synth.quick_gelu_inputs(1 << 22, "f16", seed=0)["X"].cuda()
    lib.ep_quick_gelu(x)
    assert lib.ep_pipeline_timeouts() == 0


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_selftest_wait_runs_out_and_returns(lib, limit_us):
    lib.ep_pipeline_timeouts(clear=True)
    t0 = time.perf_counter()
    seen = lib.ep_selftest_bounded_wait(limit_us)
    elapsed = time.perf_counter() - t0
    assert seen == 1
    assert elapsed >= limit_us * 1e-6 * 0.9        # it did wait for the limit
    assert elapsed < limit_us * 1e-6 + 5.0         # and came back
    assert lib.ep_pipeline_timeouts(clear=True) == 1
    # the context is still usable: a normal call after the self-test is correct
    d = synth.bias_softmax_inputs((64, 512), (4, 512), "f32", seed=3)
    out = lib.ep_bias_softmax(d["data"].cuda(), d["bias"].cuda(), axis=1, is_inner_broadcast=1)
    torch.cuda.synchronize()
    assert_norm_close(out.cpu(), oracle.bias_softmax(d["data"], d["bias"], 1, 1), torch.float32)
    assert lib.ep_pipeline_timeouts() == 0


def test_selftest_on_a_side_stream(lib):
    s = torch.cuda.Stream()
    assert lib.ep_selftest_bounded_wait(1000, stream=s) == 1
    lib.ep_pipeline_timeouts(clear=True)
