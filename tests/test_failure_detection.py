"""Failure detection on the GPU without a fault: a bounded device-side wait
runs out (nothing arrives on its mbarrier, nothing increments its counter),
the kernel records a timeout and returns, and the context stays usable."""
import numpy as np
import pytest
import torch

import workloads as W
from fp8_routed_expert_gb300 import C, lib
from harness import DeviceWeights, check_output, check_routing, make_layer, reference, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("path", ["tcgemv", "gemm"])
def test_wait_that_runs_out_is_reported_and_the_context_recovers(path):
    fam = W.family("olmoe_decode")
    w = W.make_weights(fam)
    dw = DeviceWeights(w)
    T, k = 8, fam.top_k
    layer = make_layer(fam, T)
    which = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    limit_ns = 1_000_000  # 1 ms per wait
    a.record(s)
    rc = lib().moe_selftest_wait_timeout(layer.handle, limit_ns, which.data_ptr(), s.cuda_stream)
    b.record(s)
    assert rc == 0
    torch.cuda.synchronize()
    assert which.item() == 3, "both waits (mbarrier and counter) must give up"
    assert a.elapsed_time(b) >= 2 * limit_ns / 1e6 * 0.99, "the waits ended before their limit"
    assert layer.status() == C["MOE_ERR_DEVICE_TIMEOUT"]
    assert layer.status() == C["MOE_OK"]  # reported once, then cleared
    # the same context still computes the layer (its tensor memory was freed)
    x = W.make_x(fam, T)
    out, r = run(layer, x, dw, k, path)
    ref = reference(x, w, k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_selftest_argument_errors():
    fam = W.family("tiny")
    layer = make_layer(fam, 4)
    assert lib().moe_selftest_wait_timeout(layer.handle, 0, None, None) == C["MOE_ERR_ARG"]
    assert lib().moe_selftest_wait_timeout(layer.handle, 2_000_000_000, None, None) == C["MOE_ERR_ARG"]
    buf = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert lib().moe_selftest_wait_timeout(layer.handle, 1000, buf.data_ptr() + 2, None) == \
        C["MOE_ERR_ALIGN"]
