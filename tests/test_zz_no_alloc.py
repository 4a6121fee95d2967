"""moe_route_noalloc: routing for callers that may not allocate device memory.

The entry point keeps its temporary buffers in a statically sized device
array instead of calling cudaMalloc.  Its outputs must equal the oracle's
routing (indices, counts, offsets, permutation and inverse bit for bit,
weights within the weight tolerance) and the context-based entry point's
(moe_layer_forward + moe_get_routing) on the same inputs, on consecutive calls
(the array is shared by every call and keeps the previous call's contents).
The cases reach the array's limits: 64 tokens, and 1024 experts (the largest
shared-memory configuration of the routing kernel).  This file runs last so
that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import workloads as W
from fp8_routed_expert_gb300 import C, lib
from harness import WTS_ATOL, DeviceWeights, make_layer, reference_threaded, x_dev

pytestmark = pytest.mark.gpu

# a router at the array's expert limit (E = 1024) with a small hidden size
E1024 = W.Family("route_e1024", 256, 1024, 8, 128, 7, (64,), bias_std=1.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _family(name):
    return E1024 if name == E1024.name else W.family(name)


def _noalloc(x, dw, fam, T, k):
    dev = torch.device("cuda", 0)
    out = dict(idx=torch.full((T, k), -1, dtype=torch.int32, device=dev),
               wts=torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
               counts=torch.full((fam.n_experts,), -1, dtype=torch.int32, device=dev),
               offsets=torch.full((fam.n_experts + 1,), -1, dtype=torch.int32, device=dev),
               perm=torch.full((T * k,), -1, dtype=torch.int32, device=dev),
               inv=torch.full((T * k,), -1, dtype=torch.int32, device=dev))
    bias = dw.router_bias.data_ptr() if dw.router_bias is not None else None
    rc = lib().moe_route_noalloc(x.data_ptr(), T, fam.hidden, dw.router_w.data_ptr(), bias,
                                 fam.n_experts, k, out["idx"].data_ptr(), out["wts"].data_ptr(),
                                 out["counts"].data_ptr(), out["offsets"].data_ptr(),
                                 out["perm"].data_ptr(), out["inv"].data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in out.items()}


def _same_routing(got, want, what):
    for n in ("idx", "counts", "offsets", "perm", "inv"):
        assert np.array_equal(got[n], want[n]), f"{n} differs from the {what}"
    err = np.abs(got["wts"].astype(np.float64) - want["wts"]).max()
    assert err <= WTS_ATOL, f"weights differ from the {what} by {err:.2e}"


@pytest.mark.parametrize("name,T", [("tiny", 3), ("olmoe_decode", 8), ("olmoe_prefill", 16),
                                    ("wide_decode", 64), ("route_e1024", 64)])
def test_noalloc_routing_matches_oracle_and_context_entry_point(name, T):
    fam = _family(name)
    w = W.make_weights(fam)
    dw = DeviceWeights(w)
    xb = W.make_x(fam, T)
    x = x_dev(xb)
    k = fam.top_k
    oracle_r = reference_threaded(xb, w, k, tokens=[])
    layer = make_layer(fam, T)
    layer.forward(x, *dw.args(), k)
    ctx_r = {n: t.cpu().numpy() for n, t in layer.routing(T, k).items()}
    assert layer.status() == 0
    for _ in range(2):  # the shared array keeps the previous call's contents
        got = _noalloc(x, dw, fam, T, k)
        _same_routing(got, oracle_r, "oracle")
        _same_routing(got, ctx_r, "context entry point")


def test_noalloc_rejects_sizes_beyond_its_array():
    fam = W.family("olmoe_decode")
    dw = DeviceWeights(W.make_weights(fam))
    x = x_dev(W.make_x(fam, 65))
    buf = torch.empty(65 * 64 * 8, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    rc = lib().moe_route_noalloc(x.data_ptr(), 65, fam.hidden, dw.router_w.data_ptr(), None,
                                 fam.n_experts, fam.top_k, p, p, p, p, p, p, None)
    assert rc == C["MOE_ERR_SHAPE"]
    rc = lib().moe_route_noalloc(x.data_ptr(), 8, fam.hidden, dw.router_w.data_ptr(), None,
                                 1025, fam.top_k, p, p, p, p, p, p, None)
    assert rc == C["MOE_ERR_SHAPE"]
