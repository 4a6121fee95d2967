"""FP4 (NVFP4) experts: the CUDA path against the FP4 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import nvfp4 as F
from harness import (check_expert_y, check_output, check_routing, dev, make_layer, x_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


_cache = {}


def weights_fp4(name):
    if name not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        fam = W.family(name)
        w = W.make_weights_fp4(fam)
        dw = [None if a is None else dev(a) for a in
              (w.router_w, w.router_bias, w.w13, w.sf13, w.g13, w.w2, w.sf2, w.g2)]
        _cache[name] = (fam, w, dw)
    return _cache[name]


def run_fp4(layer, x_bits, dw, k):
    out = layer.forward_nvfp4(x_dev(x_bits), *dw, k)
    r = layer.routing(x_bits.shape[0], k)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return (out.view(torch.int16).cpu().numpy().astype(np.uint16),
            {n: t.cpu().numpy() for n, t in r.items()})


def reference_fp4(x_bits, w, k, tokens=None):
    return F.moe_forward_nvfp4(x_bits, w.router_w, w.router_bias, w.w13, w.sf13, w.g13, w.w2,
                               w.sf2, w.g2, k, tokens=tokens)


def _check_y(layer, ref, P, H):
    """y of every position against the oracle's (expert by expert)."""
    y = layer.debug_buffer("y", torch.float32, (P, H)).cpu().numpy().astype(np.float64)
    ref_y = ref["y"].reshape(P, H)[ref["perm"]]
    off = ref["offsets"]
    for e in np.nonzero(ref["counts"])[0]:
        check_expert_y(y[off[e]:off[e + 1]], ref_y[off[e]:off[e + 1]], f"expert {e}")


@pytest.mark.parametrize("name,T", [("tiny", 4), ("olmoe_decode", 1), ("olmoe_decode", 8),
                                    ("olmoe_decode", 17), ("olmoe_decode", 64),
                                    ("olmoe_decode", 65), ("olmoe_prefill", 300)])
def test_nvfp4_layer_matches_oracle(name, T):
    """Routing bit-exact, every token's output and every position's y within
    tolerance; T = 17 and 64 take several 8-position groups per pass, T = 65
    and 300 the large-batch routing and several passes per expert."""
    fam, w, dw = weights_fp4(name)
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run_fp4(layer, x, dw, fam.top_k)
    ref = reference_fp4(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)
    _check_y(layer, ref, T * fam.top_k, fam.hidden)


@pytest.mark.parametrize("T", [1, 16])
def test_nvfp4_wide_decode(T):
    fam, w, dw = weights_fp4("wide_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run_fp4(layer, x, dw, fam.top_k)
    ref = reference_fp4(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_nvfp4_nibble_order_matters():
    """The pages' control: with the nibbles of every byte swapped the output
    must move far outside the tolerance (the kernel reads the low nibble as
    the even element)."""
    fam, w, dw = weights_fp4("olmoe_decode")
    T = 8
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, _ = run_fp4(layer, x, dw, fam.top_k)
    sw = list(dw)
    for i in (2, 5):
        b = dw[i]
        sw[i] = ((b & 0x0F) << 4) | (b >> 4)
    out_sw, _ = run_fp4(layer, x, sw, fam.top_k)
    ref = reference_fp4(x, w, fam.top_k)
    check_output(out, ref)
    with pytest.raises(AssertionError):
        check_output(out_sw, ref)


def test_nvfp4_deterministic_and_arguments():
    fam, w, dw = weights_fp4("olmoe_decode")
    x = W.make_x(fam, 8)
    layer = make_layer(fam, 8)
    a, _ = run_fp4(layer, x, dw, fam.top_k)
    b, _ = run_fp4(layer, x, dw, fam.top_k)
    assert np.array_equal(a, b)
    from fp8_routed_expert_gb300 import C, lib
    xt = x_dev(x)
    p = [None if t is None else t.data_ptr() for t in dw]
    rc = lib().moe_layer_forward_nvfp4(layer.handle, xt.data_ptr(), 8, p[0], p[1], p[2], None, p[4],
                                       p[5], p[6], p[7], fam.top_k, xt.data_ptr(), None)
    assert rc == C["MOE_ERR_ARG"]
    rc = lib().moe_layer_forward_nvfp4(layer.handle, xt.data_ptr(), 8, p[0], p[1], p[2], p[3] + 1,
                                       p[4], p[5], p[6], p[7], fam.top_k, xt.data_ptr(), None)
    assert rc == C["MOE_ERR_ALIGN"]
