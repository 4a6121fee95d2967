"""Shortcut-connected MoE: sub-block-1's decode attention against its
oracle, and the MoE and the attention run concurrently on two streams
(with an SM budget for the MoE) giving the same bits as run one after the
other."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import attention as A
from fp8_routed_expert_gb300 import C, lib
from harness import DeviceWeights, make_layer, output_errors, x_dev, REL_L2, MAXABS_RMS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _attn_inputs(B, S, nh, nkv, seed):
    q = W.normal_bf16(seed, 11, (B, nh, 128))
    k = W.normal_bf16(seed, 12, (B, S, nkv, 128))
    v = W.normal_bf16(seed, 13, (B, S, nkv, 128))
    return q, k, v


def _attention(q, k, v, nh, nkv, stream=None):
    B, S = k.shape[0], k.shape[1]
    dq, dk, dv = x_dev(q), x_dev(k), x_dev(v)
    out = torch.empty_like(dq)
    ws = torch.empty(lib().moe_attention_workspace_bytes(B, S, nh, 128), dtype=torch.uint8, device="cuda")
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = lib().moe_decode_attention(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, S, nh, nkv, 128,
                                    out.data_ptr(), ws.data_ptr(), ws.numel(), st)
    assert rc == 0, rc
    return out, (dq, dk, dv, ws)


@pytest.mark.parametrize("S,nh,nkv", [(1000, 16, 16), (4096, 16, 4), (257, 8, 1)])
def test_decode_attention_matches_oracle(S, nh, nkv):
    B = 8
    q, k, v = _attn_inputs(B, S, nh, nkv, S + nh)
    out, _ = _attention(q, k, v, nh, nkv)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().astype(np.uint16).reshape(B * nh, 128)
    ref = A.decode_attention(q, k, v).reshape(B * nh, 128)
    rel, mx, _ = output_errors(got, ref)
    assert rel <= REL_L2 and mx <= MAXABS_RMS, (rel, mx)


def test_attention_argument_errors():
    assert lib().moe_decode_attention(None, None, None, 1, 16, 16, 16, 64, None, None, 0, None) == \
        C["MOE_ERR_SHAPE"]
    assert lib().moe_decode_attention(None, None, None, 1, 16, 16, 3, 128, None, None, 0, None) == \
        C["MOE_ERR_SHAPE"]
    assert lib().moe_decode_attention(None, None, None, 1, 16, 16, 16, 128, None, None, 0, None) == \
        C["MOE_ERR_ARG"]


@pytest.mark.parametrize("budget", [0, 120])
def test_moe_and_attention_overlap_bit_identical(budget):
    fam = W.family("olmoe_decode")
    w = W.make_weights(fam)
    dw = DeviceWeights(w)
    T, k = 8, fam.top_k
    xb = W.make_x(fam, T)
    q, kc, vc = _attn_inputs(T, 4096, 16, 16, 77)
    layer = make_layer(fam, T)
    x = x_dev(xb)
    # one after the other
    moe_ref = layer.forward(x, *dw.args(), k)
    att_ref, keep = _attention(q, kc, vc, 16, 16)
    torch.cuda.synchronize()
    moe_ref, att_ref = moe_ref.clone(), att_ref.clone()
    # concurrently: the MoE on one stream, the attention on another
    assert lib().moe_set_sm_budget(layer.handle, budget) == 0
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(sa):
            moe = layer.forward(x, *dw.args(), k, stream=sa)
        with torch.cuda.stream(sb):
            att, keep2 = _attention(q, kc, vc, 16, 16, stream=sb)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(moe.view(torch.int16), moe_ref.view(torch.int16))
        assert torch.equal(att.view(torch.int16), att_ref.view(torch.int16))
    assert lib().moe_set_sm_budget(layer.handle, 0) == 0
