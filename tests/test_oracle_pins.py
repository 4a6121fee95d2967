"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute itself: a
library routine (torch's float8_e4m3fn conversion), a brute-force search, a
pure-Python definition with exactly rounded sums (math.fsum), invariants, or
closed-form special cases.  ``test_planted_mistakes_fail`` shows that plausible
mistakes in the oracle break at least one of these pins.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as mo
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- formats

def test_e4m3_table_matches_torch_exhaustively():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    ours = oracle.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]


def test_e4m3_golden_facts():
    facts = json.load(open(os.path.join(GOLDEN, "format_facts.json")))
    assert len(oracle.E4M3_TABLE) == facts["e4m3_bit_patterns"]
    # closed forms of the e4m3 ("fn") definition: bias 7, 3 mantissa bits,
    # no infinities, 0x7E the largest finite value
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xC4) == -3.0
    assert math.isnan(oracle.e4m3_value(0x7F))


def test_bf16_widening_is_a_shift():
    # dragon.c, §8 Round 3: a bf16 widened to f32 is a 16-bit left shift
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, struct.unpack("<f", struct.pack("<I", 1 << 16))[0],
            struct.unpack("<f", struct.pack("<I", 0x7F7F << 16))[0]]
    assert oracle.bf16_to_f64(bits).tolist() == want


def _bf16_brute(v: float) -> int:
    """Nearest bf16 by searching the f32 bit patterns whose low half is zero."""
    f = np.float32(v)
    u = int(np.array([f]).view(np.uint32)[0])
    cands = []
    for hi in ((u >> 16) - 1, u >> 16, (u >> 16) + 1):
        hi &= 0xFFFF
        val = float(np.array([hi << 16], dtype=np.uint32).view(np.float32)[0])
        if math.isfinite(val):
            cands.append((abs(val - v), hi & 1, hi))  # ties: even mantissa first
    cands.sort()
    return cands[0][2]


def test_round_to_bf16_brute_force():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8),
                         1.0 + 2.0 ** -8 + 2.0 ** -40, 2.0 ** -130, 0.0]])
    got = oracle.round_to_bf16(v)
    for val, b in zip(v.tolist(), got.tolist()):
        assert b == _bf16_brute(val), val


def test_dequantize_block_mapping():
    # distinct power-of-two scale per block exposes any transposed or shifted grid
    R, C = 256, 384
    codes = np.full((R, C), 0x38, dtype=np.uint8)  # 1.0
    scales = np.array([[2.0 ** (3 * i + j) for j in range(3)] for i in range(2)], np.float32)
    d = oracle.dequantize(codes, scales)
    for r in (0, 127, 128, 255):
        for c in (0, 127, 128, 255, 256, 383):
            assert d[r, c] == 2.0 ** (3 * (r // 128) + (c // 128))


# ----------------------------------------------------------------------------- brute force

def _torch_decode_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).double().tolist()


def brute_layer(x_bits, rw, bias, w13, s13, w2, s2, k):
    """Per-token, per-expert loops with exactly rounded sums; full softmax."""
    dec = _torch_decode_table()
    T, H = x_bits.shape
    E = rw.shape[0]
    inter = w13.shape[1] // 2
    x = [[struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in row] for row in x_bits]
    res_idx, res_w, res_out = [], [], []
    for t in range(T):
        logits = []
        for e in range(E):
            s = math.fsum(x[t][h] * float(rw[e, h]) for h in range(H))
            logits.append(s + (float(bias[e]) if bias is not None else 0.0))
        m = max(logits)
        p = [math.exp(v - m) for v in logits]
        z = math.fsum(p)
        p = [v / z for v in p]
        order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        ssel = math.fsum(p[e] for e in order)
        wts = [p[e] / ssel for e in order]
        acc = [0.0] * H
        for r, e in enumerate(order):
            w13e = [[dec[w13[e, i, h]] * float(s13[e, i // 128, h // 128]) for h in range(H)]
                    for i in range(2 * inter)]
            w2e = [[dec[w2[e, j, i]] * float(s2[e, j // 128, i // 128]) for i in range(inter)]
                   for j in range(H)]
            g = [math.fsum(w13e[i][h] * x[t][h] for h in range(H)) for i in range(inter)]
            u = [math.fsum(w13e[inter + i][h] * x[t][h] for h in range(H)) for i in range(inter)]
            hh = [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(inter)]
            y = [math.fsum(w2e[j][i] * hh[i] for i in range(inter)) for j in range(H)]
            for j in range(H):
                acc[j] += wts[r] * y[j]
        res_idx.append(order)
        res_w.append(wts)
        res_out.append(acc)
    return np.array(res_idx), np.array(res_w), np.array(res_out)


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _tiny(bias=False, T=None):
    fam = W.family("tiny")
    w = W.make_weights(fam)
    if bias:
        w.router_bias = W.normal_f32(99, 3, (fam.n_experts,), 0.5)
    x = W.make_x(fam, T or fam.tokens[0])
    return fam, w, x


@pytest.fixture(scope="module")
def tiny_case():
    fam, w, x = _tiny()
    bf = brute_layer(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2, fam.top_k)
    return fam, w, x, bf


def _check_against_brute(fam, w, x, bf, forward=None):
    forward = forward or oracle.moe_forward
    res = forward(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2, fam.top_k)
    b_idx, b_w, b_out = bf
    assert np.array_equal(res["idx"], b_idx)
    assert np.allclose(res["wts"], b_w, rtol=1e-12, atol=0)
    assert _rel(res["out"], b_out) < 1e-12
    return res


def test_layer_matches_brute_force_tiny(tiny_case):
    fam, w, x, bf = tiny_case
    _check_against_brute(fam, w, x, bf)


def test_layer_matches_brute_force_with_bias():
    fam, w, x = _tiny(bias=True, T=3)
    bf = brute_layer(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2, fam.top_k)
    _check_against_brute(fam, w, x, bf)


def test_oracle_agrees_with_independent_torch_f64():
    """Same layer through torch's f64 CPU matmuls on torch-decoded weights."""
    fam = W.family("olmoe_decode")
    w = W.make_weights(fam)
    x = W.make_x(fam, 8)
    res = oracle.moe_forward(x, w.router_w, None, w.w13, w.s13, w.w2, w.s2, fam.top_k)
    xt = torch.from_numpy(x.astype(np.int16)).view(torch.bfloat16).double()
    rw = torch.from_numpy(w.router_w).double()
    logits = xt @ rw.T
    dec = torch.tensor(_torch_decode_table(), dtype=torch.float64)
    I = fam.inter
    out = torch.zeros(8, fam.hidden, dtype=torch.float64)
    for t in range(8):
        vals, order = torch.sort(logits[t], descending=True, stable=True)
        sel = order[:fam.top_k]
        p = torch.softmax(logits[t], 0)[sel]
        p = p / p.sum()
        assert sel.tolist() == res["idx"][t].tolist()
        for r, e in enumerate(sel.tolist()):
            s13 = torch.from_numpy(w.s13[e]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
            s2 = torch.from_numpy(w.s2[e]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
            w13 = dec[torch.from_numpy(w.w13[e]).long()] * s13
            w2 = dec[torch.from_numpy(w.w2[e]).long()] * s2
            hh = torch.nn.functional.silu(w13[:I] @ xt[t]) * (w13[I:] @ xt[t])
            out[t] += p[r] * (w2 @ hh)
    assert _rel(res["out"], out.numpy()) < 1e-10


def test_one_expert_is_the_dense_ffn():
    """With one expert and k = 1 the layer is a dense SwiGLU FFN in the same
    blockwise-FP8 format (dragon.c, "Precision": the dense branches share the
    routed experts' format): every token has weight exactly 1, the permutation
    is the identity, and the output is bf16(W2 (silu(W1 x) * (W3 x))), here
    through torch's decode table and f64 matmuls."""
    fam = W.family("dense_ffn")
    assert fam.n_experts == 1 and fam.top_k == 1
    w = W.make_weights(fam)
    T = 4
    x = W.make_x(fam, fam.tokens[0])[:T]
    res = oracle.moe_forward(x, w.router_w, None, w.w13, w.s13, w.w2, w.s2, 1)
    assert (res["idx"] == 0).all() and (res["wts"] == 1.0).all()
    assert res["counts"].tolist() == [T] and res["perm"].tolist() == list(range(T))
    dec = torch.tensor(_torch_decode_table(), dtype=torch.float64)
    I = fam.inter
    s13 = torch.from_numpy(w.s13[0]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    s2 = torch.from_numpy(w.s2[0]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    w13 = dec[torch.from_numpy(w.w13[0]).long()] * s13
    w2 = dec[torch.from_numpy(w.w2[0]).long()] * s2
    xt = torch.from_numpy(x.astype(np.int16)).view(torch.bfloat16).double()
    dense = (torch.nn.functional.silu(xt @ w13[:I].T) * (xt @ w13[I:].T)) @ w2.T
    assert _rel(res["out"], dense.numpy()) < 1e-10
    want = dense.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    # one rounding of the f64 sum; the float32 detour may double-round only
    # where f64 lies within 2^-29 relative of a bf16 midpoint
    assert (oracle.round_to_bf16(res["out"]) != want).mean() < 1e-3


# ----------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("name,T", [("tiny", 4), ("olmoe_decode", 8), ("olmoe_prefill", 64)])
def test_routing_invariants(name, T):
    fam = W.family(name)
    w = W.make_weights(fam) if name != "olmoe_prefill" else None
    rw = w.router_w if w else W.normal_f32(fam.seed, 2, (fam.n_experts, fam.hidden), 0.02)
    bias = None if fam.bias_std is None else W.normal_f32(fam.seed, 3, (fam.n_experts,), fam.bias_std)
    x = oracle.bf16_to_f64(W.make_x(fam, T))
    logits = oracle.router_logits(x, rw, bias)
    idx = oracle.select_topk(logits, fam.top_k)
    wts = oracle.topk_weights(logits, idx)
    counts, offsets, perm, inv = oracle.permutation(idx, fam.n_experts)
    k, P = fam.top_k, T * fam.top_k
    assert np.allclose(wts.sum(1), 1.0, atol=1e-15)
    assert (np.diff(np.take_along_axis(logits, idx, 1), axis=1) <= 0).all()
    assert counts.sum() == P and offsets[-1] == P
    assert np.array_equal(np.sort(perm), np.arange(P))            # bijection
    assert np.array_equal(perm[inv], np.arange(P))                # inverse
    assert np.array_equal(np.bincount(perm // k, minlength=T), np.full(T, k))  # k per token
    for e in range(fam.n_experts):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()                           # stable: ascending p
        assert (idx.reshape(-1)[seg] == e).all()
    # each row of idx has distinct experts and nothing outside it beats its last
    for t in range(T):
        assert len(set(idx[t].tolist())) == k
        rest = np.setdiff1d(np.arange(fam.n_experts), idx[t])
        assert (logits[t, rest] <= logits[t, idx[t, -1]]).all()


# ----------------------------------------------------------------------------- closed forms

def _fwd(x, w, k, bias=None):
    return oracle.moe_forward(x, w.router_w, bias, w.w13, w.s13, w.w2, w.s2, k)


def test_k_equals_E_gives_full_softmax():
    fam, w, x = _tiny()
    res = _fwd(x, w, fam.n_experts)
    lg = res["logits"]
    full = np.exp(lg - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    assert np.allclose(np.take_along_axis(full, res["idx"], 1), res["wts"], rtol=1e-13)


def test_k1_is_the_argmax_expert():
    fam, w, x = _tiny()
    res = _fwd(x, w, 1)
    assert (res["wts"] == 1.0).all()
    assert np.array_equal(res["idx"][:, 0], np.argmax(res["logits"], axis=1))
    assert np.array_equal(res["out"], res["y"][:, 0, :])


def test_zero_input_gives_zero_output_and_lowest_experts():
    fam, w, _ = _tiny()
    x = np.zeros((3, fam.hidden), dtype=np.uint16)
    res = _fwd(x, w, fam.top_k)
    assert (res["out"] == 0).all() and (res["out_bf16"] == 0).all()
    assert (res["idx"] == np.arange(fam.top_k)).all()            # all logits tie at 0
    assert (res["wts"] == 1.0 / fam.top_k).all()


def test_identical_router_rows_tie_to_lower_index():
    fam, w, x = _tiny()
    w.router_w[:] = w.router_w[5]
    res = _fwd(x, w, 3)
    assert (res["idx"] == np.array([0, 1, 2])).all()
    assert (res["wts"] == 1.0 / 3).all()


def test_one_hot_input_reads_single_weight_column():
    """x = e_j with unit scales: g_i, u_i are single codes; closed-form SwiGLU."""
    fam, w, _ = _tiny()
    w.s13[:] = 1.0
    w.s2[:] = 1.0
    j = 37
    x = np.zeros((1, fam.hidden), dtype=np.uint16)
    x[0, j] = 0x3F80  # 1.0
    res = oracle.moe_forward(x, w.router_w, None, w.w13, w.s13, w.w2, w.s2, 1)
    e = int(res["idx"][0, 0])
    assert res["logits"][0, e] == float(w.router_w[e, j])
    I = fam.inter
    g = oracle.E4M3_TABLE[w.w13[e, :I, j]]
    u = oracle.E4M3_TABLE[w.w13[e, I:, j]]
    h = g / (1 + np.exp(-g)) * u
    y = oracle.E4M3_TABLE[w.w2[e]] @ h
    assert np.allclose(res["out"][0], y, rtol=1e-14, atol=0)


def test_negating_up_rows_negates_output():
    fam, w, x = _tiny()
    a = _fwd(x, w, fam.top_k)
    w.w13[:, fam.inter:, :] ^= 0x80           # flip the sign bit of every up code
    b = _fwd(x, w, fam.top_k)
    assert np.array_equal(a["out"], -b["out"])
    assert np.array_equal(a["out_bf16"] ^ 0x8000, b["out_bf16"]) or \
        np.array_equal(a["out_bf16"][a["out"] != 0] ^ 0x8000, b["out_bf16"][a["out"] != 0])


def test_power_of_two_scale_on_w2_scales_output_exactly():
    fam, w, x = _tiny()
    a = _fwd(x, w, fam.top_k)
    w.s2 *= 4.0
    b = _fwd(x, w, fam.top_k)
    assert np.array_equal(4.0 * a["out"], b["out"])


def test_bytes_per_token_worked_examples():
    """Bytes per token = experts chosen x layers x bytes per expert, as the
    DeepSeek-V4.1-Flash post works it out ('Bytes per token decide everything')."""
    facts = json.load(open(os.path.join(GOLDEN, "bytes_per_token.json")))
    for case in facts["cases"]:
        gib = case["k"] * case["layers"] * case["mib_per_expert"] / 1024.0
        assert abs(gib - case["gib_per_token"]) <= 0.01, case
    # the expert-size formula used for the decode roofline: 3*H*I codes + f32 scales
    assert W.family("tiny").expert_bytes == 98328
    assert W.family("olmoe_decode").expert_bytes == 6292992


# ----------------------------------------------------------------------------- controls

def _swap_gate_up(x_rows, w13_e, w2_e):
    inter = w13_e.shape[0] // 2
    return mo.__dict__["_orig_expert_ffn"](x_rows, np.concatenate([w13_e[inter:], w13_e[:inter]]), w2_e)


def _transposed_scales(codes, scales):
    s = scales
    if s.shape[-1] != s.shape[-2]:
        s = np.swapaxes(s, -1, -2).reshape(s.shape)
    else:
        s = np.swapaxes(s, -1, -2)
    return mo.__dict__["_orig_dequantize"](codes, s)


def _ties_high(logits, k):
    idx = np.empty((logits.shape[0], k), dtype=np.int64)
    for t in range(logits.shape[0]):
        idx[t] = np.lexsort((-np.arange(logits.shape[1]), -logits[t]))[:k]
    return idx


def _no_renorm(logits, idx):
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    return np.take_along_axis(p, idx, 1)


def _silu_wrong(z):
    return z / (1.0 + np.exp(z))


@pytest.mark.parametrize("target,mutant", [
    ("expert_ffn", _swap_gate_up),
    ("dequantize", _transposed_scales),
    ("topk_weights", _no_renorm),
    ("silu", _silu_wrong),
])
def test_planted_mistakes_fail(tiny_case, monkeypatch, target, mutant):
    fam, w, x, bf = tiny_case
    mo.__dict__["_orig_expert_ffn"] = mo.expert_ffn
    mo.__dict__["_orig_dequantize"] = mo.dequantize
    monkeypatch.setattr(mo, target, mutant)
    with pytest.raises(AssertionError):
        _check_against_brute(fam, w, x, bf, forward=mo.moe_forward)


def test_planted_tie_break_mistake_fails(monkeypatch):
    fam, w, x = _tiny()
    w.router_w[:] = w.router_w[5]
    monkeypatch.setattr(mo, "select_topk", _ties_high)
    res = mo.moe_forward(x, w.router_w, None, w.w13, w.s13, w.w2, w.s2, 3)
    assert not (res["idx"] == np.array([0, 1, 2])).all()


# ----------------------------------------------------------------------------- threaded driver

@pytest.mark.parametrize("name,T,tokens", [("tiny", 4, None), ("olmoe_prefill", 48, [0, 7, 47]),
                                           ("olmoe_decode", 8, None)])
def test_threaded_driver_is_the_oracle(name, T, tokens):
    """oracle.threaded runs the oracle's own functions over tokens and expert
    segments on a thread pool: every result equals moe_forward's exactly."""
    from oracle import threaded
    fam = W.family(name)
    w = W.make_weights(fam)
    x = W.make_x(fam, T)
    a = oracle.moe_forward(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2, fam.top_k,
                           tokens=tokens)
    b = threaded.moe_forward(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2, fam.top_k,
                             tokens=tokens, workers=3)
    assert a.keys() == b.keys()
    for key in a:
        assert np.array_equal(a[key], b[key]), key
