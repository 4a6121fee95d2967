"""Pins of the FP4 (NVFP4) oracle to facts outside itself (no GPU).

* the e2m1 value set of the published format definition (OCP Microscaling
  formats, E2M1: the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6);
* a generic sign/exponent/mantissa decoder, checked exhaustively against
  torch's float8_e4m3fn and float8_e5m2 conversions, gives the same table;
* the Qwen post's expert block size (tests/golden/nvfp4_facts.json) follows
  from half a byte per weight plus one byte per 16 weights;
* hand-built bytes pin the nibble order and the 16-weight scale groups;
* the whole layer equals per-token loops with exactly rounded sums over
  weights decoded by the generic decoder;
* planted mistakes (swapped nibbles, 32-weight scale groups, a dropped
  global scale) break that pin.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as F
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def minifloat(code: int, e_bits: int, m_bits: int, bias: int) -> float:
    """Generic decode of a sign | exponent | mantissa code with subnormals."""
    s = -1.0 if (code >> (e_bits + m_bits)) & 1 else 1.0
    e = (code >> m_bits) & ((1 << e_bits) - 1)
    m = code & ((1 << m_bits) - 1)
    if e == 0:
        return s * math.ldexp(m / (1 << m_bits), 1 - bias)
    return s * math.ldexp(1.0 + m / (1 << m_bits), e - bias)


def test_generic_decoder_matches_torch_e4m3_and_e5m2():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    e4 = codes.view(torch.float8_e4m3fn).to(torch.float32).double().tolist()
    e5 = codes.view(torch.float8_e5m2).to(torch.float32).double().tolist()
    for c in range(256):
        if c & 0x7F != 0x7F:                  # e4m3fn: only S.1111.111 is NaN
            assert minifloat(c, 4, 3, 7) == e4[c], c
        if (c >> 2) & 0x1F != 0x1F:           # e5m2: exponent 31 is inf / NaN
            assert minifloat(c, 5, 2, 15) == e5[c], c


def test_e2m1_table_is_the_format_definition():
    published = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.E2M1_TABLE[:8].tolist() == published
    assert F.E2M1_TABLE[8:].tolist() == [-v for v in published]
    assert math.copysign(1.0, F.E2M1_TABLE[8]) == -1.0   # code 8 is -0
    for c in range(16):
        assert F.E2M1_TABLE[c] == minifloat(c, 2, 1, 1), c


def test_expert_block_size_of_the_pages():
    f = json.load(open(os.path.join(GOLDEN, "nvfp4_facts.json")))
    R, C = f["matrix_rows"], f["matrix_cols"]
    codes = np.zeros((R, C // 2), np.uint8)            # two codes per byte
    scales = np.zeros((R, C // F.GROUP), np.uint8)     # one e4m3 per 16 weights
    assert f["matrices"] * (codes.nbytes + scales.nbytes) == f["expert_block_bytes"]


def test_nibble_order_and_scale_groups():
    # byte 0x31: low nibble 1 (0.5) is element 0, high nibble 3 (1.5) element 1
    packed = np.full((1, 16), 0x31, np.uint8)          # 32 weights: two groups
    sc = np.array([[0x38, 0x40]], np.uint8)            # e4m3 1.0 and 2.0
    d = F.dequantize_nvfp4(packed, sc, np.float32(0.25))
    assert d[0, :16].tolist() == [0.5 * 0.25, 1.5 * 0.25] * 8
    assert d[0, 16:].tolist() == [0.5 * 0.5, 1.5 * 0.5] * 8
    # negative codes: 0xF9 = high 15 (-6), low 9 (-0.5)
    d = F.dequantize_nvfp4(np.full((1, 8), 0xF9, np.uint8), np.array([[0x38]], np.uint8), 1.0)
    assert d[0, :2].tolist() == [-0.5, -6.0]


def _decode_brute(packed, sc, g, R, C):
    """Weights decoded element by element with the generic decoder."""
    e4 = [minifloat(c, 4, 3, 7) for c in range(256)]
    out = [[0.0] * C for _ in range(R)]
    for r in range(R):
        for c in range(C):
            byte = int(packed[r, c // 2])
            code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
            out[r][c] = minifloat(code, 2, 1, 1) * e4[int(sc[r, c // 16])] * float(g)
    return out


def brute_layer_fp4(x_bits, w, k, mistake=None):
    T, H = x_bits.shape
    E = w.router_w.shape[0]
    inter = w.w13.shape[1] // 2
    x = [[struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in row] for row in x_bits]
    res_idx, res_w, res_out = [], [], []
    for t in range(T):
        logits = [math.fsum(x[t][h] * float(w.router_w[e, h]) for h in range(H)) for e in range(E)]
        m = max(logits)
        p = [math.exp(v - m) for v in logits]
        z = math.fsum(p)
        order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        ssel = math.fsum(p[e] / z for e in order)
        wts = [p[e] / z / ssel for e in order]
        acc = [0.0] * H
        for r, e in enumerate(order):
            w13e = _decode_brute(w.w13[e], w.sf13[e], w.g13[e], 2 * inter, H)
            w2e = _decode_brute(w.w2[e], w.sf2[e], w.g2[e], H, inter)
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


@pytest.fixture(scope="module")
def tiny_fp4():
    fam = W.family("tiny")
    w = W.make_weights_fp4(fam)
    x = W.make_x(fam, 2)
    return fam, w, x, brute_layer_fp4(x, w, fam.top_k)


def _forward(w, x, k, **kw):
    return F.moe_forward_nvfp4(x, w.router_w, w.router_bias, w.w13, w.sf13, w.g13, w.w2, w.sf2,
                               w.g2, k, **kw)


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def test_layer_fp4_matches_brute_force(tiny_fp4):
    fam, w, x, (b_idx, b_w, b_out) = tiny_fp4
    res = _forward(w, x, fam.top_k)
    assert np.array_equal(res["idx"], b_idx)
    assert np.allclose(res["wts"], b_w, rtol=1e-12, atol=0)
    assert _rel(res["out"], b_out) < 1e-12


def test_planted_mistakes_break_the_pin(tiny_fp4, monkeypatch):
    fam, w, x, (_, _, b_out) = tiny_fp4

    def swapped(packed):
        p = np.asarray(packed, np.uint8)
        out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0x0F
        return out

    with monkeypatch.context() as m:
        m.setattr(F, "unpack_e2m1", swapped)
        assert _rel(_forward(w, x, fam.top_k)["out"], b_out) > 1e-3
    with monkeypatch.context() as m:
        orig = F.dequantize_nvfp4

        def groups32(packed, sc, g):
            return orig(packed, np.repeat(sc[..., ::2], 2, axis=-1), g)

        m.setattr(F, "dequantize_nvfp4", groups32)
        assert _rel(_forward(w, x, fam.top_k)["out"], b_out) > 1e-3
    with monkeypatch.context() as m:
        orig = F.dequantize_nvfp4
        m.setattr(F, "dequantize_nvfp4", lambda p, s, g: orig(p, s, 1.0))
        assert _rel(_forward(w, x, fam.top_k)["out"], b_out) > 1e-3


def test_fp4_weights_follow_the_same_streams():
    """The generator quantises the same normal values as the FP8 weights:
    the two dequantised expert sets agree to the FP4 grid's resolution."""
    fam = W.family("tiny")
    w4 = W.make_weights_fp4(fam)
    w8 = W.make_weights(fam)
    d4 = F.dequantize_nvfp4(w4.w13, w4.sf13, 1.0) * w4.g13[:, None, None].astype(np.float64)
    d8 = oracle.dequantize(w8.w13, w8.s13)
    assert 0.05 < _rel(d4, d8) < 0.15
    assert np.array_equal(w4.router_w, w8.router_w)
