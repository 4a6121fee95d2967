"""Plain f64 CPU oracle of the routed-MoE layer with FP4 (NVFP4) expert weights.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: imported by
``tests/`` and ``bench.py``'s CPU legs, never by the CUDA library.

The format is the one the Qwen post's experts use ("Why this model, of all
models" and piece 1, "Repack experts for the disk", of "The engine"): 4-bit
e2m1 codes plus one e4m3 scale per 16 weights -- its expert block of three
2560x640 matrices is 2,764,800 bytes, i.e. half a byte per weight plus one
byte per 16 weights.  The NVFP4 format adds one f32 scale per matrix; the
pages' byte count leaves no room for it inside the expert block, so it is
carried beside the block (reading D18).  A weight's value is

    e2m1(code) * e4m3(block scale of its 16-weight group along K) * global

Codes are packed two per byte along K, the even element in the low nibble
(reading D19; the pages only show that the nibble order matters: swapping
the nibbles is their control that must break the model).

Everything after dequantisation -- router, selection, weights, permutation,
SwiGLU expert, rank-order combine -- is the FP8 oracle's own functions.
"""
from __future__ import annotations

import math

import numpy as np

from . import moe_oracle as mo

GROUP = 16  # weights per e4m3 block scale


def e2m1_value(code: int) -> float:
    """Value of one 4-bit e2m1 code, from the format definition: sign bit 3,
    two exponent bits with bias 1, one mantissa bit; exponent field 0 is
    subnormal (0.5 * m); no infinities or NaN, so the largest value is 6."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * 0.5 * m
    return s * math.ldexp(1.0 + 0.5 * m, e - 1)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Codes [..., 2n] of packed bytes [..., n]: element 2j is the low nibble
    of byte j, element 2j + 1 its high nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def dequantize_nvfp4(packed: np.ndarray, block_scales: np.ndarray, global_scale) -> np.ndarray:
    """f64 weights [..., R, C] of packed codes [..., R, C/2], e4m3 block-scale
    codes [..., R, C/16] and the matrix's f32 global scale."""
    vals = E2M1_TABLE[unpack_e2m1(packed)]
    sc = mo.E4M3_TABLE[np.asarray(block_scales, dtype=np.uint8)]
    if np.isnan(sc).any():
        raise ValueError("e4m3 NaN code in block scales")
    return vals * np.repeat(sc, GROUP, axis=-1) * float(global_scale)


def moe_forward_nvfp4(x_bits, router_w, router_bias, w13, sf13, g13, w2, sf2, g2, top_k: int,
                      tokens=None) -> dict:
    """The whole layer in f64 with FP4 experts.

    w13 u8 [E, 2I, H/2] (rows [0, I) gate, [I, 2I) up), sf13 e4m3 [E, 2I, H/16],
    g13 f32 [E]; w2 u8 [E, H, I/2], sf2 e4m3 [E, H, I/16], g2 f32 [E].  Same
    result keys as ``moe_oracle.moe_forward``.
    """
    x = mo.bf16_to_f64(x_bits)
    T, H = x.shape
    E = router_w.shape[0]
    logits = mo.router_logits(x, router_w, router_bias)
    idx = mo.select_topk(logits, top_k)
    wts = mo.topk_weights(logits, idx)
    counts, offsets, perm, inv = mo.permutation(idx, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = np.zeros((tok.size, top_k, H), dtype=np.float64)
    if tok.size:
        sel = idx[tok]
        for e in np.unique(sel):
            rows_t, rows_r = np.nonzero(sel == e)
            w13_e = dequantize_nvfp4(w13[e], sf13[e], g13[e])
            w2_e = dequantize_nvfp4(w2[e], sf2[e], g2[e])
            _, y_e = mo.expert_ffn(x[tok[rows_t]], w13_e, w2_e)
            y[rows_t, rows_r] = y_e
    out = mo.combine(wts[tok], y)
    return dict(logits=logits, idx=idx, wts=wts, counts=counts, offsets=offsets, perm=perm,
                inv=inv, tokens=tok, y=y, out=out, out_bf16=mo.round_to_bf16(out))
