"""Plain f64 CPU oracle of decode attention: the sub-block that a
shortcut-connected MoE layer overlaps (dragon.c, "Shortcut-connected MoE").

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.

For every sequence b, query head h and its key/value head c = h // g
(g = n_heads // n_kv_heads query heads share one key/value head):

    s_j = q[b, h] . K[b, j, c] / sqrt(d)            (j = 0 .. S-1)
    o[b, h] = sum_j softmax(s)_j V[b, j, c]

The softmax is evaluated shifted by the largest score.  Reading D20: the
pages name the sub-block (attention, bf16) but not its arithmetic; this is
the plain scaled dot-product attention of one new token over its cache.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import bf16_to_f64


def decode_attention(q_bits, k_bits, v_bits) -> np.ndarray:
    """q bf16 bits [B, nh, d], K / V bf16 bits [B, S, nkv, d] -> f64 [B, nh, d]."""
    q, K, V = bf16_to_f64(q_bits), bf16_to_f64(k_bits), bf16_to_f64(v_bits)
    B, nh, d = q.shape
    nkv = K.shape[2]
    g = nh // nkv
    out = np.empty((B, nh, d), dtype=np.float64)
    for b in range(B):
        for h in range(nh):
            c = h // g
            s = K[b, :, c, :] @ q[b, h] / np.sqrt(d)
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ V[b, :, c, :]
    return out
