"""The oracle's own functions run over independent pieces on a thread pool.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: imported by ``tests/``
and by ``bench.py``'s CPU-baseline and reference legs, never by the CUDA
library or its binding.

No arithmetic lives here.  The layer is cut where its definition is already
independent: router logits per token (each token's row of x against W), and
the expert FFN per expert segment (the pairs routed to one expert, with that
expert's weights dequantised once).  Every piece is computed by the same
``moe_oracle`` function, on the same rows, in the same order as
``moe_oracle.moe_forward`` computes it, so the results are identical to it
element for element (pinned by a test); numpy releases the interpreter lock
inside its array loops, so the pieces run on all host cores.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import moe_oracle as mo


def default_workers() -> int:
    return os.cpu_count() or 1


def router_logits(x: np.ndarray, router_w, router_bias=None, workers: int | None = None,
                  chunk: int = 8) -> np.ndarray:
    """``moe_oracle.router_logits`` over chunks of tokens (the bias is added by
    the same call, per chunk)."""
    T = x.shape[0]
    out = np.empty((T, router_w.shape[0]), dtype=np.float64)

    def piece(t0):
        out[t0:t0 + chunk] = mo.router_logits(x[t0:t0 + chunk], router_w, router_bias, chunk=chunk)

    with ThreadPoolExecutor(workers or default_workers()) as ex:
        list(ex.map(piece, range(0, T, chunk)))
    return out


def expert_segments(x: np.ndarray, idx: np.ndarray, experts, w13, s13, w2, s2,
                    workers: int | None = None, keep_h: bool = False) -> dict:
    """h and y of every pair routed to each expert in ``experts``.

    Returns {e: (rows_t, rows_r, h_e or None, y_e)}: the pairs (token, rank) of
    expert e in ascending token order, as ``moe_forward`` finds them, and
    ``moe_oracle.expert_ffn`` of their x rows with e's dequantised weights.
    """
    def piece(e):
        rows_t, rows_r = np.nonzero(idx == e)
        w13_e = mo.dequantize(w13[e], s13[e])
        w2_e = mo.dequantize(w2[e], s2[e])
        h_e, y_e = mo.expert_ffn(x[rows_t], w13_e, w2_e)
        return e, (rows_t, rows_r, h_e if keep_h else None, y_e)

    with ThreadPoolExecutor(workers or default_workers()) as ex:
        return dict(ex.map(piece, [int(e) for e in experts]))


def moe_forward(x_bits, router_w, router_bias, w13, s13, w2, s2, top_k: int, tokens=None,
                workers: int | None = None) -> dict:
    """``moe_oracle.moe_forward`` with its per-token and per-expert loops on a
    thread pool; same arguments (no ``keep_h``) and the same result keys."""
    x = mo.bf16_to_f64(x_bits)
    T, H = x.shape
    E = router_w.shape[0]
    logits = router_logits(x, router_w, router_bias, workers)
    idx = mo.select_topk(logits, top_k)
    wts = mo.topk_weights(logits, idx)
    counts, offsets, perm, inv = mo.permutation(idx, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = np.zeros((tok.size, top_k, H), dtype=np.float64)
    if tok.size:
        sel = idx[tok]
        seg = expert_segments(x[tok], sel, np.unique(sel), w13, s13, w2, s2, workers)
        for rows_t, rows_r, _, y_e in seg.values():
            y[rows_t, rows_r] = y_e
    out = mo.combine(wts[tok], y)
    return dict(logits=logits, idx=idx, wts=wts, counts=counts, offsets=offsets, perm=perm,
                inv=inv, tokens=tok, y=y, out=out, out_bf16=mo.round_to_bf16(out))
