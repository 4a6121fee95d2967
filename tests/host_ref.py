"""Host restatement of the combine's f32 arithmetic, for the bit-exact
combine test (WARP BACKENDS.md, "Coherent memory": each token's expert
partials are reduced in the router's rank order).

The combine computes, per output element, one fused multiply-add chain in f32
over the ranks r = 0..k-1, starting from zero:
    acc = fma(w[t, r], y_r, acc),
where y_r is the pair's y (on the decode path the sum, in f32 and in plane
order, of its three term planes), and rounds acc once to bf16.  numpy has no
fused multiply-add, so ``fma_f32`` forms it exactly: the product of two f32
values is exact in f64, the f64 sum's rounding error is recovered exactly
(Knuth's TwoSum), and a sum that lands exactly halfway between two f32 values
is resolved by the sign of that error before the final rounding.
"""
from __future__ import annotations

import numpy as np

_LOW29 = np.uint64((1 << 29) - 1)  # f64 mantissa bits below f32 precision
_HALF29 = np.uint64(1 << 28)


def fma_f32(a, b, c) -> np.ndarray:
    """Correctly rounded f32 fma(a, b, c) of f32 arrays (normal-range results)."""
    a = np.asarray(a, dtype=np.float32).astype(np.float64)
    b = np.asarray(b, dtype=np.float32).astype(np.float64)
    c = np.asarray(c, dtype=np.float32).astype(np.float64)
    p = a * b                       # exact: 24 + 24 significant bits
    p, c = np.broadcast_arrays(p, c)
    s = p + c                       # f64 rounding of the exact p + c
    pp = s - c                      # TwoSum (Knuth): s + err == p + c exactly
    cc = s - pp
    err = (c - cc) + (p - pp)
    r = s.astype(np.float32)
    bits = s.view(np.uint64)
    tie = ((bits & _LOW29) == _HALF29) & (err != 0)
    if tie.any():
        # s is the midpoint of two f32 neighbours: the exact sum lies on the
        # side of err, so round toward it
        trunc = (bits[tie] & ~_LOW29).view(np.float64).astype(np.float32)  # lower magnitude
        away = np.nextafter(trunc, np.copysign(np.float32(np.inf), trunc))
        up = np.sign(err[tie]) == np.sign(s[tie])
        r[tie] = np.where(up, away, trunc)
    return r


def combine_f32(y_planes: np.ndarray, inv: np.ndarray, wts: np.ndarray) -> np.ndarray:
    """f32 acc [T, H] of the rank-order fma chain.

    y_planes f32 [NP, P, H] (position order), inv int [T*k] (pair -> position),
    wts f32 [T, k]."""
    T, k = wts.shape
    H = y_planes.shape[2]
    acc = np.zeros((T, H), dtype=np.float32)
    for r in range(k):
        pos = inv.reshape(T, k)[:, r]
        s = y_planes[0][pos].astype(np.float32)
        for q in range(1, y_planes.shape[0]):
            s = (s + y_planes[q][pos]).astype(np.float32)  # f32 add, plane order
        acc = fma_f32(wts[:, r:r + 1], s, acc)
    return acc
