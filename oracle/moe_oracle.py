"""Plain, slow, f64 CPU oracle of the blockwise-FP8 routed-MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this module.  The CUDA
library never calls it, links it or shares code with it; the two meet only in
the seeded inputs of ``workloads/``.

What the layer computes, step by step, and where each step comes from:

1. e4m3 decode and blockwise dequantisation.  Expert weights are e4m3 codes
   with one f32 scale per 128x128 block, stored with the weights (dragon.c,
   "Precision"); the value of a weight is its code's value times its block's
   scale, applied inline rather than by expanding the expert (dragon.c, §8
   "Round 2 — native-precision compute" and "Round 3", where the scale of each
   128-column block is folded out of the inner loop).
2. Router in f32 inputs (dragon.c, "Precision": "router f32"), activations
   kept unrounded (Trochilus, "Results": activations in float, never rounded
   to 8 bits before a product).  Logits are computed here in f64 from exact
   products (bf16 x f32 fits in f64's 53 bits).
3. Selection: top-k by logit, descending; equal logits go to the lower expert
   index (Trochilus, "What makes it different": the lowest row wins a tie).
4. Weights: softmax over all E, keep the k selected, renormalise; equal to the
   softmax over the k selected logits.
5. Permutation: counting sort of the (token, expert) pairs p = t*k + r by
   expert (Trochilus, "Acknowledgements", the ds4 row): histogram, exclusive
   scan, stable scatter in ascending p.
6. Expert FFN with SwiGLU: g = W13[e, :I] x, u = W13[e, I:] x (gate rows
   before up rows, the gate | up | down order of the repacked expert block in
   the DeepSeek-V4.1-Flash post, §1 "Repack experts for the disk"),
   h = silu(g) * u with silu(z) = z / (1 + e^-z), y = W2[e] h.
7. Combine: out[t] = sum over r = 0..k-1, in router rank order, of
   wts[t, r] * y[t, r] (WARP BACKENDS.md, "Coherent memory": partials reduced
   in original router order), rounded once to bf16 (round to nearest even).

Readings where the pages are silent are listed at the top of each function.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 128  # the 128x128 scale block of the weight format


# ----------------------------------------------------------------------------- formats

def e4m3_value(code: int) -> float:
    """Value of one e4m3 ("fn") code, from the format definition.

    Sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0
    is subnormal: 2^-6 * m/8.  The codes 0x7F and 0xFF are NaN; there are no
    infinities, so the largest finite value is 0x7E = 448.  The dragon.c page
    (§8, "Round 3") notes that e4m3 has exactly 256 bit patterns, which is why
    a 256-entry table decodes it.
    """
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """f64 weights of e4m3 codes [..., R, C] with block scales [..., R/128, C/128].

    Reading: the scale multiplies (value = code value x scale); the scale grid
    is row-major over (row block, column block).
    """
    vals = E4M3_TABLE[codes]
    if np.isnan(vals).any():
        raise ValueError("e4m3 NaN code in weights")
    s = np.repeat(np.repeat(scales.astype(np.float64), BLOCK, axis=-2), BLOCK, axis=-1)
    return vals * s


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """A bf16 is the upper half of an f32 (dragon.c, §8 "Round 3": widening is a
    16-bit left shift)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32) \
        .astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round f64 values once to bf16 (nearest, ties to even); returns uint16 bits.

    bf16 keeps 8 significant bits and f32's exponent range, so the spacing of
    representable values in [2^e, 2^(e+1)) is 2^(e-7), and 2^-133 below 2^-126.
    Scaling by a power of two is exact, so rint on v / spacing rounds once.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.float64)
    nz = (v != 0) & np.isfinite(v)
    _, ex = np.frexp(v[nz])          # |v| in [2^(ex-1), 2^ex)
    e = np.maximum(ex - 1, -126)
    spacing = np.ldexp(1.0, e - 7)
    out[nz] = np.rint(v[nz] / spacing) * spacing
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    f32 = out.astype(np.float32)     # exact: at most 8 significant bits
    big = np.abs(out) > 3.3895313892515355e38  # beyond the largest finite bf16
    f32[big] = np.copysign(np.inf, out[big]).astype(np.float32)
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(v)
    bits[nan] = 0x7FC0
    return bits


# ----------------------------------------------------------------------------- routing

def router_logits(x: np.ndarray, router_w: np.ndarray, router_bias=None,
                  chunk: int = 8) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W[e, h] (+ bias[e]), in f64.

    x: f64 [T, H] (exact bf16 values), W: f32 [E, H].  Each product is exact in
    f64; every row is reduced by the same summation, so two identical router
    rows give identical logits.  Reading: the optional bias is added to the
    logits before selection and softmax.
    """
    W = np.asarray(router_w, dtype=np.float64)
    T = x.shape[0]
    out = np.empty((T, W.shape[0]), dtype=np.float64)
    for t0 in range(0, T, chunk):
        xs = x[t0:t0 + chunk]
        out[t0:t0 + chunk] = (xs[:, None, :] * W[None, :, :]).sum(axis=-1)
    if router_bias is not None:
        out += np.asarray(router_bias, dtype=np.float64)[None, :]
    return out


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """idx[t, 0..k-1]: experts in descending logit order, ties to the lower index.

    Reading: selection is on logits, not on probabilities (softmax is strictly
    increasing, so the order is the same, and logits keep distinct values apart).
    """
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("top_k must be in [1, E]")
    idx = np.empty((T, k), dtype=np.int64)
    e_ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((e_ids, -logits[t]))  # primary: -logit, then index
        idx[t] = order[:k]
    return idx


def topk_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Softmax over all experts, keep the selected, renormalise over them.

    The full softmax's common factor cancels, so this equals the softmax over
    the k selected logits; it is evaluated that way, shifted by the largest.
    Reading: no extra routed scaling factor, no shared expert.
    """
    sel = np.take_along_axis(logits, idx, axis=1)
    ex = np.exp(sel - sel[:, :1])
    return ex / ex.sum(axis=1, keepdims=True)


def permutation(idx: np.ndarray, n_experts: int):
    """Counting sort of pairs p = t*k + r by expert, stable in p.

    Returns counts [E], offsets [E+1] (exclusive scan), perm [P] (position ->
    pair) and inv [P] (pair -> position).
    """
    flat = idx.reshape(-1)
    P = flat.size
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    perm = np.empty(P, dtype=np.int64)
    inv = np.empty(P, dtype=np.int64)
    for p in range(P):
        e = flat[p]
        perm[fill[e]] = p
        inv[p] = fill[e]
        fill[e] += 1
    return counts, offsets, perm, inv


# ----------------------------------------------------------------------------- experts

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + e^-z) (reading: no clamp, no bias)."""
    return z / (1.0 + np.exp(-z))


def expert_ffn(x_rows: np.ndarray, w13_e: np.ndarray, w2_e: np.ndarray):
    """SwiGLU expert on rows x [n, H] with dequantised W13 [2I, H], W2 [H, I].

    Returns (h [n, I], y [n, H]).  Gate rows are W13[:I], up rows W13[I:].
    """
    inter = w13_e.shape[0] // 2
    g = x_rows @ w13_e[:inter].T
    u = x_rows @ w13_e[inter:].T
    h = silu(g) * u
    y = h @ w2_e.T
    return h, y


def combine(wts: np.ndarray, y_pairs: np.ndarray) -> np.ndarray:
    """out[t] = sum_r wts[t, r] * y[t, r], summed in rank order r = 0..k-1."""
    out = np.zeros((y_pairs.shape[0], y_pairs.shape[2]), dtype=np.float64)
    for r in range(y_pairs.shape[1]):
        out += wts[:, r:r + 1] * y_pairs[:, r, :]
    return out


# ----------------------------------------------------------------------------- the layer

def moe_forward(x_bits, router_w, router_bias, w13, s13, w2, s2, top_k: int,
                tokens=None, keep_h: bool = False) -> dict:
    """The whole layer in f64.

    x_bits: bf16 bit patterns [T, H]; router_w f32 [E, H]; router_bias f32 [E]
    or None; w13 e4m3 [E, 2I, H] with s13 f32 [E, 2I/128, H/128]; w2 e4m3
    [E, H, I] with s2 f32 [E, H/128, I/128].

    Routing (logits, idx, wts, counts, offsets, perm, inv) is computed for all
    T tokens.  The expert FFN and the output are computed for ``tokens`` (a
    list of token ids; default all), so that a sample of a large batch can be
    checked one token at a time.  Returns a dict of numpy arrays; ``out`` is
    f64 [len(tokens), H] before rounding and ``out_bf16`` its bf16 bits;
    ``y`` is f64 [len(tokens), k, H] (per pair, rank order) and, with
    ``keep_h``, ``h`` is f64 [len(tokens), k, I].
    """
    x = bf16_to_f64(x_bits)
    T, H = x.shape
    E = router_w.shape[0]
    inter = w13.shape[1] // 2
    logits = router_logits(x, router_w, router_bias)
    idx = select_topk(logits, top_k)
    wts = topk_weights(logits, idx)
    counts, offsets, perm, inv = permutation(idx, E)

    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = np.zeros((tok.size, top_k, H), dtype=np.float64)
    h = np.zeros((tok.size, top_k, inter), dtype=np.float64) if keep_h else None
    if tok.size:
        sel = idx[tok]                       # [n, k]
        for e in np.unique(sel):
            rows_t, rows_r = np.nonzero(sel == e)
            w13_e = dequantize(w13[e], s13[e])
            w2_e = dequantize(w2[e], s2[e])
            h_e, y_e = expert_ffn(x[tok[rows_t]], w13_e, w2_e)
            y[rows_t, rows_r] = y_e
            if keep_h:
                h[rows_t, rows_r] = h_e
    out = combine(wts[tok], y)
    res = dict(logits=logits, idx=idx, wts=wts, counts=counts, offsets=offsets, perm=perm,
               inv=inv, tokens=tok, y=y, out=out, out_bf16=round_to_bf16(out))
    if keep_h:
        res["h"] = h
    return res
