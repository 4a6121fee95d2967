"""Pins of the decode-attention oracle (no GPU): per-element loops with
exactly rounded sums, closed forms, and planted mistakes."""
import math
import struct

import numpy as np

import oracle
from oracle import attention as A


def _bits(a):
    return oracle.round_to_bf16(np.asarray(a, dtype=np.float64))


def _rand(shape, seed):
    return _bits(np.random.default_rng(seed).standard_normal(shape))


def _brute(qb, kb, vb):
    f = lambda b: struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]
    B, nh, d = qb.shape
    S, nkv = kb.shape[1], kb.shape[2]
    g = nh // nkv
    out = np.zeros((B, nh, d))
    for b in range(B):
        for h in range(nh):
            c = h // g
            s = [math.fsum(f(qb[b, h, i]) * f(kb[b, j, c, i]) for i in range(d)) / math.sqrt(d)
                 for j in range(S)]
            m = max(s)
            e = [math.exp(v - m) for v in s]
            z = math.fsum(e)
            for i in range(d):
                out[b, h, i] = math.fsum(e[j] / z * f(vb[b, j, c, i]) for j in range(S))
    return out


def test_matches_brute_force_with_grouped_heads():
    qb, kb, vb = _rand((2, 4, 8), 1), _rand((2, 5, 2, 8), 2), _rand((2, 5, 2, 8), 3)
    got = A.decode_attention(qb, kb, vb)
    want = _brute(qb, kb, vb)
    assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()


def test_closed_forms():
    # identical keys: uniform weights, the output is the mean of the values
    qb = _rand((1, 2, 8), 4)
    kb = np.repeat(_rand((1, 1, 1, 8), 5), 6, axis=1)
    vb = _rand((1, 6, 1, 8), 6)
    got = A.decode_attention(qb, kb, vb)
    mean = oracle.bf16_to_f64(vb)[0, :, 0, :].mean(axis=0)
    assert np.allclose(got[0, 0], mean, rtol=1e-13) and np.allclose(got[0, 1], mean, rtol=1e-13)
    # one key far above the others takes all the weight
    kb2 = np.zeros((1, 3, 1, 8), np.uint16)
    kb2[0, 1, 0, 0] = _bits([64.0])[0]
    q2 = np.zeros((1, 1, 8), np.uint16)
    q2[0, 0, 0] = _bits([64.0])[0]
    got2 = A.decode_attention(q2, kb2, vb[:, :3])
    assert np.allclose(got2[0, 0], oracle.bf16_to_f64(vb)[0, 1, 0], rtol=1e-12)


def test_planted_mistakes_fail():
    qb, kb, vb = _rand((1, 4, 8), 7), _rand((1, 6, 2, 8), 8), _rand((1, 6, 2, 8), 9)
    want = _brute(qb, kb, vb)
    # wrong head grouping (h % nkv instead of h // g)
    q = oracle.bf16_to_f64(qb); K = oracle.bf16_to_f64(kb); V = oracle.bf16_to_f64(vb)
    bad = np.empty_like(want)
    for h in range(4):
        c = h % 2
        s = K[0, :, c] @ q[0, h] / np.sqrt(8)
        p = np.exp(s - s.max())
        bad[0, h] = p / p.sum() @ V[0, :, c]
    assert np.abs(bad - want).max() > 1e-3
    # missing 1/sqrt(d)
    s = K[0, :, 0] @ q[0, 0]
    p = np.exp(s - s.max())
    assert np.abs(p / p.sum() @ V[0, :, 0] - want[0, 0]).max() > 1e-3
