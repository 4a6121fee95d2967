"""The host restatement of the combine's f32 fma chain (tests/host_ref.py)
against exact rational arithmetic (no GPU)."""
from fractions import Fraction

import numpy as np

from host_ref import combine_f32, fma_f32


def _exact_fma(a, b, c) -> np.float32:
    v = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    # nearest f32 by bracketing: candidates around the f64 approximation
    f = np.float32(float(v))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    best = min(cands, key=lambda x: (abs(Fraction(float(x)) - v),
                                     int(np.array([x]).view(np.uint32)[0]) & 1))
    return best


def test_fma_matches_exact_rounding_on_random_values():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(4000) * 2.0 ** rng.integers(-8, 8, 4000)).astype(np.float32)
    b = (rng.standard_normal(4000) * 2.0 ** rng.integers(-8, 8, 4000)).astype(np.float32)
    c = (rng.standard_normal(4000) * 2.0 ** rng.integers(-8, 8, 4000)).astype(np.float32)
    got = fma_f32(a, b, c)
    want = np.array([_exact_fma(x, y, z) for x, y, z in zip(a, b, c)], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fma_resolves_double_rounding_ties():
    # a*b = 2^-24 (1 - 2^-40): c + a*b rounds in f64 exactly onto the midpoint
    # of two f32 values; the exact sum lies below it
    a = np.float32(2.0 ** -24 * (1 + 2.0 ** -20))
    b = np.float32(1 - 2.0 ** -20)
    for c in (np.float32(1 + 2.0 ** -23), np.float32(1.0), np.float32(-(1 + 2.0 ** -23))):
        for sa in (a, -a):
            got = fma_f32(np.array([sa]), np.array([b]), np.array([c]))[0]
            assert got == _exact_fma(sa, b, c), (sa, c)
    # the naive double rounding would give the even neighbour instead
    naive = np.float32(float(a) * float(b) + float(np.float32(1 + 2.0 ** -23)))
    assert naive != fma_f32(np.array([a]), np.array([b]), np.array([np.float32(1 + 2.0 ** -23)]))[0]


def test_combine_chain_order():
    # two pairs per token; the chain starts from zero in rank order
    y = np.array([[[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0]]], dtype=np.float32)
    inv = np.array([2, 0, 1, 3])
    w = np.array([[0.25, 0.75], [0.5, 0.5]], dtype=np.float32)
    acc = combine_f32(y, inv, w)
    assert acc.tolist() == [[0.25 * 5 + 0.75 * 1, 0.25 * 6 + 0.75 * 2], [0.5 * 3 + 0.5 * 7, 0.5 * 4 + 0.5 * 8]]


def test_bf16_half_ulp_bounds_the_correct_rounding():
    import oracle
    from harness import bf16_half_ulp
    rng = np.random.default_rng(5)
    v = rng.standard_normal(20000) * 2.0 ** rng.integers(-20, 20, 20000)
    r = oracle.bf16_to_f64(oracle.round_to_bf16(v))
    assert (np.abs(r - v) <= bf16_half_ulp(v)).all()
    # at a midpoint the bound is attained: 1 + 2^-8 lies halfway between
    # the bf16 values 1 and 1 + 2^-7
    assert bf16_half_ulp(np.array([1.0 + 2.0 ** -8]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([-3.0]))[0] == 2.0 ** -7
