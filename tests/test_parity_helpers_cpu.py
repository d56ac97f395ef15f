"""The parity helpers that stand in for the kernel's own fp32 arithmetic:
``fma_f32`` (one rounding of a*b + c to float32) against exact rational
arithmetic, ``kernel_z32`` against the same, and the counting of elements that
rely on the fp32 evaluation term."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from parity import Tally, amax_f32, check_float, fma_f32, kernel_z32, same_f32_bits


def _round_f32(q: Fraction) -> np.float32:
    """Exact round-to-nearest-even of a rational to float32 (normal range)."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    e = max(e, -126)
    step = Fraction(2) ** (e - 23)
    n = q / step
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return np.float32(sign * float(lo * step))


def _exact_fma(a, b, c):
    return _round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def test_fma_f32_matches_exact_rounding_on_random_triples():
    g = np.random.default_rng(5)
    a = (g.standard_normal(3000) * 10.0 ** g.uniform(-3, 3, 3000)).astype(np.float32)
    b = (g.standard_normal(3000) * 10.0 ** g.uniform(-3, 3, 3000)).astype(np.float32)
    c = (g.standard_normal(3000) * 10.0 ** g.uniform(-6, 6, 3000)).astype(np.float32)
    got = fma_f32(a, b, c)
    want = np.array([_exact_fma(*t) for t in zip(a, b, c)], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fma_f32_ties_decided_by_the_low_part():
    # a*b = 1.5 + 2^-23 + 2^-24 lies exactly halfway between two float32
    # values; a tiny c decides the direction, c = 0 ties to even.
    a = np.float32(1.0 + 2.0 ** -23)
    b = np.float32(1.5)
    p = 1.5 + 1.5 * 2.0 ** -23
    lo, hi = np.float32(1.5 + 2.0 ** -23), np.float32(1.5 + 2.0 ** -22)
    assert float(lo) < p < float(hi)
    for c, want in [(2.0 ** -60, hi), (-(2.0 ** -60), lo), (0.0, hi if int(lo.view(np.uint32)) & 1
                                                             else lo)]:
        got = fma_f32(np.array([a]), np.array([b]), np.array([np.float32(c)]))[0]
        assert got == want == _exact_fma(a, b, np.float32(c)), (c, got, want)
    # a product at a midpoint with a plain float32 c of the same size
    c = np.float32(3.0)
    assert fma_f32(np.array([a]), np.array([b]), np.array([c]))[0] == _exact_fma(a, b, c)


def test_fma_f32_nan_and_inf():
    a = np.array([np.nan, 1.0, np.inf, 3e38], np.float32)
    b = np.array([1.0, np.nan, 0.0, 10.0], np.float32)
    c = np.array([0.0, 0.0, 1.0, 0.0], np.float32)
    r = fma_f32(a, b, c)
    assert np.isnan(r[0]) and np.isnan(r[1]) and np.isnan(r[2]) and np.isinf(r[3])


@pytest.mark.parametrize("norm,zcg", [(0, False), (0, True), (1, False), (1, True)])
def test_kernel_z32_is_the_stated_fp32_sequence(norm, zcg):
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(6, 40, generator=g) * 3 + 0.5).to(torch.bfloat16)
    gamma = (torch.randn(40, generator=g) * 0.1 + (0.0 if zcg else 1.0))
    beta = torch.randn(40, generator=g) * 0.1
    mu = (torch.randn(6, generator=g) * 0.2).numpy().astype(np.float32)
    rs = (torch.rand(6, generator=g) + 0.5).numpy().astype(np.float32)
    z = kernel_z32(x, gamma, beta if norm == 0 else None, mu, rs, norm, zcg)
    xf = x.float().numpy()
    gf = gamma.numpy().astype(np.float32)
    for i in range(6):
        for j in range(40):
            gp = _round_f32(Fraction(float(gf[j])) + 1) if zcg else gf[j]
            if norm == 0:
                d = _round_f32(Fraction(float(xf[i, j])) - Fraction(float(mu[i])))
                t = _round_f32(Fraction(float(d)) * Fraction(float(rs[i])))
                want = _exact_fma(t, gp, np.float32(beta[j]))
            else:
                t = _round_f32(Fraction(float(xf[i, j])) * Fraction(float(rs[i])))
                want = _round_f32(Fraction(float(t)) * Fraction(float(gp)))
            assert z[i, j] == want, (i, j, z[i, j], want)


def test_amax_f32_and_bit_comparison():
    assert same_f32_bits(amax_f32(np.array([[1.0, -3.5], [2.0, 0.0]], np.float32)), 3.5)
    assert np.isnan(amax_f32(np.array([1.0, np.nan], np.float32)))
    assert same_f32_bits(np.float32(np.nan), np.float32(np.nan))
    assert not same_f32_bits(np.float32(1.0), np.nextafter(np.float32(1.0), np.float32(2.0)))
    assert amax_f32(np.zeros((0, 4), np.float32)) == 0.0


def test_check_float_counts_elements_that_rely_on_the_fp32_term():
    ref = np.array([1e-6, 1e-6, 1e-6, 2.0])
    got = torch.tensor([1.3e-6, 1.3e-6, 1.3e-6, 2.0], dtype=torch.float32)
    # the first three are far beyond rel 1e-5 of their tiny value, but within
    # 8 * 2^-24 * T for T = 1 (the magnitude they were computed from)
    n = check_float("x", got, ref, torch.float32, terms=np.ones(4), max_relied=0.25)
    assert n == 3
    # the bound: max_relied of the elements plus two
    with pytest.raises(AssertionError):
        check_float("x", got, ref, torch.float32, terms=np.ones(4), max_relied=0.1)
    with pytest.raises(AssertionError):   # beyond the fp32 term too
        check_float("x", got, ref, torch.float32, terms=np.full(4, 0.1))
    t = Tally("relied-on-fp32-term", "x", 0.3)
    check_float("x", got, ref, torch.float32, terms=np.ones(4), tally=t)
    check_float("x", got, ref, torch.float32, terms=np.ones(4), tally=t)
    assert (t.count, t.total) == (6, 8)
    with pytest.raises(AssertionError):
        t.close()
