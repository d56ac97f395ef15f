"""Tolerance checks and oracle-side expected values for the GPU parity tests.

Tolerances (from the stated targets, with the fp32 evaluation error of the
kernel's arithmetic added where cancellation can make a 1-ulp bound on the
result meaningless):
  * fp32 results: |got - ref| <= 1e-5 |ref| + 8 * 2^-24 * T
  * bf16 / f16 results: |got - ref| <= 1 ulp(ref) + 8 * 2^-24 * T
    where T is the magnitude of the terms the kernel adds in fp32
    (for z: |x - mu| rsigma |g'| + |beta|, plus mean|x| rsigma |g'| for
    LayerNorm, the summands of mu standing for its fp32 error; for dx: rsigma (|dy| +
    mean|dy| + |xhat| mean|dy xhat|) + |dresidual|, the summands of c1 =
    mean(dy) and c2 = mean(dy xhat) standing for their fp32 error).
  * mu / rsigma: rel 1e-4 (plus the same fp32 term bound for mu).
  * dgamma / dbeta: rel 1e-4 plus 1e-6 * sum_i |term_i| (fp32 partial sums
    over all rows; far below one row's contribution, so a dropped or doubled
    row still fails).  bf16 weights: 1 bf16 ulp plus the same.
  * E4M3 codes: within 1 step everywhere, at most 0.1% of codes differ.
  * E8M0 scales: bit-exact except blocks whose amax lies within 4 fp32 ulp of
    a power of two (counted).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TWO_M24 = 2.0 ** -24


def ulp(ref: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the format `dtype` at |ref| (round-to-nearest half-spacing * 2)."""
    mant, emin = {torch.float32: (23, -126), torch.bfloat16: (7, -126),
                  torch.float16: (10, -14)}[dtype]
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - mant).astype(np.int64))


def to64(t) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def check_float(name, got, ref, dtype, terms=None, rel=None, k=8.0):
    """got: torch tensor (any device) of dtype; ref: float64 oracle values."""
    g = to64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    if dtype == torch.float32 or rel is not None:
        allowed = (rel if rel is not None else 1e-5) * np.abs(ref)
    else:
        allowed = ulp(ref, dtype)
    if terms is not None:
        allowed = allowed + k * TWO_M24 * np.asarray(terms, dtype=np.float64)
    nan_ok = np.isnan(g) == np.isnan(ref)
    assert nan_ok.all(), f"{name}: NaN pattern differs"
    err = np.abs(np.nan_to_num(g) - np.nan_to_num(ref))
    bad = err > allowed
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), g[tuple(i)], ref[tuple(i)], allowed[tuple(i)]) for i in idx]
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance, e.g. {detail}")


def e4m3_ordinal(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def is_e4m3_nan(codes):
    return (codes.astype(np.int32) & 0x7F) == 0x7F


def check_codes(name, got, ref, max_frac=1e-3, mask=None):
    """E4M3 codes within one step, at most max_frac of them different."""
    g = got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    if mask is not None:
        g, r = g[mask], r[mask]
    gn, rn = is_e4m3_nan(g), is_e4m3_nan(r)
    assert (gn == rn).all(), f"{name}: NaN codes differ"
    d = np.abs(e4m3_ordinal(g) - e4m3_ordinal(r))
    d[gn] = 0
    assert d.max(initial=0) <= 1, f"{name}: a code differs by {d.max()} steps"
    frac = (d != 0).mean() if d.size else 0.0
    assert frac <= max_frac, f"{name}: {frac:.4%} of codes differ"
    return frac


def near_pow2(a: np.ndarray, ulps=4) -> np.ndarray:
    a = a.astype(np.float64)
    hi = np.floor(np.log2(np.maximum(a * (1 + ulps * 2.0 ** -23), 1e-300)))
    lo = np.floor(np.log2(np.maximum(a * (1 - ulps * 2.0 ** -23), 1e-300)))
    return (hi != lo) & (a > 0)


def check_scales(name, got, ref, block_amax):
    """E8M0 scales bit-exact except blocks whose amax is within 4 ulp of a power of two."""
    g = got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape
    amb = near_pow2(block_amax)
    diff = g != r
    assert not (diff & ~amb).any(), f"{name}: {(diff & ~amb).sum()} scales differ"
    assert (np.abs(g.astype(int) - r.astype(int)) <= 1).all()
    return int((diff & amb).sum())


# ---------------------------------------------------------------- expected values

def z_terms(x, gamma, beta, mu, rs, norm, zcg):
    """Magnitude of the fp32 terms of z per element: |x - mu| rsigma |g'| +
    |beta|, and for LayerNorm mean_j |x_j| rsigma |g'| -- the kernel's mu is
    an fp32 sum of the row, whose evaluation error scales with its summands,
    not with |x - mu| (an element close to the mean would otherwise get no
    room for it)."""
    xd = to64(x) if not isinstance(x, np.ndarray) else x
    g = to64(gamma) + (1.0 if zcg else 0.0)
    t = np.abs(xd - (mu[:, None] if norm == 0 else 0.0)) * rs[:, None] * np.abs(g)[None, :]
    if norm == 0:
        t = t + np.abs(xd).mean(axis=1, keepdims=True) * rs[:, None] * np.abs(g)[None, :]
    if beta is not None and norm == 0:
        t = t + np.abs(to64(beta))[None, :]
    return t


def block_amax_rowwise(z):
    a = np.abs(z.astype(np.float32)).astype(np.float64)
    r, h = a.shape
    return a.reshape(r, h // 32, 32).max(axis=2)


def block_amax_colwise(z):
    a = np.abs(z.astype(np.float32)).astype(np.float64)
    r, h = a.shape
    return a.reshape(r // 32, 32, h).max(axis=1)


def bwd_terms(dz, x, mu, rs, gamma, dres, norm, zcg):
    """Magnitudes for the dx tolerance and the dgamma/dbeta sums."""
    dzd = to64(dz)
    xd = to64(x)
    g = to64(gamma) + (1.0 if zcg else 0.0)
    mu64 = np.zeros(xd.shape[0]) if mu is None else np.asarray(mu, np.float64)
    rs64 = np.asarray(rs, np.float64)
    xh = (xd - mu64[:, None]) * rs64[:, None]
    dy = dzd * g[None, :]
    # c1 = mean(dy) and c2 = mean(dy * xhat) are fp32 sums: their evaluation
    # error scales with the magnitude of their summands, not with |c1|, |c2|
    # (which cancellation can make arbitrarily small).
    m1 = np.abs(dy).mean(1, keepdims=True) if norm == 0 else 0.0
    m2 = np.abs(dy * xh).mean(1, keepdims=True)
    t_dx = rs64[:, None] * (np.abs(dy) + m1 + np.abs(xh) * m2)
    if dres is not None:
        t_dx = t_dx + np.abs(to64(dres))
    t_dg = np.abs(dzd * xh).sum(0)
    t_db = np.abs(dzd).sum(0)
    return t_dx, t_dg, t_db
