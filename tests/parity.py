"""Tolerance checks and oracle-side expected values for the GPU parity tests.

Every bound is the stated target for a correctly rounded result plus, where
noted, the fp32 evaluation error of the kernel's arithmetic (the kernels
compute in fp32, the oracle in float64).  Where cancellation makes the
result much smaller than the values it is computed from, a 1-ulp bound on
the result would require more precision than fp32 has; the extra term is
what fp32 evaluation of the same formula can be off by.  Each check counts
the elements that are within tolerance only because of that extra term, and
the tests bound and report the count.

  * fp32 results: |got - ref| <= 1e-5 |ref| + k * 2^-24 * T
  * bf16 / f16 results: |got - ref| <= 1 ulp(ref) + k * 2^-24 * T,
    k = 8, where T is the magnitude of the terms the kernel adds in fp32
    (for z: |x - mu| rsigma |g'| + |beta|, plus mean|x| rsigma |g'| for
    LayerNorm, the summands of mu standing for its fp32 error; for dx: rsigma (|dy| +
    mean|dy| + |xhat| mean|dy xhat|) + |dresidual|, the summands of c1 =
    mean(dy) and c2 = mean(dy xhat) standing for their fp32 error).
  * mu: rel 1e-4 plus 64 * 2^-24 * mean|x| (an fp32 sum of the row);
    rsigma: rel 1e-4.
  * The counts of elements relying on the fp32 term are bounded by 0.1% of
    the elements (z, dx, mu) or 2% (dgamma / dbeta, whose exact value is a
    sum over all rows that often nearly cancels), plus two elements.
  * dgamma / dbeta: rel 1e-4 plus 1e-6 * sum_i |term_i| (fp32 partial
    sums over all rows; far below one row's contribution, so a dropped or
    doubled row still fails).  bf16 weights: 1 bf16 ulp plus the same.
  * E4M3 codes: within 1 step everywhere, at most 0.1% of codes differ.
  * E8M0 scales: bit-exact except blocks whose amax lies within 4 fp32
    ulp of a power of two (counted, bounded).
  * amax, delayed scaling: bit-exact against max|z| of the kernel's own
    fp32 z (``kernel_z32``, from the kernel's saved statistics), rel 1e-5
    against the oracle.

Set GBN_PARITY_REPORT to a file path to have every count appended there as
one JSON line per check.
"""
from __future__ import annotations

import json
import os

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


def report(kind, name, count, total, **extra):
    """Prints one count of a parity check and appends it to GBN_PARITY_REPORT."""
    print(f"[parity] {kind} {name}: {count} of {total}", flush=True)
    path = os.environ.get("GBN_PARITY_REPORT")
    if path:
        rec = {"kind": kind, "name": name, "count": int(count), "total": int(total)}
        rec.update(extra)
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


class Tally:
    """Accumulates the counts of several chunked checks of one output, then
    bounds and reports the total once."""

    def __init__(self, kind, name, max_frac):
        self.kind, self.name, self.max_frac = kind, name, max_frac
        self.count = 0
        self.total = 0

    def add(self, count, total):
        self.count += int(count)
        self.total += int(total)

    def close(self, **extra):
        report(self.kind, self.name, self.count, self.total, **extra)
        assert self.count <= self.max_frac * self.total + 2, (
            f"{self.name}: {self.count} of {self.total} {self.kind} exceed the bound "
            f"{self.max_frac:g}")
        return self.count


def check_float(name, got, ref, dtype, terms=None, rel=None, k=8.0, max_relied=1e-3,
                tally=None):
    """got: torch tensor (any device) of dtype; ref: float64 oracle values.

    Returns the number of elements whose error exceeds the stated bound
    (1 ulp, or ``rel`` |ref|) and that pass only through the fp32 evaluation
    term k 2^-24 T.  That count is bounded by max_relied of the elements and
    reported -- or, with ``tally``, added to it for the caller to bound."""
    g = to64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    if dtype == torch.float32 or rel is not None:
        base = (rel if rel is not None else 1e-5) * np.abs(ref)
    else:
        base = ulp(ref, dtype)
    allowed = base
    if terms is not None:
        allowed = base + k * TWO_M24 * np.asarray(terms, dtype=np.float64)
    nan_ok = np.isnan(g) == np.isnan(ref)
    assert nan_ok.all(), f"{name}: NaN pattern differs"
    err = np.abs(np.nan_to_num(g) - np.nan_to_num(ref))
    bad = err > allowed
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), g[tuple(i)], ref[tuple(i)], allowed[tuple(i)]) for i in idx]
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance, e.g. {detail}")
    relied = int((err > base).sum()) if terms is not None else 0
    if tally is not None:
        tally.add(relied, err.size)
    elif terms is not None:
        report("relied-on-fp32-term", name, relied, err.size)
        assert relied <= max_relied * err.size + 2, (
            f"{name}: {relied} of {err.size} elements pass only through the fp32 term")
    return relied


WGRAD_K = 1e-6 / TWO_M24   # dgamma / dbeta: 1e-6 * sum_i |term_i|


def check_wgrad(name, got, ref, dtype, terms, tally=None):
    """dgamma / dbeta: rel 1e-4 (fp32 weights) or 1 ulp (bf16 / f16 weights)
    plus 1e-6 * sum_i |term_i|; at most 2% of the columns may rely on the
    second term."""
    return check_float(name, got, ref, dtype, terms=terms, k=WGRAD_K,
                       rel=1e-4 if dtype == torch.float32 else None, max_relied=2e-2,
                       tally=tally)


def e4m3_ordinal(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def is_e4m3_nan(codes):
    return (codes.astype(np.int32) & 0x7F) == 0x7F


def check_codes(name, got, ref, max_frac=1e-3, mask=None, report_it=True):
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
    if report_it:
        report("e4m3-codes-one-step-off", name, int((d != 0).sum()), d.size)
    return frac


def near_pow2(a: np.ndarray, ulps=4) -> np.ndarray:
    a = a.astype(np.float64)
    hi = np.floor(np.log2(np.maximum(a * (1 + ulps * 2.0 ** -23), 1e-300)))
    lo = np.floor(np.log2(np.maximum(a * (1 - ulps * 2.0 ** -23), 1e-300)))
    return (hi != lo) & (a > 0)


def check_scales(name, got, ref, block_amax, max_near=1e-3, tally=None):
    """E8M0 scales bit-exact except blocks whose amax is within 4 ulp of a
    power of two, where they may differ by one.  Returns the number of blocks
    that differ (all of them near a power of two); it is bounded by max_near
    of the blocks and reported -- or, with ``tally``, added to it."""
    g = got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape
    amb = near_pow2(block_amax)
    diff = g != r
    assert not (diff & ~amb).any(), f"{name}: {(diff & ~amb).sum()} scales differ"
    assert (np.abs(g.astype(int) - r.astype(int)) <= 1).all()
    n = int((diff & amb).sum())
    if tally is not None:
        tally.add(n, g.size)
    else:
        report("e8m0-near-power-of-two", name, n, g.size, near=int(amb.sum()))
        assert n <= max_near * g.size + 2
    return n


# ---------------------------------------------------------------- the kernel's fp32 z

def fma_f32(a, b, c):
    """fl32(a * b + c) rounded once, as the fp32 fused multiply-add, for
    float32 arrays.  The product is exact in float64 (24 + 24 bits); the sum
    is held as a float64 value s plus its exact error e (two-sum), and the
    float32 rounding of s + e is that of s, except where s lies exactly
    halfway between two float32 values and e is not zero: there the sign of
    e picks the neighbour."""
    a64 = np.asarray(a, np.float32).astype(np.float64)
    b64 = np.asarray(b, np.float32).astype(np.float64)
    c64 = np.asarray(c, np.float32).astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        p = a64 * b64
        s = p + c64
        bv = s - p
        e = (p - (s - bv)) + (c64 - bv)
        r = s.astype(np.float32)
        r64 = r.astype(np.float64)
        other = 2.0 * s - r64              # the neighbour on the other side, if s is a midpoint
        mid = (s != r64) & np.isfinite(s) & (other.astype(np.float32).astype(np.float64) == other)
        flip = mid & (e != 0) & (np.sign(e) == np.sign(other - r64))
    return np.where(flip, other.astype(np.float32), r)


def kernel_z32(x, gamma, beta, mu, rs, norm, zcg):
    """z exactly as the kernels evaluate it in fp32, from the statistics the
    kernel saved (its fp32 mu and rsigma): g' = fl(gamma + 1) or gamma;
    LayerNorm z = fma(fl(fl(x - mu) * rsigma), g', beta), RMSNorm
    z = fl(fl(x * rsigma) * g').  Every forward kernel of the library
    evaluates z in this order (packed-pair or scalar fp32, round to nearest
    even, no flush of subnormals).  Returns float32 [rows, hidden]."""
    x32 = to64(x).astype(np.float32) if not isinstance(x, np.ndarray) else x.astype(np.float32)
    g = to64(gamma).astype(np.float32)
    if zcg:
        g = (g + np.float32(1.0)).astype(np.float32)
    r = np.asarray(rs, np.float32)[:, None]
    with np.errstate(invalid="ignore", over="ignore"):
        if norm == 0:
            m = np.asarray(mu, np.float32)[:, None]
            t = ((x32 - m).astype(np.float32) * r).astype(np.float32)
            b = to64(beta).astype(np.float32)
            return fma_f32(t, np.broadcast_to(g, t.shape), np.broadcast_to(b, t.shape))
        t = (x32 * r).astype(np.float32)
        return (t * g[None, :]).astype(np.float32)


def amax_f32(z32):
    """max |z| of float32 values, NaN if any is NaN (as the kernels' max)."""
    a = np.abs(np.asarray(z32, np.float32))
    if a.size == 0:
        return np.float32(0.0)
    if np.isnan(a).any():
        return np.float32(np.nan)
    return np.float32(a.max())


def same_f32_bits(a, b):
    """Equal float32 bit patterns, or both NaN."""
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a.view(np.uint32) == b.view(np.uint32)


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
