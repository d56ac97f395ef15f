"""CPU oracle for the scaled (masked) softmax forward and backward.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: the tests, the smoke
check and the benchmark's CPU legs use it; the product path never does.

The kernels are named on "Migrate norms and softmax kernels to NVRTC"
(Description: scaled_masked_softmax, scaled_upper_triang_masked_softmax,
scaled_aligned_causal_masked_softmax, forward and backward; JIT compilation
cost table).  The page gives no formulas, so these are the plain definitions
(readings, listed with the norms' readings):

* forward: y = softmax over the last axis of scale * x, taken over the
  positions the mask keeps; masked positions are 0; a row with no kept
  position is all 0;
* padding mask: mask [mask_batches, 1, sq, sk], nonzero = masked out,
  broadcast over heads, batch b uses mask batch b % mask_batches;
* upper-triangular (causal, sq == sk): (i, j) kept iff j <= i;
* aligned causal (bottom-right aligned): (i, j) kept iff j <= i + (sk - sq);
* backward: dx = scale * y * (dy - sum_j dy * y), from the forward's stored
  output y (the softmax Jacobian applied to dy, times the input scale).

Everything is float64 numpy, one result rounded once to the output type by
``oracle.round_to``.
"""
from __future__ import annotations

import numpy as np

NONE, PADDING, CAUSAL_UPPER, CAUSAL_ALIGNED = 0, 1, 2, 3


def keep_mask(kind: int, batches: int, heads: int, sq: int, sk: int, pad_mask=None):
    """bool [batches, heads, sq, sk]: True where the position takes part."""
    i = np.arange(sq)[:, None]
    j = np.arange(sk)[None, :]
    if kind == NONE:
        k = np.ones((sq, sk), dtype=bool)
    elif kind == CAUSAL_UPPER:
        assert sq == sk
        k = j <= i
    elif kind == CAUSAL_ALIGNED:
        k = j <= i + (sk - sq)
    elif kind == PADDING:
        m = np.asarray(pad_mask).astype(bool)          # [mb, 1, sq, sk], True = masked
        mb = m.shape[0]
        sel = np.arange(batches) % mb
        return np.broadcast_to(~m[sel], (batches, heads, sq, sk)).copy()
    else:
        raise ValueError(kind)
    return np.broadcast_to(k, (batches, heads, sq, sk)).copy()


def softmax_fwd(x, kind: int, scale: float, pad_mask=None):
    """y (float64) of x [batches, heads, sq, sk] (any float type, widened exactly)."""
    x = np.asarray(x, dtype=np.float64)
    b, h, sq, sk = x.shape
    keep = keep_mask(kind, b, h, sq, sk, pad_mask)
    t = np.where(keep, scale * x, -np.inf)
    m = t.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)               # rows with nothing kept
    e = np.where(keep, np.exp(t - m), 0.0)
    s = e.sum(axis=-1, keepdims=True)
    return np.where(s > 0, e / np.where(s > 0, s, 1.0), 0.0)


def softmax_bwd(dy, y, scale: float):
    """dx (float64) = scale * y * (dy - sum(dy * y)) over the last axis."""
    dy = np.asarray(dy, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    c = (dy * y).sum(axis=-1, keepdims=True)
    return scale * y * (dy - c)
