"""Pins of the softmax oracle against what the mathematics fixes: torch's
float64 softmax with -inf masking (a library routine), closed forms, the
mask shapes, invariants, and central finite differences for the backward."""
import math

import numpy as np
import pytest
import torch

from oracle import softmax as S


def _rng(seed=0):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("kind", [S.NONE, S.PADDING, S.CAUSAL_UPPER, S.CAUSAL_ALIGNED])
def test_forward_matches_torch_float64(kind):
    g = _rng(1)
    b, h, sq, sk = 3, 2, 5, 5 if kind == S.CAUSAL_UPPER else 7
    x = g.normal(size=(b, h, sq, sk)) * 3
    pad = (g.random(size=(1, 1, sq, sk)) < 0.3) if kind == S.PADDING else None
    y = S.softmax_fwd(x, kind, 0.7, pad)
    keep = torch.from_numpy(S.keep_mask(kind, b, h, sq, sk, pad))
    t = torch.from_numpy(x * 0.7).masked_fill(~keep, float("-inf"))
    ref = torch.softmax(t, dim=-1)
    ref = torch.nan_to_num(ref, nan=0.0)               # fully masked rows: 0 by the reading
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=1e-15)


def test_uniform_row_and_two_element_closed_form():
    y = S.softmax_fwd(np.full((1, 1, 1, 9), 2.5), S.NONE, 1.3)
    assert np.all(y == 1.0 / 9.0)
    a, c = 0.4, -1.1
    y = S.softmax_fwd(np.array([[[[a, c]]]]), S.NONE, 2.0)
    assert y[0, 0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(2.0 * (c - a))), rel=1e-15)


def test_mask_shapes():
    sq, sk = 4, 6
    up = S.keep_mask(S.CAUSAL_UPPER, 1, 1, 5, 5)[0, 0]
    assert [int(r.sum()) for r in up] == [1, 2, 3, 4, 5]
    al = S.keep_mask(S.CAUSAL_ALIGNED, 1, 1, sq, sk)[0, 0]
    assert [int(r.sum()) for r in al] == [3, 4, 5, 6]          # last row sees every key
    al2 = S.keep_mask(S.CAUSAL_ALIGNED, 1, 1, 6, 4)[0, 0]
    assert [int(r.sum()) for r in al2] == [0, 0, 1, 2, 3, 4]   # rows before the keys: none
    pad = np.zeros((2, 1, 2, 3), dtype=np.uint8)
    pad[1, 0, 0, 2] = 1
    k = S.keep_mask(S.PADDING, 4, 3, 2, 3, pad)
    assert k[0].all() and k[2].all()                           # batch 0, 2 -> mask batch 0
    assert not k[1, :, 0, 2].any() and not k[3, :, 0, 2].any() # batch 1, 3 -> mask batch 1
    assert k[1, :, 1].all()


def test_invariants_masked_zero_rows_sum_one_shift():
    g = _rng(2)
    x = g.normal(size=(2, 3, 6, 9)) * 4
    for kind in (S.NONE, S.CAUSAL_ALIGNED):
        y = S.softmax_fwd(x, kind, 1.0)
        keep = S.keep_mask(kind, 2, 3, 6, 9)
        assert np.all(y[~keep] == 0.0)
        np.testing.assert_allclose(y.sum(-1), 1.0, rtol=0, atol=1e-14)
        np.testing.assert_allclose(S.softmax_fwd(x + 123.25, kind, 1.0), y, rtol=1e-12, atol=0)


def test_fully_masked_row_is_zero():
    y = S.softmax_fwd(np.ones((1, 1, 6, 4)), S.CAUSAL_ALIGNED, 1.0)
    assert np.all(y[0, 0, :2] == 0.0) and np.all(np.abs(y[0, 0, 2:].sum(-1) - 1) < 1e-15)


@pytest.mark.parametrize("kind", [S.NONE, S.CAUSAL_UPPER])
def test_backward_finite_differences(kind):
    g = _rng(3)
    sk = 6
    x = g.normal(size=(1, 1, sk, sk))
    w = g.normal(size=(1, 1, sk, sk))
    scale = 0.8
    y = S.softmax_fwd(x, kind, scale)
    dx = S.softmax_bwd(w, y, scale)
    hstep = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += hstep
        xm[idx] -= hstep
        num[idx] = ((w * S.softmax_fwd(xp, kind, scale)).sum()
                    - (w * S.softmax_fwd(xm, kind, scale)).sum()) / (2 * hstep)
    np.testing.assert_allclose(dx, num, rtol=1e-6, atol=1e-9)


def test_backward_rows_sum_to_zero_and_masked_zero():
    g = _rng(4)
    x = g.normal(size=(2, 2, 5, 5))
    y = S.softmax_fwd(x, S.CAUSAL_UPPER, 1.5)
    dx = S.softmax_bwd(g.normal(size=x.shape), y, 1.5)
    np.testing.assert_allclose(dx.sum(-1), 0.0, atol=1e-14)
    assert np.all(dx[~S.keep_mask(S.CAUSAL_UPPER, 2, 2, 5, 5)] == 0.0)
