"""torch.autograd functions over the C ABI.

``layer_norm`` / ``rms_norm`` run the library's fused forward (saving mu and
rsigma) and, on backward, its fused backward.  ``*_with_residual`` also return
the input itself as a second, "extra" output (the residual branch of a
pre-norm block); when both outputs receive gradients, the backward adds the
residual's gradient inside the norm's backward kernel instead of in a
separate add ("Implementation:NVIDIA TransformerEngine Ops Fused Backward Add
RMSNorm", Description and I/O Contract: grad_input = norm backward +
residual gradient, plus grad_weight).

Shapes: x is [..., hidden], contiguous, on a CUDA device; gamma (and beta)
[hidden].  The outputs have x's dtype; weight gradients have the weights'
dtype.  Every step runs in the library's kernels; this module only reshapes
and marshals.
"""
from __future__ import annotations

import torch

from . import ops

__all__ = ["layer_norm", "rms_norm", "layer_norm_with_residual", "rms_norm_with_residual"]


def _rows(x: torch.Tensor, hidden: int) -> torch.Tensor:
    if x.shape[-1] != hidden:
        raise ValueError(f"last dimension {x.shape[-1]} != hidden {hidden}")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    return x.view(-1, hidden)


class _Norm(torch.autograd.Function):
    """Outputs (y, residual); residual is x passed through (or None)."""

    @staticmethod
    def forward(ctx, x, gamma, beta, norm, eps, zero_centered_gamma, sm_margin, residual):
        hidden = gamma.shape[0]
        x2 = _rows(x, hidden)
        o = ops.norm_fwd(x2, gamma, beta, norm=norm, eps=eps,
                         zero_centered_gamma=zero_centered_gamma, sm_margin=sm_margin,
                         training=True)
        ctx.save_for_backward(x2, gamma, o["mu"], o["rsigma"])
        ctx.norm, ctx.zcg, ctx.sm_margin = norm, zero_centered_gamma, sm_margin
        ctx.shape, ctx.has_beta = x.shape, beta is not None
        y = o["out"].view(x.shape)
        if not residual:
            return y, None
        # A new tensor object sharing x's storage: the extra output.
        return y, x.view(x.shape)

    @staticmethod
    def backward(ctx, dy, dres):
        x2, gamma, mu, rsigma = ctx.saved_tensors
        hidden = gamma.shape[0]
        if dy is None:
            dy = torch.zeros(ctx.shape, dtype=x2.dtype, device=x2.device)
        dz = dy.contiguous().view(-1, hidden)
        dr = None if dres is None else dres.contiguous().view(-1, hidden)
        dx, dg, db = ops.norm_bwd(dz, x2, mu, rsigma, gamma, dr, norm=ctx.norm,
                                  zero_centered_gamma=ctx.zcg, sm_margin=ctx.sm_margin)
        return (dx.view(ctx.shape), dg, db if ctx.has_beta else None,
                None, None, None, None, None)


def layer_norm(x, gamma, beta, eps=1e-5, zero_centered_gamma=False, sm_margin=0):
    """LayerNorm over the last dimension: (x - mu) * rsigma * g' + beta."""
    return _Norm.apply(x, gamma, beta, "layernorm", eps, zero_centered_gamma, sm_margin,
                       False)[0]


def rms_norm(x, gamma, eps=1e-6, zero_centered_gamma=False, sm_margin=0):
    """RMSNorm over the last dimension: x * rsigma * g'."""
    return _Norm.apply(x, gamma, None, "rmsnorm", eps, zero_centered_gamma, sm_margin, False)[0]


def layer_norm_with_residual(x, gamma, beta, eps=1e-5, zero_centered_gamma=False, sm_margin=0):
    """(layer_norm(x), x); the backward adds the second output's gradient to
    dx inside the norm's backward kernel."""
    return _Norm.apply(x, gamma, beta, "layernorm", eps, zero_centered_gamma, sm_margin, True)


def rms_norm_with_residual(x, gamma, eps=1e-6, zero_centered_gamma=False, sm_margin=0):
    """(rms_norm(x), x); the backward adds the second output's gradient to dx
    inside the norm's backward kernel (the fused backward-add)."""
    return _Norm.apply(x, gamma, None, "rmsnorm", eps, zero_centered_gamma, sm_margin, True)
