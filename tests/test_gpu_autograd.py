"""The autograd layer on the GPU: its outputs and gradients are the library's
(bit-identical to direct calls of the C ABI, which the parity tests check
against the oracle), they agree with torch's own fp32 autograd of the same
formulas, and the residual variant folds the residual's gradient into the
one backward kernel."""
import dataclasses

import pytest
import torch

from rmsnorm_fp8_quantization_gb300 import autograd as A
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _close(a, b, rel, terms=None):
    """|a - b| <= rel * |b| + 1e-5 * terms: rounding of the stored result plus
    fp32 reordering of sums whose terms have magnitude `terms`."""
    a, b = a.float(), b.float()
    floor = 1e-5 * (terms.float() if terms is not None else 1.0) + 1e-30
    assert ((a - b).abs() <= rel * b.abs() + floor).all(), (a - b).abs().max().item()


def _dx_terms(dy, xhat, rs):
    """Magnitude of the terms of dx = rs * (dy - mean(dy) - xhat * mean(dy * xhat))."""
    return rs * (dy.abs() + dy.mean(-1, keepdim=True).abs()
                 + xhat.abs() * (dy * xhat).mean(-1, keepdim=True).abs())


@pytest.mark.parametrize("zcg", [False, True])
def test_layer_norm_autograd(gpu, zcg):
    w = dataclasses.replace(WORKLOADS["ln_bf16_16384x4096"].with_shape(300, 4096),
                            zero_centered_gamma=zcg)
    inp = make_inputs(w)
    H = w.hidden
    x = inp["x"].cuda().view(3, 100, H).requires_grad_()
    g = inp["gamma"].cuda().requires_grad_()
    b = inp["beta"].cuda().requires_grad_()
    dz = inp["dz"].cuda().view(3, 100, H)
    y = A.layer_norm(x, g, b, w.eps, zcg)
    y.backward(dz)

    o = gpu.norm_fwd(x.detach().view(-1, H), g.detach(), b.detach(), norm="layernorm",
                     eps=w.eps, zero_centered_gamma=zcg)
    assert torch.equal(y.detach().view(-1, H), o["out"])
    dx, dg, db = gpu.norm_bwd(dz.reshape(-1, H), x.detach().view(-1, H), o["mu"], o["rsigma"],
                              g.detach(), None, norm="layernorm", zero_centered_gamma=zcg)
    assert torch.equal(x.grad.view(-1, H), dx)
    assert torch.equal(g.grad, dg) and torch.equal(b.grad, db)

    # torch fp32 autograd of the same formula
    xr = x.detach().float().requires_grad_()
    gr = g.detach().clone().requires_grad_()
    br = b.detach().clone().requires_grad_()
    yr = torch.nn.functional.layer_norm(xr, (H,), gr + 1 if zcg else gr, br, w.eps)
    yr.backward(dz.float())
    rs = o["rsigma"].view(3, 100, 1)
    xhat = (xr.detach() - o["mu"].view(3, 100, 1)) * rs
    dy = dz.float() * (gr.detach() + 1 if zcg else gr.detach())
    _close(y, yr, 2 ** -7, xhat.abs())
    _close(x.grad, xr.grad, 2 ** -7, _dx_terms(dy, xhat, rs))
    _close(g.grad, gr.grad, 1e-4, 10 * (dz.float() * xhat).abs().sum((0, 1)))
    _close(b.grad, br.grad, 1e-4, 10 * dz.float().abs().sum((0, 1)))


def test_rms_norm_with_residual_fuses_the_add(gpu):
    w = WORKLOADS["rms_bwd_add_bf16_32768x12288"].with_shape(200, 12288)
    inp = make_inputs(w)
    H = w.hidden
    x = inp["x"].cuda().view(2, 100, H).requires_grad_()
    g = inp["gamma"].cuda().requires_grad_()
    dz = inp["dz"].cuda().view(2, 100, H)
    dres = inp["dresidual"].cuda().view(2, 100, H)
    y, r = A.rms_norm_with_residual(x, g, w.eps)
    assert r.data_ptr() == x.data_ptr()
    torch.autograd.backward([y, r], [dz, dres])

    o = gpu.norm_fwd(x.detach().view(-1, H), g.detach(), None, norm="rmsnorm", eps=w.eps)
    assert torch.equal(y.detach().view(-1, H), o["out"])
    dx, dg, _ = gpu.norm_bwd(dz.reshape(-1, H), x.detach().view(-1, H), None, o["rsigma"],
                             g.detach(), dres.reshape(-1, H), norm="rmsnorm")
    assert torch.equal(x.grad.view(-1, H), dx)
    assert torch.equal(g.grad, dg)

    xr = x.detach().float().requires_grad_()
    gr = g.detach().float().requires_grad_()
    yr = torch.nn.functional.rms_norm(xr, (H,), gr, w.eps)
    torch.autograd.backward([yr, xr], [dz.float(), dres.float()])
    rs = o["rsigma"].view(2, 100, 1)
    xhat = xr.detach() * rs
    dy = dz.float() * gr.detach()
    _close(y, yr, 2 ** -7, xhat.abs())
    _close(x.grad, xr.grad, 2 ** -7, _dx_terms(dy, xhat, rs) + dres.float().abs())
    _close(g.grad, gr.grad, 2 ** -7, 10 * (dz.float() * xhat).abs().sum((0, 1)))
