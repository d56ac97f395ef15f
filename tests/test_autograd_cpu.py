"""The autograd layer's plumbing on CPU: the library calls are replaced by
oracle-backed stand-ins (test infrastructure only), so what is checked here
is the wrapper -- reshaping, what it saves, that the residual's gradient goes
into the single backward call as `dresidual`, and that the gradients reach
the right inputs -- against float64 torch autograd of the same formulas.
The kernels themselves are checked through this layer in
test_gpu_autograd.py."""
import numpy as np
import pytest
import torch

import oracle
from rmsnorm_fp8_quantization_gb300 import autograd as A


class FakeOps:
    """norm_fwd / norm_bwd with the library's signatures, computed by the oracle."""

    def __init__(self):
        self.bwd_calls = []

    def norm_fwd(self, x, gamma, beta=None, *, norm, eps, zero_centered_gamma, sm_margin,
                 training):
        n = 0 if norm == "layernorm" else 1
        z, mu, rs = oracle.norm_fwd(x, gamma, beta, n, zero_centered_gamma, eps)
        out = torch.from_numpy(z).to(x.dtype)
        return {"out": out, "mu": torch.from_numpy(mu.astype(np.float32)) if n == 0 else None,
                "rsigma": torch.from_numpy(rs.astype(np.float32))}

    def norm_bwd(self, dz, x, mu, rsigma, gamma, dresidual=None, *, norm, zero_centered_gamma,
                 sm_margin):
        self.bwd_calls.append(dresidual is not None)
        n = 0 if norm == "layernorm" else 1
        dx, dg, db = oracle.norm_bwd(dz, x, mu, rsigma, gamma, dresidual, n, zero_centered_gamma)
        return (torch.from_numpy(dx).to(x.dtype), torch.from_numpy(dg).to(gamma.dtype),
                None if db is None else torch.from_numpy(db).to(gamma.dtype))


@pytest.fixture
def fake(monkeypatch, orc):
    f = FakeOps()
    monkeypatch.setattr(A, "ops", f)
    return f


def _ref_norm(x, g, b, norm, eps, zcg):
    gg = g + 1 if zcg else g
    if norm == "layernorm":
        return torch.nn.functional.layer_norm(x, (x.shape[-1],), gg, b, eps)
    return torch.nn.functional.rms_norm(x, (x.shape[-1],), gg, eps)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("zcg", [False, True])
def test_gradients_match_float64_autograd(fake, norm, residual, zcg):
    g = torch.Generator().manual_seed(1)
    x = torch.randn(2, 3, 16, generator=g)
    gam = torch.randn(16, generator=g) * 0.1 + (0 if zcg else 1)
    bet = torch.randn(16, generator=g) * 0.1 if norm == "layernorm" else None
    wy = torch.randn(2, 3, 16, generator=g)
    wr = torch.randn(2, 3, 16, generator=g)
    eps = 1e-5

    def run(fn, dt):
        xi = x.to(dt).clone().requires_grad_()
        gi = gam.to(dt).clone().requires_grad_()
        bi = None if bet is None else bet.to(dt).clone().requires_grad_()
        y, r = fn(xi, gi, bi)
        loss = (y * wy.to(dt)).sum() + ((r * wr.to(dt)).sum() if r is not None else 0)
        loss.backward()
        out = (y.detach(), xi.grad, gi.grad, None if bi is None else bi.grad)
        return [None if t is None else t.double() for t in out]

    def ours(xi, gi, bi):
        if norm == "layernorm":
            if residual:
                return A.layer_norm_with_residual(xi, gi, bi, eps, zcg)
            return A.layer_norm(xi, gi, bi, eps, zcg), None
        if residual:
            return A.rms_norm_with_residual(xi, gi, eps, zcg)
        return A.rms_norm(xi, gi, eps, zcg), None

    def ref(xi, gi, bi):
        return _ref_norm(xi, gi, bi, norm, eps, zcg), (xi if residual else None)

    # ours: fp32 tensors through the stand-ins (double inside, fp32 saved
    # statistics); reference: float64 end to end from the same fp32 values
    got, want = run(ours, torch.float32), run(ref, torch.float64)
    for a, b in zip(got, want):
        if b is None:
            assert a is None
        else:
            torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-5)
    assert fake.bwd_calls == [residual], "one backward call, fused add iff residual"


def test_residual_output_is_the_input(fake):
    x = torch.randn(4, 8)
    y, r = A.rms_norm_with_residual(x, torch.ones(8))
    assert torch.equal(r, x) and r.data_ptr() == x.data_ptr()


def test_shape_checks(fake):
    with pytest.raises(ValueError):
        A.rms_norm(torch.randn(4, 8), torch.ones(7))
    with pytest.raises(ValueError):
        A.rms_norm(torch.randn(8, 4).t(), torch.ones(8))
