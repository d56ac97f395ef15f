"""Degenerate rows on every kernel path, against the oracle: constant rows
(zero variance -- LayerNorm gives z = beta exactly and rsigma = 1/sqrt(eps)),
all-zero rows (RMSNorm gives z = 0, rsigma = 1/sqrt(eps); MXFP8 blocks of
zeros take scale code 0), and rows with a single non-zero element, mixed
with ordinary rows, through the row ring, the columnwise stripe (delayed and
MXFP8) and the cluster (long-row) kernels, forward and backward."""
import dataclasses

import pytest
import torch

from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
from test_gpu_parity import run_bwd_and_check, run_fwd_and_check

pytestmark = pytest.mark.gpu


def wl(name, **kw):
    return dataclasses.replace(WORKLOADS[name], **kw)


LN2 = "ln_bf16_16384x4096"
DEL = "rms_bf16_e4m3_delayed_32768x8192"
MX = "rms_bf16_mxfp8_16384x5120"

CASES = [
    ("ring layernorm", wl(LN2, rows=64, hidden=4096)),
    ("ring rmsnorm", wl(LN2, rows=64, hidden=4096, norm="rmsnorm")),
    ("stripe delayed rows+cols", wl(DEL, rows=64, hidden=8192)),
    ("stripe mxfp8 rows+cols", wl(MX, rows=64, hidden=5120)),
    ("stripe mxfp8 layernorm", wl(MX, rows=64, hidden=5120, norm="layernorm", w_dtype="f32",
                                  beta_std=0.1, zero_centered_gamma=False, gamma_mean=1.0,
                                  gamma_std=0.1)),
    ("cluster layernorm 32768", wl(LN2, rows=16, hidden=32768)),
]


def degenerate(w):
    """The workload's inputs with rows r % 4 == 0 constant (the row's first
    value), == 1 all zero, == 2 zero but for one element; the rest as drawn."""
    inp = make_inputs(w)
    x = inp["x"].clone()
    for r in range(x.shape[0]):
        kind = r % 4
        if kind == 0:
            x[r] = x[r, 0]
        elif kind == 1:
            x[r] = 0
        elif kind == 2:
            v = x[r, (7 * r) % x.shape[1]].clone()
            x[r] = 0
            x[r, (7 * r) % x.shape[1]] = v
    inp = dict(inp)
    inp["x"] = x
    return inp


@pytest.mark.parametrize("label,w", CASES, ids=[c[0] for c in CASES])
def test_degenerate_rows_forward(gpu, label, w):
    inp = degenerate(w)
    out, _, (z, mu, rs) = run_fwd_and_check(gpu, w, inputs=inp)
    eps = torch.tensor(w.eps, dtype=torch.float64)
    # constant rows of LayerNorm and zero rows of RMSNorm have rsigma = 1/sqrt(eps)
    rows = range(0, w.rows, 4) if w.norm == "layernorm" else range(1, w.rows, 4)
    for r in rows:
        assert abs(float(out["rsigma"][r]) * float(eps.sqrt()) - 1.0) < 1e-6, r
    if w.norm == "layernorm" and w.scaling == "none":
        beta = inp["beta"].to(torch.float64)
        for r in range(0, w.rows, 4):   # z = beta exactly, rounded once
            assert torch.equal(out["out"][r].cpu(), beta.to(out["out"].dtype)), r
            assert float(out["mu"][r]) == float(inp["x"][r, 0]), r


BWD = [c for c in CASES if "bwd" in c[1].passes]


@pytest.mark.parametrize("label,w", BWD, ids=[c[0] for c in BWD])
def test_degenerate_rows_backward(gpu, label, w):
    run_bwd_and_check(gpu, w, inputs=degenerate(w))
