"""NaN inputs on every kernel path, against the oracle: a NaN anywhere in a
row makes that row's statistics and outputs NaN (unquantized NaN, E4M3 code
NaN); the delayed-scaling amax propagates it; an MXFP8 block holding it gets
the NaN scale code 255, rowwise and columnwise; the backward's dx row and
every dgamma column it touches are NaN, dbeta stays finite.  The other rows
are unaffected."""
import dataclasses
import math

import numpy as np
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
NAN_ROWS = (3, 17)

CASES = [
    ("ring layernorm", wl(LN2, rows=64, hidden=4096)),
    ("ring delayed rowwise", wl(DEL, rows=40, hidden=8192, layout="rowwise")),
    ("stripe delayed rows+cols", wl(DEL, rows=64, hidden=8192)),
    ("stripe mxfp8 rows+cols", wl(MX, rows=64, hidden=5120)),
    ("cluster layernorm 32768", wl(LN2, rows=24, hidden=32768)),
]


def with_nans(w):
    inp = dict(make_inputs(w))
    x = inp["x"].clone()
    for r in NAN_ROWS:
        x[r, (37 * r) % w.hidden] = float("nan")
    inp["x"] = x
    return inp


@pytest.mark.parametrize("label,w", CASES, ids=[c[0] for c in CASES])
def test_nan_rows_forward(gpu, label, w):
    out, _, _ = run_fwd_and_check(gpu, w, inputs=with_nans(w))
    clean = [r for r in range(w.rows) if r not in NAN_ROWS]
    rs = out["rsigma"].cpu()
    assert all(math.isnan(float(rs[r])) for r in NAN_ROWS)
    assert torch.isfinite(rs[clean]).all()
    if w.scaling == "delayed":
        assert math.isnan(float(out["updated_amax"]))
    if w.scaling == "mxfp8":
        s = out["scale_inv"].cpu().numpy()
        assert (s[list(NAN_ROWS)] == 255).all() and (s[clean] != 255).all()
        sc = out["colwise_scale_inv"].cpu().numpy()
        assert (sc[0] == 255).all()          # rows 0..31 hold both NaN rows
        assert (sc[1] != 255).all()


BWD = [c for c in CASES if "bwd" in c[1].passes]


@pytest.mark.parametrize("label,w", BWD, ids=[c[0] for c in BWD])
def test_nan_rows_backward(gpu, label, w):
    dx, dg, db = run_bwd_and_check(gpu, w, inputs=with_nans(w))
    dx = dx.cpu().float()
    clean = [r for r in range(w.rows) if r not in NAN_ROWS]
    assert torch.isnan(dx[list(NAN_ROWS)]).all() and torch.isfinite(dx[clean]).all()
    assert torch.isnan(dg.cpu()).all()
    assert torch.isfinite(db.cpu()).all()
