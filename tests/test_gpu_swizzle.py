"""MXFP8 scales in the padded, tiled GEMM order (GBN_LAYOUT_SWIZZLED_SCALES):
on every forward path (32-row stripes, the row ring, long rows over a
cluster, their columnwise tile kernel, the generic kernel), the codes are those of the compact call, the
scales are the compact call's scales (checked against the oracle) placed by
the oracle's tiling, and padding bytes are left as they were."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
from test_gpu_parity import run_fwd_and_check

pytestmark = pytest.mark.gpu

MX = "rms_bf16_mxfp8_16384x5120"
SENTINEL = 0xA5


def wl(**kw):
    return dataclasses.replace(WORKLOADS[MX], **kw)


CASES = [
    ("stripe row+col", wl(rows=96, hidden=5120)),
    ("stripe colwise, 160 rows", wl(rows=160, hidden=4096, layout="colwise")),
    ("ring rowwise, ragged rows", wl(rows=130, hidden=8192, layout="rowwise")),
    ("cluster rowwise", wl(rows=33, hidden=49152, layout="rowwise")),
    ("cluster + columnwise tiles, row+col", wl(rows=64, hidden=49152)),
    ("cluster + columnwise tiles, colwise", wl(rows=96, hidden=36896, layout="colwise")),
    ("generic row+col", wl(rows=64, hidden=160, in_dtype="f32", norm="layernorm",
                           w_dtype="f32", beta_std=0.1)),
]


@pytest.mark.parametrize("label,w", CASES, ids=[c[0] for c in CASES])
def test_swizzled_scales(gpu, label, w):
    compact, inp, _ = run_fwd_and_check(gpu, w)   # compact layout, against the oracle
    c = lambda t: None if t is None else t.cuda()
    o = gpu.fwd_outputs(w.rows, w.hidden, inp["x"].dtype, w.norm, w.scaling, w.layout,
                        swizzled_scales=True)
    for k in ("scale_inv", "colwise_scale_inv"):
        if o[k] is not None:
            o[k].fill_(SENTINEL)
    gpu.norm_fwd(c(inp["x"]), c(inp["gamma"]), c(inp["beta"]), norm=w.norm, eps=w.eps,
                 zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling, layout=w.layout,
                 outputs=o, swizzled_scales=True)
    torch.cuda.synchronize()
    for k in ("out", "colwise_out", "rsigma"):
        if compact[k] is not None:
            assert torch.equal(o[k], compact[k]), k
    for k, transpose in (("scale_inv", False), ("colwise_scale_inv", True)):
        if compact[k] is None:
            continue
        s = compact[k].cpu().numpy()
        want, held = oracle.mxfp8_swizzle(s.T if transpose else s)
        got = o[k].cpu().numpy().ravel()
        assert got.size == want.size, k
        assert np.array_equal(got[held], want[held]), k
        assert np.all(got[~held] == SENTINEL), f"{k}: padding written"
