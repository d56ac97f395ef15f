"""Delayed-scaling amax, bit for bit.

The updated amax is max|z| over the whole tensor, where z is the kernel's own
fp32 value before the scale is applied ("Implementation:NVIDIA
TransformerEngine JAX XLA Normalization", Description: scale / amax /
scale_inv; I/O Contract: updated_amax_buf).  With fp32 inputs the same kernel
also writes z unquantized (an fp32 output): the delayed run's amax must be
the exact maximum of that run's |out|, on the ring, long-row cluster and
generic paths.  The same outputs also pin ``kernel_z32`` -- the fp32
recomputation of z from the kernel's saved statistics that the other tests
use for the paths and dtypes without an fp32 output (bf16 inputs, the stripe
kernel of the columnwise layouts) -- to the kernel's z, element by element.
"""
import dataclasses

import numpy as np
import pytest
import torch

from parity import amax_f32, kernel_z32, same_f32_bits
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
from test_gpu_parity import check_amax_bits

pytestmark = pytest.mark.gpu

DEL = "rms_bf16_e4m3_delayed_32768x8192"


def wl(**kw):
    base = dict(in_dtype="f32", w_dtype="f32", layout="rowwise")
    base.update(kw)
    return dataclasses.replace(WORKLOADS[DEL], **base)


CASES = [
    ("ring rms", wl(rows=64, hidden=1024)),
    ("ring layernorm ragged", wl(rows=67, hidden=4000, norm="layernorm", beta_std=0.1)),
    ("ring layernorm zcg", wl(rows=33, hidden=2048, norm="layernorm", beta_std=0.1,
                              zero_centered_gamma=True, gamma_mean=0.0, gamma_std=0.05)),
    ("ring rms saturating", wl(rows=40, hidden=8192, amax_prev=4.0)),
    ("cluster rms", wl(rows=20, hidden=12288)),
    ("cluster layernorm", wl(rows=9, hidden=24576, norm="layernorm", beta_std=0.1)),
    ("generic rms", wl(rows=17, hidden=1001)),
    ("generic layernorm", wl(rows=5, hidden=70001, norm="layernorm", beta_std=0.1)),
    # columnwise layouts of rows too long for a stripe (the long-row kernel
    # reduces the amax, the columnwise tile kernel writes the columns)
    ("cluster + columnwise tiles, colwise", wl(rows=32, hidden=20480, layout="colwise")),
    ("cluster + columnwise tiles, layernorm row+col",
     wl(rows=64, hidden=20480, layout="rowwise_colwise", norm="layernorm", beta_std=0.1)),
]


@pytest.mark.parametrize("label,w", CASES, ids=[c[0] for c in CASES])
def test_amax_is_max_of_the_fp32_output_run(gpu, label, w):
    inp = make_inputs(w, seed=4)
    c = lambda t: None if t is None else t.cuda()
    common = dict(norm=w.norm, eps=w.eps, zero_centered_gamma=w.zero_centered_gamma)
    q = gpu.norm_fwd(c(inp["x"]), c(inp["gamma"]), c(inp["beta"]), scaling="delayed",
                     layout=w.layout, scale=c(inp["scale"]), amax=c(inp["amax"]), **common)
    f = gpu.norm_fwd(c(inp["x"]), c(inp["gamma"]), c(inp["beta"]), **common)
    torch.cuda.synchronize()
    # the same kernel template: identical statistics
    assert torch.equal(q["rsigma"], f["rsigma"])
    if w.norm == "layernorm":
        assert torch.equal(q["mu"], f["mu"])
    z = f["out"].cpu().numpy()
    assert same_f32_bits(q["updated_amax"].item(), amax_f32(z))
    # kernel_z32 reproduces the kernel's z exactly
    z32 = kernel_z32(inp["x"], inp["gamma"], inp["beta"],
                     f["mu"].cpu().numpy() if w.norm == "layernorm" else None,
                     f["rsigma"].cpu().numpy(), 0 if w.norm == "layernorm" else 1,
                     w.zero_centered_gamma)
    diff = np.argwhere(z32.view(np.uint32) != z.view(np.uint32))
    assert diff.size == 0, f"{len(diff)} elements differ, e.g. {diff[:4].tolist()}"


def test_amax_bits_after_other_calls_and_with_nan(gpu):
    """updated_amax is zeroed on the stream by every call: a call after one
    with a larger (or NaN) amax reports its own maximum, bit for bit."""
    base = dataclasses.replace(WORKLOADS[DEL], rows=96, hidden=8192)
    o = gpu.fwd_outputs(96, 8192, torch.bfloat16, "rmsnorm", "delayed", "rowwise_colwise")
    c = lambda t: None if t is None else t.cuda()
    for gain, nan in ((1000.0, False), (20.0, True), (20.0, False)):
        w = dataclasses.replace(base, outlier_gain=gain)
        inp = dict(make_inputs(w, seed=1))
        if nan:
            x = inp["x"].clone()
            x[5, 77] = float("nan")
            inp["x"] = x
        out = gpu.norm_fwd(c(inp["x"]), c(inp["gamma"]), None, norm="rmsnorm", eps=w.eps,
                           scaling="delayed", layout="rowwise_colwise", scale=c(inp["scale"]),
                           amax=c(inp["amax"]), outputs=o)
        torch.cuda.synchronize()
        check_amax_bits(out, inp, w)
        assert np.isnan(out["updated_amax"].item()) == nan
