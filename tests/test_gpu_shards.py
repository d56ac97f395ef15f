"""Row sharding on one GPU: the batch split into row shards, each shard run
by its own call (as one rank of a data-parallel job would), then combined
the way ranks combine them -- updated_amax by MAX, fp32 dgamma/dbeta by SUM --
against the unsharded call.  Row-local outputs must be bit-identical; the
combined amax bit-exact; the summed weight gradients within fp32 reordering.
"""
import dataclasses

import pytest
import torch

from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SHARDS = [0, 64, 96, 192, 256]  # 32-row aligned boundaries (MXFP8 / colwise need them)


def _fwd(ops, w, inp, rows):
    c = lambda t: None if t is None else t.cuda()
    x = inp["x"].cuda()[rows]
    return ops.norm_fwd(x, c(inp["gamma"]), c(inp["beta"]), norm=w.norm, eps=w.eps,
                        zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                        layout=w.layout, scale=c(inp["scale"]), amax=c(inp["amax"]))


@pytest.mark.parametrize("name,hidden", [
    ("rms_bf16_e4m3_delayed_32768x8192", 8192),
    ("rms_bf16_mxfp8_16384x5120", 5120),
    ("ln_bf16_16384x4096", 4096),
])
def test_forward_shards_combine_to_unsharded(gpu, name, hidden):
    w = WORKLOADS[name].with_shape(SHARDS[-1], hidden)
    inp = make_inputs(w)
    full = _fwd(gpu, w, inp, slice(None))
    amax = None
    for a, b in zip(SHARDS[:-1], SHARDS[1:]):
        part = _fwd(gpu, w, inp, slice(a, b))
        for k, v in part.items():
            if v is None or k in ("updated_amax", "scale_inv", "colwise_scale_inv",
                                  "colwise_out"):
                continue
            assert torch.equal(v, full[k][a:b]), k
        if w.scaling == "delayed":
            assert torch.equal(part["colwise_out"], full["colwise_out"][:, a:b])
            assert torch.equal(part["scale_inv"], full["scale_inv"])
            m = part["updated_amax"]
            amax = m if amax is None else torch.maximum(amax, m)
        elif w.scaling == "mxfp8":
            assert torch.equal(part["colwise_out"], full["colwise_out"][a:b])
            assert torch.equal(part["scale_inv"], full["scale_inv"][a:b])
            assert torch.equal(part["colwise_scale_inv"], full["colwise_scale_inv"][a // 32:b // 32])
    if w.scaling == "delayed":
        assert torch.equal(amax, full["updated_amax"])


@pytest.mark.parametrize("name,hidden,add", [
    ("ln_bf16_16384x4096", 4096, False),
    ("rms_bwd_add_bf16_32768x12288", 12288, True),
])
def test_backward_shards_sum_to_unsharded(gpu, name, hidden, add):
    # fp32 weights, so that dgamma/dbeta come back in fp32 and can be summed
    w = dataclasses.replace(WORKLOADS[name].with_shape(SHARDS[-1], hidden), w_dtype="f32")
    inp = make_inputs(w)
    ln = w.norm == "layernorm"
    g = torch.Generator().manual_seed(5)
    rs = (torch.rand(w.rows, generator=g) + 0.5).cuda()
    mu = (torch.randn(w.rows, generator=g) * 0.1).cuda() if ln else None
    dz, x, gam = inp["dz"].cuda(), inp["x"].cuda(), inp["gamma"].cuda()
    dres = inp["dresidual"].cuda() if add else None

    def run(rows):
        return gpu.norm_bwd(dz[rows], x[rows], mu[rows] if ln else None, rs[rows], gam,
                            dres[rows] if add else None, norm=w.norm,
                            zero_centered_gamma=w.zero_centered_gamma)

    dx, dg, db = run(slice(None))
    sg = torch.zeros_like(dg)
    sb = torch.zeros_like(dg)
    for a, b in zip(SHARDS[:-1], SHARDS[1:]):
        pdx, pdg, pdb = run(slice(a, b))
        assert torch.equal(pdx, dx[a:b])
        sg += pdg
        if ln:
            sb += pdb
    # fp32 sums in another order: within 1e-4 of the sum of |terms|
    xhat = ((x.float() - mu[:, None]) if ln else x.float()) * rs[:, None]
    tg = (dz.float() * xhat).abs().sum(0) + 1e-30
    assert ((sg - dg).abs() <= 1e-4 * tg).all()
    if ln:
        tb = dz.float().abs().sum(0) + 1e-30
        assert ((sb - db).abs() <= 1e-4 * tb).all()
