"""Parity at the full workload sizes, in the launch configuration the
benchmark times (default stream, sm_margin 0).  The forward is checked on
sampled 32-row stripes (rows are independent), the delayed-scaling amax and
the backward's dgamma/dbeta over every row, dx on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from parity import (block_amax_colwise, block_amax_rowwise, bwd_terms, check_codes, check_float,
                    check_scales, z_terms)
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CHUNK = 2048


def _sample_rows(rows):
    """Rows of four 32-row stripes: first, two inner, last (all rows if fewer)."""
    if rows <= 128:
        return np.arange(rows)
    ns = rows // 32
    stripes = sorted({0, ns // 3, (2 * ns) // 3, ns - 1})
    return np.concatenate([np.arange(32 * s, 32 * s + 32) for s in stripes])


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_parity(gpu, name):
    w = WORKLOADS[name]
    norm = 0 if w.norm == "layernorm" else 1
    inp = make_inputs(w, seed=0)
    c = lambda t: None if t is None else t.cuda()
    x = c(inp["x"])
    idx = _sample_rows(w.rows)
    xs = inp["x"][idx]
    if "fwd" in w.passes:
        out = gpu.norm_fwd(x, c(inp["gamma"]), c(inp["beta"]), norm=w.norm, eps=w.eps,
                           zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                           layout=w.layout, scale=c(inp["scale"]), amax=c(inp["amax"]))
        torch.cuda.synchronize()
        z, mu, rs = oracle.norm_fwd(xs, inp["gamma"], inp["beta"], norm, w.zero_centered_gamma,
                                    w.eps)
        check_float("rsigma", out["rsigma"].cpu()[idx], rs, torch.float32, rel=1e-4)
        if norm == 0:
            check_float("mu", out["mu"].cpu()[idx], mu, torch.float32, rel=1e-4,
                        terms=xs.abs().double().mean(1).numpy(), k=64)
        if w.scaling == "none":
            check_float("out", out["out"].cpu()[idx], z, DT[w.in_dtype],
                        terms=z_terms(xs, inp["gamma"], inp["beta"], mu, rs, norm,
                                      w.zero_centered_gamma))
        elif w.scaling == "delayed":
            s = float(inp["scale"][0])
            q, _, sinv = oracle.quant_delayed(z, s)
            check_codes("out", out["out"].cpu()[idx], q)
            check_codes("colwise_out", out["colwise_out"].cpu()[:, idx].T, q)
            assert torch.equal(out["colwise_out"].cpu()[:, idx].T, out["out"].cpu()[idx])
            assert out["scale_inv"].item() == sinv == out["colwise_scale_inv"].item()
            amax = 0.0
            for i0 in range(0, w.rows, CHUNK):
                zc, _, _ = oracle.norm_fwd(inp["x"][i0:i0 + CHUNK], inp["gamma"], inp["beta"],
                                           norm, w.zero_centered_gamma, w.eps)
                amax = max(amax, float(np.abs(zc).max()))
            check_float("amax", out["updated_amax"].cpu(), np.array([np.float32(amax)]),
                        torch.float32, rel=1e-5)
        else:
            q, s = oracle.mxfp8_rowwise(z)
            got_s = out["scale_inv"].cpu().numpy()[idx]
            check_scales("scale_inv", got_s, s, block_amax_rowwise(z))
            check_codes("out", out["out"].cpu()[idx], q, mask=np.repeat(got_s == s, 32, axis=1))
            qc, sc = oracle.mxfp8_colwise(z)
            stripes = idx[::32] // 32
            got_sc = out["colwise_scale_inv"].cpu().numpy()[stripes]
            check_scales("colwise_scale_inv", got_sc, sc, block_amax_colwise(z))
            check_codes("colwise_out", out["colwise_out"].cpu()[idx], qc,
                        mask=np.repeat(got_sc == sc, 32, axis=0))
    if "bwd" in w.passes:
        # Statistics from the oracle's forward (fp32) feed both backward passes.
        mu32 = np.empty(w.rows, np.float32)
        rs32 = np.empty(w.rows, np.float32)
        for i0 in range(0, w.rows, CHUNK):
            _, m, r = oracle.norm_fwd(inp["x"][i0:i0 + CHUNK], inp["gamma"], inp["beta"], norm,
                                      w.zero_centered_gamma, w.eps)
            mu32[i0:i0 + CHUNK] = m
            rs32[i0:i0 + CHUNK] = r
        mu_t = torch.from_numpy(mu32)
        rs_t = torch.from_numpy(rs32)
        dx, dg, db = gpu.norm_bwd(c(inp["dz"]), x, c(mu_t) if norm == 0 else None, c(rs_t),
                                  c(inp["gamma"]), c(inp["dresidual"]), norm=w.norm,
                                  zero_centered_gamma=w.zero_centered_gamma)
        torch.cuda.synchronize()
        rdg = np.zeros(w.hidden)
        rdb = np.zeros(w.hidden)
        tdg = np.zeros(w.hidden)
        tdb = np.zeros(w.hidden)
        for i0 in range(0, w.rows, CHUNK):
            sl = slice(i0, i0 + CHUNK)
            dres = None if inp["dresidual"] is None else inp["dresidual"][sl]
            _, g_, b_ = oracle.norm_bwd(inp["dz"][sl], inp["x"][sl],
                                        mu_t[sl] if norm == 0 else None, rs_t[sl], inp["gamma"],
                                        dres, norm, w.zero_centered_gamma)
            rdg += g_
            if norm == 0:
                rdb += b_
            _, t1, t2 = bwd_terms(inp["dz"][sl], inp["x"][sl], mu32[sl] if norm == 0 else None,
                                  rs32[sl], inp["gamma"], None, norm, w.zero_centered_gamma)
            tdg += t1
            tdb += t2
        dres_s = None if inp["dresidual"] is None else inp["dresidual"][idx]
        rdx, _, _ = oracle.norm_bwd(inp["dz"][idx], xs, mu_t[idx] if norm == 0 else None,
                                    rs_t[idx], inp["gamma"], dres_s, norm, w.zero_centered_gamma)
        t_dx, _, _ = bwd_terms(inp["dz"][idx], xs, mu32[idx] if norm == 0 else None, rs32[idx],
                               inp["gamma"], dres_s, norm, w.zero_centered_gamma)
        check_float("dx", dx.cpu()[idx], rdx, DT[w.in_dtype], terms=t_dx)
        wdt = DT[w.w_dtype]
        k = 1e-6 / 2.0 ** -24
        check_float("dgamma", dg, rdg, wdt, terms=tdg, k=k,
                    rel=1e-4 if wdt == torch.float32 else None)
        if norm == 0:
            check_float("dbeta", db, rdb, wdt, terms=tdb, k=k,
                        rel=1e-4 if wdt == torch.float32 else None)
