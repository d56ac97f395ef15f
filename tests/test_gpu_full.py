"""Parity at the full workload sizes, in the launch configuration the
benchmark times (default stream, sm_margin 0).  Every row is compared: the
oracle runs over the rows in chunks, and each chunk's statistics, outputs,
codes and scales (and, for the backward, dx) are checked against the GPU's;
the delayed-scaling amax and the backward's dgamma / dbeta over all rows.
The counts of elements that pass only through the fp32 evaluation term, of
one-step E4M3 code differences and of E8M0 scales that differ next to a
power of two are reported and bounded over the whole tensor."""
import numpy as np
import pytest
import torch

import oracle
from parity import (Tally, amax_f32, block_amax_colwise, block_amax_rowwise, bwd_terms,
                    check_codes, check_float, check_scales, check_wgrad, kernel_z32, report,
                    same_f32_bits, z_terms)
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CHUNK = 2048
RELIED = "relied-on-fp32-term"


class CodeTally:
    """One-step E4M3 differences summed over chunks; at most 0.1% overall."""

    def __init__(self, name):
        self.name, self.diff, self.total = name, 0.0, 0

    def add(self, frac, n):
        self.diff += frac * n
        self.total += n

    def close(self):
        report("e4m3-codes-one-step-off", self.name, int(round(self.diff)), self.total)
        assert self.diff <= 1e-3 * self.total


def _forward(gpu, w, inp, x):
    c = lambda t: None if t is None else t.cuda()
    out = gpu.norm_fwd(x, c(inp["gamma"]), c(inp["beta"]), norm=w.norm, eps=w.eps,
                       zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                       layout=w.layout, scale=c(inp["scale"]), amax=c(inp["amax"]))
    torch.cuda.synchronize()
    return out


def _check_forward(gpu, w, inp, norm):
    out = _forward(gpu, w, inp, inp["x"].cuda())
    host = {k: v.cpu() for k, v in out.items() if v is not None}
    t_rs = Tally(RELIED, "rsigma", 1e-3)
    t_mu = Tally(RELIED, "mu", 1e-3)
    t_out = Tally(RELIED, "out", 1e-3)
    codes = {k: CodeTally(k) for k in ("out", "colwise_out")}
    near = {k: Tally("e8m0-near-power-of-two", k, 1e-3) for k in ("scale_inv",
                                                                   "colwise_scale_inv")}
    amax = 0.0
    amax32 = np.float32(0.0)
    for i0 in range(0, w.rows, CHUNK):
        sl = slice(i0, min(i0 + CHUNK, w.rows))
        xs = inp["x"][sl]
        z, mu, rs = oracle.norm_fwd(xs, inp["gamma"], inp["beta"], norm, w.zero_centered_gamma,
                                    w.eps)
        check_float("rsigma", host["rsigma"][sl], rs, torch.float32, rel=1e-4, tally=t_rs)
        if norm == 0:
            check_float("mu", host["mu"][sl], mu, torch.float32, rel=1e-4,
                        terms=xs.abs().double().mean(1).numpy(), k=64, tally=t_mu)
        if w.scaling == "none":
            check_float("out", host["out"][sl], z, DT[w.in_dtype], tally=t_out,
                        terms=z_terms(xs, inp["gamma"], inp["beta"], mu, rs, norm,
                                      w.zero_centered_gamma))
        elif w.scaling == "delayed":
            s = float(inp["scale"][0])
            q, a, sinv = oracle.quant_delayed(z, s)
            n = q.size
            codes["out"].add(check_codes("out", host["out"][sl], q, report_it=False), n)
            cw = host["colwise_out"][:, sl].T
            codes["colwise_out"].add(check_codes("colwise_out", cw, q, report_it=False), n)
            assert torch.equal(cw, host["out"][sl]), "colwise is not the transpose"
            assert host["scale_inv"].item() == sinv == host["colwise_scale_inv"].item()
            amax = max(amax, float(a)) if not np.isnan(a) else float("nan")
            z32 = kernel_z32(xs, inp["gamma"], inp["beta"],
                             host["mu"][sl].numpy() if norm == 0 else None,
                             host["rsigma"][sl].numpy(), norm, w.zero_centered_gamma)
            amax32 = np.float32(np.fmax(amax32, amax_f32(z32)))
        else:
            q, s = oracle.mxfp8_rowwise(z)
            got_s = host["scale_inv"].numpy()[sl]
            check_scales("scale_inv", got_s, s, block_amax_rowwise(z), tally=near["scale_inv"])
            codes["out"].add(check_codes("out", host["out"][sl], q, report_it=False,
                                         mask=np.repeat(got_s == s, 32, axis=1)), q.size)
            qc, sc = oracle.mxfp8_colwise(z)
            got_sc = host["colwise_scale_inv"].numpy()[i0 // 32:sl.stop // 32]
            check_scales("colwise_scale_inv", got_sc, sc, block_amax_colwise(z),
                         tally=near["colwise_scale_inv"])
            codes["colwise_out"].add(
                check_codes("colwise_out", host["colwise_out"][sl], qc, report_it=False,
                            mask=np.repeat(got_sc == sc, 32, axis=0)), qc.size)
    t_rs.close()
    if norm == 0:
        t_mu.close()
    if w.scaling == "none":
        t_out.close()
    elif w.scaling == "delayed":
        for t in codes.values():
            t.close()
        got = np.float32(host["updated_amax"].item())
        check_float("amax", host["updated_amax"], np.array([np.float32(amax)]), torch.float32,
                    rel=1e-5)
        assert same_f32_bits(got, amax32), f"amax {got!r} != max|z| of the kernel's z {amax32!r}"
    else:
        for t in list(codes.values()) + list(near.values()):
            t.close()
    return out


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_parity(gpu, name):
    w = WORKLOADS[name]
    norm = 0 if w.norm == "layernorm" else 1
    inp = make_inputs(w, seed=0)
    c = lambda t: None if t is None else t.cuda()
    if "fwd" in w.passes:
        _check_forward(gpu, w, inp, norm)
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
        dx, dg, db = gpu.norm_bwd(c(inp["dz"]), c(inp["x"]), c(mu_t) if norm == 0 else None,
                                  c(rs_t), c(inp["gamma"]), c(inp["dresidual"]), norm=w.norm,
                                  zero_centered_gamma=w.zero_centered_gamma)
        torch.cuda.synchronize()
        dx = dx.cpu()
        t_dx = Tally(RELIED, "dx", 1e-3)
        rdg = np.zeros(w.hidden)
        rdb = np.zeros(w.hidden)
        tdg = np.zeros(w.hidden)
        tdb = np.zeros(w.hidden)
        for i0 in range(0, w.rows, CHUNK):
            sl = slice(i0, min(i0 + CHUNK, w.rows))
            dres = None if inp["dresidual"] is None else inp["dresidual"][sl]
            rdx, g_, b_ = oracle.norm_bwd(inp["dz"][sl], inp["x"][sl],
                                          mu_t[sl] if norm == 0 else None, rs_t[sl],
                                          inp["gamma"], dres, norm, w.zero_centered_gamma)
            rdg += g_
            if norm == 0:
                rdb += b_
            e_dx, t1, t2 = bwd_terms(inp["dz"][sl], inp["x"][sl],
                                     mu32[sl] if norm == 0 else None, rs32[sl], inp["gamma"],
                                     dres, norm, w.zero_centered_gamma)
            check_float("dx", dx[sl], rdx, DT[w.in_dtype], terms=e_dx, tally=t_dx)
            del rdx, e_dx
            tdg += t1
            tdb += t2
        t_dx.close()
        wdt = DT[w.w_dtype]
        check_wgrad("dgamma", dg, rdg, wdt, tdg)
        if norm == 0:
            check_wgrad("dbeta", db, rdb, wdt, tdb)


def test_full_size_delayed_amax_with_nan(gpu):
    """The delayed-scaling workload at full size with NaN in two rows: the
    amax is NaN; every other row's codes (rowwise and transposed) are those
    of the clean run, bit for bit."""
    w = WORKLOADS["rms_bf16_e4m3_delayed_32768x8192"]
    inp = make_inputs(w, seed=0)
    x = inp["x"].cuda()
    clean = _forward(gpu, w, inp, x)
    clean_amax = clean["updated_amax"].item()
    bad_rows = [1234, 30001]
    for r in bad_rows:
        x[r, (31 * r) % w.hidden] = float("nan")
    dirty = _forward(gpu, w, inp, x)
    assert np.isnan(dirty["updated_amax"].item()) and not np.isnan(clean_amax)
    keep = torch.ones(w.rows, dtype=torch.bool, device="cuda")
    keep[bad_rows] = False
    assert torch.equal(dirty["out"][keep], clean["out"][keep])
    assert torch.equal(dirty["colwise_out"][:, keep], clean["colwise_out"][:, keep])
    assert torch.equal(dirty["rsigma"][keep], clean["rsigma"][keep])
    assert torch.isnan(dirty["rsigma"][~keep]).all()
    nan_codes = dirty["out"][~keep].to(torch.int32) & 0x7F
    assert (nan_codes == 0x7F).all()
