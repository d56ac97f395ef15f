"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs, at sizes the oracle finishes quickly (several CTAs, 32-row
stripes and clusters, ragged rows and hidden sizes, scalar fallback)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import (amax_f32, block_amax_colwise, block_amax_rowwise, bwd_terms, check_codes,
                    check_float, check_scales, check_wgrad, kernel_z32, same_f32_bits, z_terms)
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
NORM = {"layernorm": 0, "rmsnorm": 1}


def _cuda(t):
    return None if t is None else t.cuda()


def run_fwd_and_check(ops, w: Workload, seed=0, sm_margin=0, inputs=None):
    inp = inputs if inputs is not None else make_inputs(w, seed)
    norm = NORM[w.norm]
    out = ops.norm_fwd(_cuda(inp["x"]), _cuda(inp["gamma"]), _cuda(inp["beta"]), norm=w.norm,
                       eps=w.eps, zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                       layout=w.layout, scale=_cuda(inp["scale"]), amax=_cuda(inp["amax"]),
                       sm_margin=sm_margin)
    torch.cuda.synchronize()
    z, mu, rs = oracle.norm_fwd(inp["x"], inp["gamma"], inp["beta"], norm, w.zero_centered_gamma,
                                w.eps)
    check_float("rsigma", out["rsigma"], rs, torch.float32, rel=1e-4)
    if norm == 0:
        xabs = inp["x"].abs().double().mean(1).numpy()
        check_float("mu", out["mu"], mu, torch.float32, rel=1e-4, terms=xabs, k=64)
    terms = z_terms(inp["x"], inp["gamma"], inp["beta"], mu, rs, norm, w.zero_centered_gamma)
    rowwise = w.scaling == "none" or w.layout != "colwise"
    colwise = w.scaling != "none" and w.layout != "rowwise"
    if w.scaling == "none":
        check_float("out", out["out"], z, DT[w.in_dtype], terms=terms)
    elif w.scaling == "delayed":
        q, amax, sinv = oracle.quant_delayed(z, float(inp["scale"][0]))
        if rowwise:
            check_codes("out", out["out"], q)
            assert out["scale_inv"].item() == sinv
        if colwise:
            check_codes("colwise_out", out["colwise_out"].T, q)
            assert out["colwise_scale_inv"].item() == sinv
            if rowwise:
                assert torch.equal(out["colwise_out"].T, out["out"]), "colwise is not the transpose"
        check_float("amax", out["updated_amax"], np.array([amax]), torch.float32, rel=1e-5)
        check_amax_bits(out, inp, w)
    else:
        if rowwise:
            q, s = oracle.mxfp8_rowwise(z)
            check_scales("scale_inv", out["scale_inv"], s, block_amax_rowwise(z))
            same = np.repeat(out["scale_inv"].cpu().numpy() == s, 32, axis=1)
            check_codes("out", out["out"], q, mask=same)
        if colwise:
            q, s = oracle.mxfp8_colwise(z)
            check_scales("colwise_scale_inv", out["colwise_scale_inv"], s, block_amax_colwise(z))
            same = np.repeat(out["colwise_scale_inv"].cpu().numpy() == s, 32, axis=0)
            check_codes("colwise_out", out["colwise_out"], q, mask=same)
    return out, inp, (z, mu, rs)


def check_amax_bits(out, inp, w):
    """The updated amax is max|z| of the kernel's own fp32 z, bit for bit:
    z recomputed in fp32 from the statistics the kernel saved, in the
    kernel's order of operations (``kernel_z32``)."""
    norm = NORM[w.norm]
    z32 = kernel_z32(inp["x"], inp["gamma"], inp["beta"],
                     out["mu"].cpu().numpy() if norm == 0 else None, out["rsigma"].cpu().numpy(),
                     norm, w.zero_centered_gamma)
    want = amax_f32(z32)
    got = np.float32(out["updated_amax"].item())
    assert same_f32_bits(got, want), f"amax {got!r} is not max|z| of the kernel's z {want!r}"


def run_bwd_and_check(ops, w: Workload, seed=0, sm_margin=0, inputs=None):
    inp = inputs if inputs is not None else make_inputs(w, seed)
    norm = NORM[w.norm]
    _, mu, rs = oracle.norm_fwd(inp["x"], inp["gamma"], inp["beta"], norm, w.zero_centered_gamma,
                                w.eps)
    mu32 = torch.from_numpy(mu.astype(np.float32))
    rs32 = torch.from_numpy(rs.astype(np.float32))
    dx, dg, db = ops.norm_bwd(_cuda(inp["dz"]), _cuda(inp["x"]), mu32.cuda(), rs32.cuda(),
                              _cuda(inp["gamma"]), _cuda(inp["dresidual"]), norm=w.norm,
                              zero_centered_gamma=w.zero_centered_gamma, sm_margin=sm_margin)
    torch.cuda.synchronize()
    rdx, rdg, rdb = oracle.norm_bwd(inp["dz"], inp["x"], mu32 if norm == 0 else None, rs32,
                                    inp["gamma"], inp["dresidual"], norm, w.zero_centered_gamma)
    t_dx, t_dg, t_db = bwd_terms(inp["dz"], inp["x"], mu32.numpy() if norm == 0 else None,
                                 rs32.numpy(), inp["gamma"], inp["dresidual"], norm,
                                 w.zero_centered_gamma)
    wdt = DT[w.w_dtype]
    check_float("dx", dx, rdx, DT[w.in_dtype], terms=t_dx)
    check_wgrad("dgamma", dg, rdg, wdt, t_dg)
    if norm == 0:
        check_wgrad("dbeta", db, rdb, wdt, t_db)
    return dx, dg, db


def wl(name, **kw):
    return dataclasses.replace(WORKLOADS[name], **kw)


LN2 = "ln_bf16_16384x4096"
RMS1 = "rms_f32_64x1024"
DEL = "rms_bf16_e4m3_delayed_32768x8192"
MX = "rms_bf16_mxfp8_16384x5120"
BADD = "rms_bwd_add_bf16_32768x12288"

FWD_NONE_CASES = [
    wl(RMS1),
    wl(LN2, rows=67, hidden=4096),
    wl(LN2, rows=67, hidden=4000),
    wl(LN2, rows=35, hidden=8192, zero_centered_gamma=True, gamma_mean=0.0, gamma_std=0.05),
    wl(LN2, rows=9, hidden=12288, in_dtype="f16", w_dtype="bf16"),
    wl(LN2, rows=33, hidden=40, in_dtype="f32", w_dtype="f16"),
    wl(LN2, rows=5, hidden=33),                      # hidden not a multiple of 8: scalar path
    wl(LN2, rows=3, hidden=1),
    wl(RMS1, rows=17, hidden=1000, in_dtype="bf16", w_dtype="bf16"),
    wl(RMS1, rows=70, hidden=5120, in_dtype="f16", w_dtype="f32", zero_centered_gamma=True,
       gamma_mean=0.0, gamma_std=0.05),
    wl(RMS1, rows=4, hidden=20000, in_dtype="bf16", w_dtype="bf16"),
    wl(RMS1, rows=2, hidden=70000, in_dtype="bf16", w_dtype="bf16"),  # beyond the vector path
    # the widest ring rows: 6 vectors per thread (up to 384 threads), full and ragged
    wl(LN2, rows=13, hidden=18432),
    wl(RMS1, rows=11, hidden=17000, in_dtype="bf16", w_dtype="bf16"),
    wl(RMS1, rows=9, hidden=9000),
]


@pytest.mark.parametrize("w", FWD_NONE_CASES, ids=lambda w: f"{w.norm}-{w.in_dtype}-{w.w_dtype}-"
                         f"{w.rows}x{w.hidden}-zcg{int(w.zero_centered_gamma)}")
def test_fwd_unquantized(gpu, w):
    run_fwd_and_check(gpu, w)


FWD_DELAYED_CASES = [
    wl(DEL, rows=96, hidden=8192),
    wl(DEL, rows=96, hidden=2048, layout="rowwise"),
    wl(DEL, rows=64, hidden=1024, layout="colwise"),
    wl(DEL, rows=70, hidden=1000),                          # ragged stripe: generic kernel
    wl(DEL, rows=64, hidden=5120, norm="layernorm", w_dtype="f32", beta_std=0.1),
    wl(DEL, rows=32, hidden=24, in_dtype="f32", w_dtype="f32"),
    wl(DEL, rows=40, hidden=36, in_dtype="f16"),            # hidden % 8 != 0: generic
    wl(DEL, rows=64, hidden=12288, amax_prev=4.0),          # heavy saturation
    # LayerNorm in every layout
    wl(DEL, rows=96, hidden=4096, norm="layernorm", w_dtype="f32", beta_std=0.1,
       layout="colwise"),
    wl(DEL, rows=67, hidden=4000, norm="layernorm", w_dtype="f32", beta_std=0.1,
       layout="rowwise"),
    wl(DEL, rows=64, hidden=8192, norm="layernorm", w_dtype="bf16", beta_std=0.1,
       zero_centered_gamma=True, gamma_mean=0.0, gamma_std=0.05),
    # rows a multiple of 16 but not of 32: the generic kernel for the transposed copy
    wl(DEL, rows=48, hidden=8192),
    wl(DEL, rows=80, hidden=2048, layout="colwise"),
    wl(DEL, rows=112, hidden=4096, norm="layernorm", w_dtype="f32", beta_std=0.1),
    # wide rows: clusters above 8 CTAs (non-portable sizes, up to 16)
    wl(DEL, rows=64, hidden=16384),
    wl(DEL, rows=64, hidden=8192, in_dtype="f32", w_dtype="f32"),
    # rowwise ring with 6 vectors per thread
    wl(DEL, rows=33, hidden=18432, layout="rowwise"),
]


@pytest.mark.parametrize("w", FWD_DELAYED_CASES, ids=lambda w: f"{w.norm}-{w.in_dtype}-{w.layout}-"
                         f"{w.rows}x{w.hidden}-a{w.amax_prev}")
def test_fwd_delayed_fp8(gpu, w):
    run_fwd_and_check(gpu, w)


FWD_MX_CASES = [
    wl(MX, rows=96, hidden=5120),
    wl(MX, rows=64, hidden=8192, layout="rowwise"),
    wl(MX, rows=64, hidden=4096, layout="colwise"),
    wl(MX, rows=32, hidden=32),
    wl(MX, rows=96, hidden=160, norm="layernorm", w_dtype="f32", beta_std=0.1, in_dtype="f32"),
    wl(MX, rows=64, hidden=2048, in_dtype="f16", zero_centered_gamma=False, gamma_mean=1.0,
       gamma_std=0.1),
    wl(MX, rows=40, hidden=96, layout="rowwise"),           # rowwise allows ragged rows
    # LayerNorm in every layout
    wl(MX, rows=96, hidden=5120, norm="layernorm", w_dtype="f32", beta_std=0.1,
       zero_centered_gamma=False, gamma_mean=1.0, gamma_std=0.1),
    wl(MX, rows=64, hidden=8192, norm="layernorm", w_dtype="bf16", beta_std=0.1),
    wl(MX, rows=64, hidden=2048, norm="layernorm", w_dtype="f32", beta_std=0.1,
       layout="colwise"),
    wl(MX, rows=77, hidden=4096, norm="layernorm", w_dtype="f32", beta_std=0.1,
       layout="rowwise", in_dtype="f16"),
    # wide rows: clusters above 8 CTAs (non-portable sizes, up to 16)
    wl(MX, rows=64, hidden=16384),
    wl(MX, rows=64, hidden=8192, in_dtype="f32", w_dtype="f32"),
    # rowwise ring with 6 vectors per thread, ragged
    wl(MX, rows=40, hidden=17408, layout="rowwise"),
]


@pytest.mark.parametrize("w", FWD_MX_CASES, ids=lambda w: f"{w.norm}-{w.in_dtype}-{w.layout}-"
                         f"{w.rows}x{w.hidden}")
def test_fwd_mxfp8(gpu, w):
    run_fwd_and_check(gpu, w)


BWD_CASES = [
    wl(RMS1),
    wl(LN2, rows=67, hidden=4096),
    wl(LN2, rows=67, hidden=4000),
    wl(BADD, rows=37, hidden=12288),
    wl(BADD, rows=37, hidden=12288, norm="layernorm", beta_std=0.1),
    wl(BADD, rows=50, hidden=1024, dresidual=False, zero_centered_gamma=True, gamma_mean=0.0,
       gamma_std=0.05),
    wl(LN2, rows=21, hidden=2048, in_dtype="f16", w_dtype="f16", dresidual=True),
    wl(LN2, rows=19, hidden=33, dresidual=True),                  # scalar path
    wl(RMS1, rows=600, hidden=256, in_dtype="bf16", w_dtype="f32"),  # many rows per CTA
    wl(RMS1, rows=3, hidden=40000, in_dtype="bf16", w_dtype="bf16"),  # beyond the vector path
    wl(RMS1, rows=1, hidden=64),
    # rows that would need 8 vectors per thread in the ring: split over a
    # cluster when one fits, full and ragged ...
    wl(LN2, rows=29, hidden=16384),
    wl(BADD, rows=23, hidden=14000),
    wl(RMS1, rows=17, hidden=8192),
    wl(RMS1, rows=13, hidden=7000, norm="layernorm", beta_std=0.1),
    # ... and in the ring with 8 vectors per thread when none does
    wl(LN2, rows=7, hidden=12296),
    wl(BADD, rows=5, hidden=12296),
    wl(RMS1, rows=5, hidden=7004),
    # LayerNorm rows at 3 vectors per thread: over a cluster, or in the ring
    # when no split fits
    wl(LN2, rows=23, hidden=10240),
    wl(LN2, rows=9, hidden=8216, dresidual=True),
]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: f"{w.norm}-{w.in_dtype}-{w.w_dtype}-"
                         f"{w.rows}x{w.hidden}-add{int(w.dresidual)}-zcg{int(w.zero_centered_gamma)}")
def test_bwd(gpu, w):
    run_bwd_and_check(gpu, w)


# ---------------------------------------------------------------- exact-value sweeps

def _unit_rows(rows, hidden, g):
    """Rows of +-1 with equal counts: with eps = 0 the RMSNorm statistics are
    exactly 1, so z = +-gamma exactly on both sides."""
    s = torch.stack([torch.randperm(hidden, generator=g) % 2 for _ in range(rows)]).float()
    return s * 2 - 1


@pytest.mark.parametrize("layout", ["rowwise", "rowwise_colwise"])
def test_e4m3_hardware_conversion_matches_oracle_bit_exact(gpu, layout):
    g = torch.Generator().manual_seed(7)
    codes = torch.arange(0, 0x7F, dtype=torch.float64)
    vals = torch.tensor([oracle.e4m3_decode(int(c)) for c in codes.tolist()], dtype=torch.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    f32 = lambda t: t.to(torch.float32)
    sweep = torch.cat([
        f32(vals), f32(mids),
        f32(mids).view(torch.int32).add(1).view(torch.float32),   # one fp32 ulp above each tie
        f32(mids).view(torch.int32).sub(1).view(torch.float32),   # and below
        torch.tensor([449.0, 463.99, 464.0, 480.0, 1e6, 3e38, 2.0 ** -10, 1.5 * 2.0 ** -10, 1e-30]),
        torch.randn(2000, generator=g) * 50, torch.randn(1000, generator=g) * 0.02,
    ])
    H = ((sweep.numel() + 7) // 8) * 8
    gamma = torch.zeros(H)
    gamma[:sweep.numel()] = sweep
    x = _unit_rows(32, H, g)
    scale = torch.tensor([1.0])
    out = gpu.norm_fwd(x.cuda(), gamma.cuda(), None, norm="rmsnorm", eps=0.0, scaling="delayed",
                       layout=layout, scale=scale.cuda(), amax=scale.cuda())
    torch.cuda.synchronize()
    assert torch.all(out["rsigma"] == 1.0)
    z, _, rs = oracle.norm_fwd(x, gamma, None, 1, False, 0.0)   # exactly +-gamma (and +0)
    assert np.all(rs == 1.0)
    q, amax, _ = oracle.quant_delayed(z, 1.0)
    got = out["out"].cpu().numpy()
    bad = np.argwhere(got != q)
    detail = [(float(z[i, j]), hex(got[i, j]), hex(q[i, j])) for i, j in bad[:12]]
    assert bad.size == 0, f"{len(bad)} codes differ: (value, gpu, oracle) {detail}"
    if layout == "rowwise_colwise":
        assert np.array_equal(out["colwise_out"].T.cpu().numpy(), q)
    assert out["updated_amax"].item() == amax


def test_e8m0_block_scales_bit_exact_on_crafted_blocks(gpu):
    g = torch.Generator().manual_seed(8)
    amaxes = [448.0, 511.9, 512.0, 1.0, 0.99999994, 2.0 ** -110, 2.0 ** -118, 2.0 ** -119,
              2.0 ** -126, 0.0, 3.0e38, 1.5, 3.0, 100.0, 2.0 ** 20, 1e-20]
    H = 32 * len(amaxes)
    gamma = torch.zeros(H)
    for b, a in enumerate(amaxes):
        blk = torch.rand(32, generator=g) * a
        blk[int(torch.randint(0, 32, (1,), generator=g))] = a
        gamma[32 * b:32 * (b + 1)] = blk.to(torch.float32)
    x = _unit_rows(32, H, g)
    out = gpu.norm_fwd(x.cuda(), gamma.cuda(), None, norm="rmsnorm", eps=0.0, scaling="mxfp8",
                       layout="rowwise_colwise")
    torch.cuda.synchronize()
    z, _, _ = oracle.norm_fwd(x, gamma, None, 1, False, 0.0)
    q, s = oracle.mxfp8_rowwise(z)
    assert np.array_equal(out["scale_inv"].cpu().numpy(), s)
    assert np.array_equal(out["out"].cpu().numpy(), q)
    qc, sc = oracle.mxfp8_colwise(z)
    assert np.array_equal(out["colwise_scale_inv"].cpu().numpy(), sc)
    assert np.array_equal(out["colwise_out"].cpu().numpy(), qc)
    expect = [oracle.e8m0_code(float(np.float32(a))) for a in amaxes]
    assert list(out["scale_inv"][0].cpu().numpy()) == expect
