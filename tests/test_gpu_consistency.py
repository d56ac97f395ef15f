"""Self-consistency of the CUDA path: determinism, SM margin, misaligned
pointers (scalar path), empty inputs, CUDA-graph capture, and guard bands
around every output (a bounds check without a sanitizer)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import bwd_terms, check_float, check_wgrad, z_terms
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
from test_gpu_parity import run_bwd_and_check, run_fwd_and_check

pytestmark = pytest.mark.gpu


def wl(name, **kw):
    return dataclasses.replace(WORKLOADS[name], **kw)


def _fwd(ops, w, inp, **kw):
    c = lambda t: None if t is None else t.cuda()
    return ops.norm_fwd(c(inp["x"]), c(inp["gamma"]), c(inp["beta"]), norm=w.norm, eps=w.eps,
                        zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                        layout=w.layout, scale=c(inp["scale"]), amax=c(inp["amax"]), **kw)


@pytest.mark.parametrize("name,kw", [
    ("ln_bf16_16384x4096", dict(rows=300, hidden=4096)),
    ("rms_bf16_e4m3_delayed_32768x8192", dict(rows=128, hidden=8192)),
    ("rms_bf16_mxfp8_16384x5120", dict(rows=128, hidden=5120)),
])
def test_fwd_is_deterministic(gpu, name, kw):
    w = wl(name, **kw)
    inp = make_inputs(w)
    a = _fwd(gpu, w, inp)
    b = _fwd(gpu, w, inp)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_bwd_is_deterministic(gpu):
    w = wl("rms_bwd_add_bf16_32768x12288", rows=500, hidden=12288)
    inp = make_inputs(w)
    rs = torch.rand(w.rows) + 0.5
    c = lambda t: t.cuda()
    r1 = gpu.norm_bwd(c(inp["dz"]), c(inp["x"]), None, c(rs), c(inp["gamma"]),
                      c(inp["dresidual"]), norm="rmsnorm")
    r2 = gpu.norm_bwd(c(inp["dz"]), c(inp["x"]), None, c(rs), c(inp["gamma"]),
                      c(inp["dresidual"]), norm="rmsnorm")
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])


@pytest.mark.parametrize("margin", [1, 100, 10000])
def test_sm_margin(gpu, margin):
    run_fwd_and_check(gpu, wl("ln_bf16_16384x4096", rows=200, hidden=4096), sm_margin=margin)
    run_fwd_and_check(gpu, wl("rms_bf16_mxfp8_16384x5120", rows=96, hidden=5120),
                      sm_margin=margin)
    run_bwd_and_check(gpu, wl("ln_bf16_16384x4096", rows=200, hidden=4096), sm_margin=margin)


def test_misaligned_pointers_take_the_scalar_path(gpu):
    w = wl("ln_bf16_16384x4096", rows=40, hidden=256)
    inp = make_inputs(w)
    # Offset every device buffer by one element so that nothing is 16-byte aligned.
    def shifted(t):
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = flat[1:].view(t.shape)
        v.copy_(t)
        return v
    x, gamma, beta = shifted(inp["x"]), shifted(inp["gamma"]), shifted(inp["beta"])
    assert x.data_ptr() % 16 != 0
    o = gpu.fwd_outputs(w.rows, w.hidden, torch.bfloat16, "layernorm")
    o["out"] = shifted(torch.zeros(w.rows, w.hidden, dtype=torch.bfloat16))
    out = gpu.norm_fwd(x, gamma, beta, norm="layernorm", eps=w.eps, outputs=o)
    torch.cuda.synchronize()
    z, mu, rs = oracle.norm_fwd(inp["x"], inp["gamma"], inp["beta"], 0, False, w.eps)
    check_float("out", out["out"], z, torch.bfloat16,
                terms=z_terms(inp["x"], inp["gamma"], inp["beta"], mu, rs, 0, False))
    dz = shifted(inp["dz"])
    dx, dg, db = gpu.norm_bwd(dz, x, out["mu"], out["rsigma"], gamma, None, norm="layernorm")
    torch.cuda.synchronize()
    rdx, rdg, _ = oracle.norm_bwd(inp["dz"], inp["x"], out["mu"].cpu(), out["rsigma"].cpu(),
                                  inp["gamma"], None, 0, False)
    t_dx, t_dg, _ = bwd_terms(inp["dz"], inp["x"], out["mu"].cpu().numpy(),
                              out["rsigma"].cpu().numpy(), inp["gamma"], None, 0, False)
    check_float("dx", dx, rdx, torch.bfloat16, terms=t_dx)
    check_wgrad("dgamma", dg, rdg, torch.float32, t_dg)


def test_empty_rows(gpu):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    scale = torch.tensor([2.0], device="cuda")
    out = gpu.norm_fwd(x, gamma, None, norm="rmsnorm", scaling="delayed",
                       layout="rowwise_colwise", scale=scale)
    torch.cuda.synchronize()
    assert out["updated_amax"].item() == 0.0 and out["scale_inv"].item() == 0.5
    dx, dg, _ = gpu.norm_bwd(x, x, None, torch.empty(0, device="cuda"), gamma, None,
                             norm="rmsnorm")
    torch.cuda.synchronize()
    assert dx.numel() == 0 and torch.all(dg == 0)


def test_updated_amax_is_overwritten_not_merged(gpu):
    w = wl("rms_bf16_e4m3_delayed_32768x8192", rows=64, hidden=1024)
    inp = make_inputs(w)
    o = gpu.fwd_outputs(w.rows, w.hidden, torch.bfloat16, "rmsnorm", "delayed", w.layout)
    o["updated_amax"].fill_(1e30)
    out = _fwd(gpu, w, inp, outputs=o)
    torch.cuda.synchronize()
    z, _, _ = oracle.norm_fwd(inp["x"], inp["gamma"], None, 1, False, w.eps)
    _, amax, _ = oracle.quant_delayed(z, float(inp["scale"][0]))
    check_float("amax", out["updated_amax"], np.array([amax]), torch.float32, rel=1e-5)


@pytest.mark.parametrize("mode", ["current", "object", "handle"])
def test_cuda_graph_capture_matches_eager(gpu, mode):
    """Captured on the stream the binding is given -- the current stream
    (stream=None), a torch stream object, or its raw handle: the outputs are
    zeroed after the capture, so only captured kernels can write them on
    replay."""
    w = wl("ln_bf16_16384x4096", rows=256, hidden=4096)
    inp = make_inputs(w)
    c = lambda t: t.cuda()
    x, gamma, beta, dz = c(inp["x"]), c(inp["gamma"]), c(inp["beta"]), c(inp["dz"])
    o = gpu.fwd_outputs(w.rows, w.hidden, torch.bfloat16, "layernorm")
    ws = gpu.bwd_workspace(w.rows, w.hidden, torch.bfloat16, torch.float32, "layernorm")
    dx = torch.empty_like(x)
    dg = torch.empty_like(gamma)
    db = torch.empty_like(gamma)

    def step():
        cs = torch.cuda.current_stream()
        st = None if mode == "current" else (cs if mode == "object" else cs.cuda_stream)
        gpu.norm_fwd(x, gamma, beta, norm="layernorm", eps=w.eps, outputs=o, stream=st)
        gpu.norm_bwd(dz, x, o["mu"], o["rsigma"], gamma, None, norm="layernorm", workspace=ws,
                     dx=dx, dgamma=dg, dbeta=db, stream=st)

    outs = lambda: (o["out"], o["mu"], o["rsigma"], dx, dg, db)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs()]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for t in outs():
        t.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs()):
        assert torch.equal(a, b)


GUARD = 4096


def _guarded(shape, dtype):
    n = int(np.prod(shape)) if len(shape) else 1
    esz = torch.tensor([], dtype=dtype).element_size()
    g = GUARD // esz
    buf = torch.empty(n + 2 * g, dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(0xA5)
    return buf, buf[g:g + n].view(shape), g


def _guards_intact(buf, g, n):
    b = buf.view(torch.uint8)
    esz = buf.element_size()
    head, tail = b[:g * esz], b[(g + n) * esz:]
    return bool(torch.all(head == 0xA5)) and bool(torch.all(tail == 0xA5))


@pytest.mark.parametrize("name,kw", [
    ("rms_bf16_e4m3_delayed_32768x8192", dict(rows=96, hidden=8192)),
    ("rms_bf16_e4m3_delayed_32768x8192", dict(rows=70, hidden=1000)),
    ("rms_bf16_mxfp8_16384x5120", dict(rows=64, hidden=5120)),
    ("ln_bf16_16384x4096", dict(rows=33, hidden=4000)),
])
def test_guard_bands_untouched(gpu, name, kw):
    w = wl(name, **kw)
    inp = make_inputs(w)
    R, H = w.rows, w.hidden
    o = gpu.fwd_outputs(R, H, torch.bfloat16, w.norm, w.scaling, w.layout)
    guards = {}
    for k, t in o.items():
        if t is not None:
            buf, view, g = _guarded(tuple(t.shape), t.dtype)
            o[k] = view
            guards[k] = (buf, g, view.numel())
    _fwd(gpu, w, inp, outputs=o)
    torch.cuda.synchronize()
    for k, (buf, g, n) in guards.items():
        assert _guards_intact(buf, g, n), k
    if w.norm == "rmsnorm" and w.scaling == "none":
        return
    # backward on the same shape
    mu = o["mu"] if w.norm == "layernorm" else None
    if mu is None and w.norm == "layernorm":
        return
    dxb, dx, g1 = _guarded((R, H), torch.bfloat16)
    gdt = inp["gamma"].dtype
    dgb, dg, g2 = _guarded((H,), gdt)
    dbb, db, g3 = _guarded((H,), gdt)
    c = lambda t: None if t is None else t.cuda()
    gpu.norm_bwd(c(inp["dz"]), c(inp["x"]), mu, o["rsigma"], c(inp["gamma"]), None, norm=w.norm,
                 dx=dx, dgamma=dg, dbeta=db if w.norm == "layernorm" else None)
    torch.cuda.synchronize()
    assert _guards_intact(dxb, g1, R * H) and _guards_intact(dgb, g2, H)
    if w.norm == "layernorm":
        assert _guards_intact(dbb, g3, H)
