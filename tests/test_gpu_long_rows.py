"""Rows longer than one CTA's ring (over 16384 two-byte or 8192 four-byte
elements): the forward splits each row over a thread-block cluster and
combines the row statistics across it; the backward does the same.  Parity
with the oracle, as for the short rows, including slices with a ragged tail
and every rowwise output kind."""
import dataclasses

import pytest

from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS
from test_gpu_parity import run_bwd_and_check, run_fwd_and_check

pytestmark = pytest.mark.gpu


def wl(name, rows, hidden, **kw):
    return dataclasses.replace(WORKLOADS[name].with_shape(rows, hidden), **kw)


FWD = [
    ("ln 32768", wl("ln_bf16_16384x4096", 37, 32768)),
    ("ln f16 zcg ragged slice 20000", wl("ln_bf16_16384x4096", 19, 20000, in_dtype="f16",
                                          w_dtype="f16", zero_centered_gamma=True)),
    ("rms 65536", wl("rms_bwd_add_bf16_32768x12288", 33, 65536, passes=("fwd",))),
    ("rms f32 12288", wl("rms_f32_64x1024", 20, 12288)),
    ("rms f32 24576 many clusters", wl("rms_f32_64x1024", 301, 24576)),
    ("delayed rowwise 40960", wl("rms_bf16_e4m3_delayed_32768x8192", 40, 40960,
                                 layout="rowwise")),
    ("mxfp8 rowwise 49152", wl("rms_bf16_mxfp8_16384x5120", 32, 49152, layout="rowwise")),
    ("ln mxfp8 rowwise 36864", wl("rms_bf16_mxfp8_16384x5120", 24, 36864, layout="rowwise",
                                  norm="layernorm")),
    # the longest rows the clusters take (8 CTAs x 16384 two-byte / 8192 four-byte elements)
    ("ln 131072 longest cluster row", wl("ln_bf16_16384x4096", 9, 131072)),
    ("rms f32 65536 longest cluster row", wl("rms_f32_64x1024", 7, 65536)),
    # one vector past them: the generic kernel
    ("ln 131080 generic", wl("ln_bf16_16384x4096", 5, 131080)),
    ("delayed rowwise 139264 generic", wl("rms_bf16_e4m3_delayed_32768x8192", 4, 139264,
                                           layout="rowwise")),
    # columnwise layouts of rows too long for a stripe: the long-row kernel,
    # then the columnwise tile kernel from its statistics
    ("delayed both 49152", wl("rms_bf16_e4m3_delayed_32768x8192", 64, 49152)),
    ("delayed colwise ln 40960", wl("rms_bf16_e4m3_delayed_32768x8192", 32, 40960,
                                    layout="colwise", norm="layernorm", w_dtype="f32",
                                    beta_std=0.1)),
    ("delayed both f32 20480", wl("rms_bf16_e4m3_delayed_32768x8192", 32, 20480,
                                  in_dtype="f32", w_dtype="f32")),
    ("mxfp8 both 65536", wl("rms_bf16_mxfp8_16384x5120", 32, 65536)),
    ("mxfp8 colwise ln 36896", wl("rms_bf16_mxfp8_16384x5120", 64, 36896, layout="colwise",
                                  norm="layernorm", w_dtype="f32", beta_std=0.1,
                                  zero_centered_gamma=False, gamma_mean=1.0, gamma_std=0.1)),
]


@pytest.mark.parametrize("label,w", FWD, ids=[f[0] for f in FWD])
def test_long_row_forward(gpu, label, w):
    run_fwd_and_check(gpu, w)


BWD = [
    ("ln 32768", wl("ln_bf16_16384x4096", 37, 32768)),
    ("rms add 65536", wl("rms_bwd_add_bf16_32768x12288", 21, 65536)),
    ("ln add f16 ragged 20000", wl("ln_bf16_16384x4096", 19, 20000, in_dtype="f16",
                                    w_dtype="f16", dresidual=True)),
    ("rms f32 12288", wl("rms_f32_64x1024", 20, 12288)),
    # the longest backward rows the clusters take, and one vector past them (generic kernel)
    ("ln f16 65536 longest cluster row", wl("ln_bf16_16384x4096", 9, 65536, in_dtype="f16",
                                            w_dtype="f16")),
    ("rms add 65544 generic", wl("rms_bwd_add_bf16_32768x12288", 5, 65544)),
    ("ln f32 32772 generic", wl("rms_f32_64x1024", 6, 32772, norm="layernorm")),
]


@pytest.mark.parametrize("label,w", BWD, ids=[b[0] for b in BWD])
def test_long_row_backward(gpu, label, w):
    run_bwd_and_check(gpu, w)


def test_long_row_backward_is_deterministic_and_sm_margin(gpu):
    import torch
    from rmsnorm_fp8_quantization_gb300.workloads import make_inputs
    w = wl("ln_bf16_16384x4096", 150, 32768)
    inp = make_inputs(w)
    c = lambda t: t.cuda()
    rs = torch.rand(w.rows) + 0.5
    mu = torch.randn(w.rows) * 0.1
    runs = []
    for margin in (0, 0, 100):
        runs.append(gpu.norm_bwd(c(inp["dz"]), c(inp["x"]), c(mu), c(rs), c(inp["gamma"]), None,
                                 norm="layernorm", sm_margin=margin))
    a, b, m = runs
    assert all(torch.equal(x, y) for x, y in zip(a, b)), "not deterministic"
    assert torch.equal(a[0], m[0]), "dx depends on the SM margin"
    for x, y in zip(a[1:], m[1:]):    # dgamma/dbeta: other partial rows, same values to fp32
        assert torch.allclose(x, y, rtol=1e-4, atol=1e-4)


def test_long_row_graph_capture_matches_eager(gpu):
    import torch
    from rmsnorm_fp8_quantization_gb300.workloads import make_inputs
    w = wl("rms_bwd_add_bf16_32768x12288", 64, 65536)
    inp = make_inputs(w)
    c = lambda t: t.cuda()
    x, g, dz, dres = c(inp["x"]), c(inp["gamma"]), c(inp["dz"]), c(inp["dresidual"])
    o = gpu.fwd_outputs(w.rows, w.hidden, torch.bfloat16, "rmsnorm")
    ws = gpu.bwd_workspace(w.rows, w.hidden, torch.bfloat16, torch.bfloat16, "rmsnorm")
    dx, dg = torch.empty_like(x), torch.empty_like(g)

    def step():
        gpu.norm_fwd(x, g, None, norm="rmsnorm", eps=w.eps, outputs=o)
        gpu.norm_bwd(dz, x, None, o["rsigma"], g, dres, norm="rmsnorm", workspace=ws, dx=dx,
                     dgamma=dg)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o["out"], o["rsigma"], dx, dg)]
    for t in (o["out"], dx, dg):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (o["out"], o["rsigma"], dx, dg)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("scaling,layout,norm", [("delayed", "rowwise_colwise", "rmsnorm"),
                                                 ("mxfp8", "colwise", "layernorm")])
def test_long_row_colwise_statistics_in_workspace(gpu, scaling, layout, norm):
    """Without the mu / rsigma outputs the columnwise tile kernel reads the
    row statistics from the workspace: every output is bit-identical to the
    call that writes them to mu / rsigma."""
    import torch
    from rmsnorm_fp8_quantization_gb300.workloads import make_inputs
    name = "rms_bf16_e4m3_delayed_32768x8192" if scaling == "delayed" else "rms_bf16_mxfp8_16384x5120"
    w = wl(name, 64, 49152, layout=layout, norm=norm, w_dtype="f32", beta_std=0.1)
    inp = make_inputs(w)
    c = lambda t: None if t is None else t.cuda()
    kw = dict(norm=norm, eps=w.eps, zero_centered_gamma=w.zero_centered_gamma, scaling=scaling,
              layout=layout, scale=c(inp["scale"]), amax=c(inp["amax"]))
    x, g, b = c(inp["x"]), c(inp["gamma"]), c(inp["beta"])
    train = gpu.norm_fwd(x, g, b, training=True, **kw)
    infer = gpu.norm_fwd(x, g, b, training=False, **kw)
    assert infer["rsigma"] is None
    for k, v in infer.items():
        if v is not None:
            assert torch.equal(v, train[k]), k


def test_long_row_colwise_without_statistics_falls_back(gpu):
    """Without mu / rsigma and with a workspace below the queried size the
    columnwise long-row call still succeeds, on the generic kernel: its codes
    match the two-kernel path's except where the two kernels' fp32 statistics
    put a value next to a rounding boundary (at most 0.1 % of the codes, one
    step apart), and the amax agrees to rel 1e-5."""
    import torch
    from rmsnorm_fp8_quantization_gb300.workloads import make_inputs
    w = wl("rms_bf16_e4m3_delayed_32768x8192", 64, 49152, layout="colwise")
    inp = make_inputs(w)
    c = lambda t: None if t is None else t.cuda()
    kw = dict(norm=w.norm, eps=w.eps, scaling="delayed", layout="colwise",
              scale=c(inp["scale"]), amax=c(inp["amax"]))
    x, g = c(inp["x"]), c(inp["gamma"])
    two = gpu.norm_fwd(x, g, None, training=True, **kw)
    fall = gpu.norm_fwd(x, g, None, training=False,
                        workspace=torch.empty(0, dtype=torch.uint8, device="cuda"), **kw)
    a = two["colwise_out"].cpu().to(torch.int16)
    b = fall["colwise_out"].cpu().to(torch.int16)
    diff = (a != b)
    assert diff.float().mean().item() <= 1e-3
    # E4M3 codes of one sign are ordered like their values: a step is +-1
    assert ((a - b).abs()[diff] == 1).all()
    ra, rb = two["updated_amax"].item(), fall["updated_amax"].item()
    assert abs(ra - rb) <= 1e-5 * abs(ra)
