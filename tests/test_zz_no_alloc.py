"""gbn_norm_bwd_noalloc, the backward for callers that cannot allocate device
memory at the point where they run it (a framework replaying a fixed memory
plan, a plugin host without an allocator, a caller inside a custom
allocator's own callback): it must give exactly what gbn_norm_bwd gives with
a caller-provided workspace, because it runs the same kernels on the same
grid with the partial sums in the library's own scratch array instead.

Collected last (file name) so that a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(G, dz, x, mu, rs, gamma, dres, dx, dg, db, norm, zcg):
    rows, hidden = x.shape
    return G.gbn_norm_bwd_noalloc(dz, x, mu, rs, gamma, dres, dx, dg, db, rows, hidden,
                                  G.TORCH_DTYPE[x.dtype], G.TORCH_DTYPE[gamma.dtype],
                                  G.GBN_LAYERNORM if norm == "layernorm" else G.GBN_RMSNORM,
                                  zcg, 0)


def _problem(name, rows, hidden, seed):
    w = WORKLOADS[name].with_shape(rows, hidden)
    inp = make_inputs(w, seed=seed)
    c = lambda t: None if t is None else t.cuda()
    ln = w.norm == "layernorm"
    g = torch.Generator().manual_seed(seed)
    rs = (torch.rand(rows, generator=g) + 0.5).cuda()
    mu = (torch.randn(rows, generator=g) * 0.1).cuda() if ln else None
    return w, c(inp["dz"]), c(inp["x"]), mu, rs, c(inp["gamma"]), c(inp["dresidual"])


def _outputs(x, gamma, ln):
    nan = float("nan")
    return (torch.full_like(x, nan), torch.full_like(gamma, nan),
            torch.full_like(gamma, nan) if ln else None)


@pytest.mark.parametrize("name,rows,hidden", [
    ("ln_bf16_16384x4096", 300, 4096),
    ("rms_bwd_add_bf16_32768x12288", 257, 12288),
    ("rms_f32_64x1024", 64, 1024),
])
def test_noalloc_matches_workspace_backward(gpu, name, rows, hidden):
    from rmsnorm_fp8_quantization_gb300 import gbnorm as G
    w, dz, x, mu, rs, gamma, dres = _problem(name, rows, hidden, seed=3)
    ln = w.norm == "layernorm"
    # Reference: the allocating entry point with a NaN-filled workspace, so a
    # partial row the kernels failed to write would show.
    ws = gpu.bwd_workspace(rows, hidden, x.dtype, gamma.dtype, w.norm).fill_(0xFF)
    ref = gpu.norm_bwd(dz, x, mu, rs, gamma, dres, norm=w.norm, workspace=ws)
    torch.cuda.synchronize()
    # Another problem that fills more of the scratch, with other values.
    w2, *other = _problem("ln_bf16_16384x4096", 2000, 8192, seed=11)
    for call in range(2):
        if call == 1:
            o2 = _outputs(other[1], other[4], True)
            st = _noalloc(G, *other, *o2, "layernorm", False)
            assert st == G.GBN_OK, G.gbn_status_string(st)
        dx, dg, db = _outputs(x, gamma, ln)
        st = _noalloc(G, dz, x, mu, rs, gamma, dres, dx, dg, db, w.norm, False)
        assert st == G.GBN_OK, G.gbn_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(dx, ref[0]), f"call {call}: dx differs"
        assert torch.equal(dg, ref[1]), f"call {call}: dgamma differs"
        if ln:
            assert torch.equal(db, ref[2]), f"call {call}: dbeta differs"


def test_noalloc_rejects_oversized_problem(gpu):
    from rmsnorm_fp8_quantization_gb300 import gbnorm as G
    # partial rows of (SMs x CTAs per SM) x hidden fp32 do not fit the scratch
    rows, hidden = 1 << 20, 1 << 22
    st, need = G.gbn_norm_bwd_workspace_size(rows, hidden, G.GBN_BF16, G.GBN_BF16,
                                             G.GBN_LAYERNORM, 0, 0)
    assert st == G.GBN_OK and need > (32 << 20)
    # Row-sized buffers are NULL: were the size check ever moved after the
    # argument checks, the call would return GBN_ERR_NULL, never launch.
    gamma = torch.ones(8, dtype=torch.bfloat16, device="cuda")
    dg, db = torch.empty_like(gamma), torch.empty_like(gamma)
    st = G.gbn_norm_bwd_noalloc(None, None, None, None, gamma, None, None, dg, db, rows, hidden,
                                G.GBN_BF16, G.GBN_BF16, G.GBN_LAYERNORM, 0, 0, stream=0)
    assert st == G.GBN_ERR_WORKSPACE
