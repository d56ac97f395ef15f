"""GPU parity of the scaled (masked) softmax, forward and backward, against
the float64 oracle on the same seeded inputs: every mask kind, bf16 / f16 /
f32, vector and scalar paths, rows from 1 group of 32 lanes up to the longest
row (eight warps), fully masked rows, in-place calls and shape errors.

Tolerance (per element, written here from the arithmetic): the stored
result's rounding (1 ulp of the reference for bf16 / f16, 1e-5 relative for
fp32) plus 8 * 2^-24 * T, T the magnitude the fp32 evaluation can be off by:
forward, y * (|scale * x - max| * log2(e) + 64 + log2(sk)) -- the exp2
argument's rounding and the row sum's; backward,
|scale| * y * (|dy| + sum_j |dy_j| y_j)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import softmax as S
from parity import check_float
from rmsnorm_fp8_quantization_gb300.workloads import SOFTMAX_WORKLOADS, make_softmax_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
KIND = {"none": S.NONE, "padding": S.PADDING, "causal": S.CAUSAL_UPPER,
        "causal_aligned": S.CAUSAL_ALIGNED}
CAUSAL = SOFTMAX_WORKLOADS["softmax_causal_bf16_8x16x2048x2048"]


def wl(b, h, sq, sk, dtype="bf16", mask="none", **kw):
    return dataclasses.replace(CAUSAL, batches=b, heads=h, sq=sq, sk=sk, dtype=dtype, mask=mask,
                               **kw)


CASES = [
    wl(2, 4, 64, 1000),
    wl(1, 2, 33, 2048, dtype="f16"),
    wl(3, 2, 40, 256, dtype="f16", mask="padding", mask_batches=1),
    wl(3, 2, 40, 256, mask="padding", mask_batches=3, mask_frac=0.6),
    wl(4, 2, 128, 128, mask="causal"),
    wl(2, 2, 48, 80, mask="causal_aligned"),
    wl(2, 2, 80, 48, mask="causal_aligned"),          # rows before the keys: all masked
    wl(1, 1, 16, 16384),                               # longest row: 8 warps per row
    wl(1, 2, 9, 8192, dtype="f32", mask="causal_aligned"),
    wl(2, 1, 21, 1001),                                # odd row length: scalar path
    wl(1, 1, 33, 777, dtype="f32", mask="padding", mask_batches=1),
    wl(1, 3, 5, 8, dtype="f32"),                       # one short vector per row
]


def _ids(w):
    return f"{w.mask}-{w.dtype}-{w.batches}x{w.heads}x{w.sq}x{w.sk}"


def _fwd_terms(x, scale, keep, y):
    t = np.where(keep, scale * x.astype(np.float64), -np.inf)
    m = t.max(-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    d = np.where(keep, np.abs(t - m), 0.0)
    return y * (d * math.log2(math.e) + 64 + math.log2(x.shape[-1]))


@pytest.mark.parametrize("w", CASES, ids=_ids)
def test_softmax_forward_and_backward(gpu, w):
    inp = make_softmax_inputs(w)
    x, dy, mask = inp["x"], inp["dy"], inp["mask"]
    dt = DT[w.dtype]
    y = gpu.softmax_fwd(x.cuda(), w.scale, w.mask, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    xd = x.double().numpy()
    ref = S.softmax_fwd(xd, KIND[w.mask], w.scale, None if mask is None else mask.numpy())
    keep = S.keep_mask(KIND[w.mask], w.batches, w.heads, w.sq, w.sk,
                       None if mask is None else mask.numpy())
    check_float("y", y, ref, dt, terms=_fwd_terms(xd, w.scale, keep, ref))
    assert torch.all(y.cpu()[torch.from_numpy(~keep)] == 0)

    # backward from the GPU forward's stored output (both sides)
    dx = gpu.softmax_bwd(dy.cuda(), y, w.scale)
    torch.cuda.synchronize()
    yd = y.cpu().double().numpy()
    dyd = dy.double().numpy()
    rdx = S.softmax_bwd(dyd, yd, w.scale)
    t_dx = abs(w.scale) * yd * (np.abs(dyd) + (np.abs(dyd) * yd).sum(-1, keepdims=True))
    check_float("dx", dx, rdx, dt, terms=t_dx)


def test_in_place_matches_out_of_place(gpu):
    w = wl(2, 2, 64, 512, mask="causal_aligned")
    inp = make_softmax_inputs(w)
    x = inp["x"].cuda()
    y = gpu.softmax_fwd(x, w.scale, w.mask)
    x2 = x.clone()
    gpu.softmax_fwd(x2, w.scale, w.mask, out=x2)
    assert torch.equal(x2, y)
    dy = inp["dy"].cuda()
    dx = gpu.softmax_bwd(dy, y, w.scale)
    gpu.softmax_bwd(dy, y, w.scale, out=dy)
    assert torch.equal(dy, dx)


def test_shape_errors(gpu):
    from rmsnorm_fp8_quantization_gb300.gbnorm import GbnError
    with pytest.raises(GbnError):   # beyond the longest row
        gpu.softmax_fwd(torch.zeros(1, 1, 2, 16392, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(GbnError):   # scalar path beyond 2048 keys
        gpu.softmax_fwd(torch.zeros(1, 1, 2, 3001, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(GbnError):   # upper-triangular needs sq == sk
        gpu.softmax_fwd(torch.zeros(1, 1, 4, 8, dtype=torch.bfloat16, device="cuda"),
                        mask_kind="causal")


def test_softmax_graph_capture_and_guard_bands(gpu):
    w = wl(2, 2, 128, 2048, mask="causal_aligned")
    inp = make_softmax_inputs(w)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    n = x.numel()
    G = 2048
    ybuf = torch.full((n + 2 * G,), 7.0, dtype=x.dtype, device="cuda")
    y = ybuf[G:G + n].view(x.shape)
    dxbuf = torch.full((n + 2 * G,), 7.0, dtype=x.dtype, device="cuda")
    dx = dxbuf[G:G + n].view(x.shape)

    def step():
        gpu.softmax_fwd(x, w.scale, w.mask, out=y)
        gpu.softmax_bwd(dy, y, w.scale, out=dx)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = (y.clone(), dx.clone())
    y.zero_()
    dx.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager[0], y) and torch.equal(eager[1], dx)
    for buf in (ybuf, dxbuf):
        assert torch.all(buf[:G] == 7.0) and torch.all(buf[G + n:] == 7.0), "guard band written"
