"""Allocating wrappers over the C ABI: build the output tensors with torch,
call ``gbn_norm_fwd`` / ``gbn_norm_bwd`` and raise on a non-OK status.

The norm itself runs in the library's CUDA kernels; these functions only
allocate device memory and marshal arguments.
"""
from __future__ import annotations

import torch

from . import gbnorm as G

_NORM = {"layernorm": G.GBN_LAYERNORM, "rmsnorm": G.GBN_RMSNORM}
_SCALING = {"none": G.GBN_SCALING_NONE, "delayed": G.GBN_SCALING_DELAYED_TENSOR,
            "mxfp8": G.GBN_SCALING_MXFP8_1D}
_LAYOUT = {"rowwise": G.GBN_LAYOUT_ROWWISE, "colwise": G.GBN_LAYOUT_COLWISE,
           "rowwise_colwise": G.GBN_LAYOUT_ROWWISE_COLWISE}


def _check(st, where):
    if st != G.GBN_OK:
        raise G.GbnError(st, where)


def _roundup(a, b):
    return (a + b - 1) // b * b


def mx_scale_shapes(rows, hidden, swizzled=False):
    """Shapes of the MXFP8 (rowwise, colwise) E8M0 scale buffers.  Swizzled:
    padded to the 128 x 4 tiles of the GEMM order (colwise as the transposed
    operand: hidden outer, rows/32 inner)."""
    if not swizzled:
        return (rows, hidden // 32), (rows // 32, hidden)
    return ((_roundup(rows, 128), _roundup(hidden // 32, 4)),
            (_roundup(hidden, 128), _roundup(rows // 32, 4)))


def fwd_outputs(rows, hidden, in_dtype, norm="layernorm", scaling="none", layout="rowwise",
                device="cuda", training=True, swizzled_scales=False):
    """Allocates every output buffer the forward writes for this configuration."""
    dev = torch.device(device)
    o = {"out": None, "colwise_out": None, "mu": None, "rsigma": None, "scale_inv": None,
         "colwise_scale_inv": None, "updated_amax": None}
    rowwise = scaling == "none" or layout != "colwise"
    colwise = scaling != "none" and layout != "rowwise"
    if rowwise:
        o["out"] = torch.empty(rows, hidden, dtype=in_dtype if scaling == "none" else torch.uint8,
                               device=dev)
    if training:
        o["rsigma"] = torch.empty(rows, dtype=torch.float32, device=dev)
        if norm == "layernorm":
            o["mu"] = torch.empty(rows, dtype=torch.float32, device=dev)
    if scaling == "delayed":
        o["updated_amax"] = torch.empty(1, dtype=torch.float32, device=dev)
        if rowwise:
            o["scale_inv"] = torch.empty(1, dtype=torch.float32, device=dev)
        if colwise:
            o["colwise_out"] = torch.empty(hidden, rows, dtype=torch.uint8, device=dev)
            o["colwise_scale_inv"] = torch.empty(1, dtype=torch.float32, device=dev)
    elif scaling == "mxfp8":
        rs, cs = mx_scale_shapes(rows, hidden, swizzled_scales)
        if rowwise:
            o["scale_inv"] = torch.empty(rs, dtype=torch.uint8, device=dev)
        if colwise:
            o["colwise_out"] = torch.empty(rows, hidden, dtype=torch.uint8, device=dev)
            o["colwise_scale_inv"] = torch.empty(cs, dtype=torch.uint8, device=dev)
    return o


def norm_fwd(x, gamma, beta=None, *, norm="layernorm", eps=1e-5, zero_centered_gamma=False,
             scaling="none", layout="rowwise", scale=None, amax=None, sm_margin=0,
             training=True, outputs=None, stream=None, swizzled_scales=False, workspace=None):
    """Runs the fused forward; returns the dict of output tensors.
    ``swizzled_scales`` (MXFP8): scales in the padded, tiled GEMM order.
    ``workspace``: a uint8 device tensor of at least the queried size; allocated
    here when the call needs one (columnwise layouts of long rows without the
    mu / rsigma outputs)."""
    rows, hidden = x.shape
    o = outputs if outputs is not None else fwd_outputs(rows, hidden, x.dtype, norm, scaling,
                                                        layout, x.device, training,
                                                        swizzled_scales)
    in_dt = G.TORCH_DTYPE[x.dtype]
    out_dt = in_dt if scaling == "none" else G.GBN_E4M3
    lay = _LAYOUT[layout] | (G.GBN_LAYOUT_SWIZZLED_SCALES if swizzled_scales else 0)
    if workspace is None and (o["rsigma"] is None or (norm == "layernorm" and o["mu"] is None)):
        st, n = G.gbn_norm_fwd_workspace_size(rows, hidden, in_dt, G.TORCH_DTYPE[gamma.dtype],
                                              out_dt, _NORM[norm], _SCALING[scaling], lay,
                                              zero_centered_gamma, sm_margin, training)
        _check(st, "gbn_norm_fwd_workspace_size")
        if n:
            workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = G.gbn_norm_fwd(x, gamma, beta, scale, amax, o["out"], o["colwise_out"], o["mu"],
                        o["rsigma"], o["scale_inv"], o["colwise_scale_inv"], o["updated_amax"],
                        workspace, workspace.numel() if workspace is not None else 0, rows,
                        hidden, in_dt, G.TORCH_DTYPE[gamma.dtype], out_dt, _NORM[norm],
                        _SCALING[scaling], lay, zero_centered_gamma, eps, sm_margin, stream)
    _check(st, "gbn_norm_fwd")
    return o


def bwd_workspace(rows, hidden, in_dtype, w_dtype, norm="layernorm", zero_centered_gamma=False,
                  sm_margin=0, device="cuda"):
    st, n = G.gbn_norm_bwd_workspace_size(rows, hidden, G.TORCH_DTYPE[in_dtype],
                                          G.TORCH_DTYPE[w_dtype], _NORM[norm],
                                          zero_centered_gamma, sm_margin)
    _check(st, "gbn_norm_bwd_workspace_size")
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def norm_bwd(dz, x, mu, rsigma, gamma, dresidual=None, *, norm="layernorm",
             zero_centered_gamma=False, sm_margin=0, workspace=None, dx=None, dgamma=None,
             dbeta=None, stream=None):
    """Runs the fused backward; returns (dx, dgamma, dbeta or None)."""
    rows, hidden = x.shape
    if workspace is None:
        workspace = bwd_workspace(rows, hidden, x.dtype, gamma.dtype, norm, zero_centered_gamma,
                                  sm_margin, x.device)
    dx = torch.empty_like(x) if dx is None else dx
    dgamma = torch.empty_like(gamma) if dgamma is None else dgamma
    if norm == "layernorm" and dbeta is None:
        dbeta = torch.empty_like(gamma)
    st = G.gbn_norm_bwd(dz, x, mu if norm == "layernorm" else None, rsigma, gamma, dresidual, dx,
                        dgamma, dbeta if norm == "layernorm" else None, workspace,
                        workspace.numel(), rows, hidden, G.TORCH_DTYPE[x.dtype],
                        G.TORCH_DTYPE[gamma.dtype], _NORM[norm], zero_centered_gamma, sm_margin,
                        stream)
    _check(st, "gbn_norm_bwd")
    return dx, dgamma, dbeta if norm == "layernorm" else None


_SOFTMAX_MASK = {"none": G.GBN_SOFTMAX_NO_MASK, "padding": G.GBN_SOFTMAX_PADDING,
                 "causal": G.GBN_SOFTMAX_CAUSAL_UPPER,
                 "causal_aligned": G.GBN_SOFTMAX_CAUSAL_ALIGNED}


def softmax_fwd(x, scale=1.0, mask_kind="none", mask=None, out=None, stream=None):
    """Scaled (masked) softmax over the last axis of x [batches, heads, sq, sk];
    mask [mask_batches, 1, sq, sk] uint8 (nonzero = masked) for "padding"."""
    b, h, sq, sk = x.shape
    y = torch.empty_like(x) if out is None else out
    mb = 0 if mask is None else mask.shape[0]
    st = G.gbn_softmax_fwd(x, mask, y, b, h, sq, sk, mb, G.TORCH_DTYPE[x.dtype],
                           _SOFTMAX_MASK[mask_kind], scale, stream)
    _check(st, "gbn_softmax_fwd")
    return y


def softmax_bwd(dy, y, scale=1.0, out=None, stream=None):
    """dx = scale * y * (dy - sum(dy * y)) over the last axis."""
    sk = y.shape[-1]
    dx = torch.empty_like(dy) if out is None else out
    st = G.gbn_softmax_bwd(dy, y, dx, y.numel() // sk, sk, G.TORCH_DTYPE[y.dtype], scale, stream)
    _check(st, "gbn_softmax_bwd")
    return dx
