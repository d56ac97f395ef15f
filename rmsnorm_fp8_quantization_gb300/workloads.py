"""Seeded synthetic workloads for the fused norm path.

This module only draws random inputs; it holds none of the normalization or
quantization arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method's code.

Draw order for every workload (one ``torch.Generator`` on the CPU, seeded):
x, gamma, beta, dz, dresidual, then the structure (outlier channels, per-row
magnitudes).  Each tensor is drawn in float32 and cast once to its stored
dtype, so both sides see the same stored bytes.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    norm: str                  # "layernorm" | "rmsnorm"
    rows: int
    hidden: int
    in_dtype: str              # "f32" | "bf16" | "f16"
    w_dtype: str
    eps: float
    scaling: str = "none"      # "none" | "delayed" | "mxfp8"
    layout: str = "rowwise"    # "rowwise" | "colwise" | "rowwise_colwise"
    zero_centered_gamma: bool = False
    passes: tuple = ("fwd", "bwd")
    x_mean: float = 0.0
    x_std: float = 1.0
    gamma_mean: float = 1.0    # gamma ~ gamma_mean + gamma_std * N(0,1)
    gamma_std: float = 0.1
    beta_std: float = 0.0      # LayerNorm beta ~ beta_std * N(0,1)
    outlier_frac: float = 0.0  # fraction of channels multiplied by outlier_gain
    outlier_gain: float = 1.0
    row_log10_range: Optional[tuple] = None  # per-row magnitude 10^U(lo, hi)
    dresidual: bool = False
    amax_prev: float = 0.0     # delayed scaling: scale = 448 / amax_prev

    def with_shape(self, rows: int, hidden: Optional[int] = None) -> "Workload":
        return dataclasses.replace(self, rows=rows, hidden=self.hidden if hidden is None else hidden)


WORKLOADS = {
    # RMSNorm fwd+bwd, fp32 in/out/weights, 64 x 1024.
    "rms_f32_64x1024": Workload(
        "rms_f32_64x1024", "rmsnorm", 64, 1024, "f32", "f32", 1e-6),
    # LayerNorm fwd+bwd, bf16 in/out, fp32 gamma/beta, 16384 x 4096.
    "ln_bf16_16384x4096": Workload(
        "ln_bf16_16384x4096", "layernorm", 16384, 4096, "bf16", "f32", 1e-5,
        x_mean=0.5, x_std=2.0, beta_std=0.1),
    # Same with a hidden size that is not a power of two.
    "ln_bf16_16384x4000": Workload(
        "ln_bf16_16384x4000", "layernorm", 16384, 4000, "bf16", "f32", 1e-5,
        x_mean=0.5, x_std=2.0, beta_std=0.1),
    # Long rows (each split over a thread-block cluster): LayerNorm fwd+bwd, 4096 x 65536.
    "ln_bf16_4096x65536": Workload(
        "ln_bf16_4096x65536", "layernorm", 4096, 65536, "bf16", "f32", 1e-5,
        x_mean=0.5, x_std=2.0, beta_std=0.1),
    # RMSNorm fwd bf16 -> E4M3, delayed per-tensor scaling, rowwise + transposed colwise.
    "rms_bf16_e4m3_delayed_32768x8192": Workload(
        "rms_bf16_e4m3_delayed_32768x8192", "rmsnorm", 32768, 8192, "bf16", "bf16", 1e-6,
        scaling="delayed", layout="rowwise_colwise", passes=("fwd",),
        outlier_frac=0.001, outlier_gain=20.0, amax_prev=30.0),
    # RMSNorm fwd bf16 -> MXFP8 (1x32 rowwise, 32x1 colwise E8M0 scales), zero-centered gamma.
    "rms_bf16_mxfp8_16384x5120": Workload(
        "rms_bf16_mxfp8_16384x5120", "rmsnorm", 16384, 5120, "bf16", "bf16", 1e-6,
        scaling="mxfp8", layout="rowwise_colwise", zero_centered_gamma=True, passes=("fwd",),
        gamma_mean=0.0, gamma_std=0.05, row_log10_range=(-2.0, 2.0)),
    # Fused backward-add RMSNorm, bf16 tensors, 32768 x 12288.
    "rms_bwd_add_bf16_32768x12288": Workload(
        "rms_bwd_add_bf16_32768x12288", "rmsnorm", 32768, 12288, "bf16", "bf16", 1e-6,
        passes=("bwd",), dresidual=True),
}


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu") -> dict:
    """Draws the workload's inputs in their stored dtypes on `device`.

    The same seed gives the same values on every run on one device type; the
    CPU and CUDA generators draw different streams.

    Keys: x, gamma, beta (LayerNorm, else None), dz, dresidual (or None),
    scale (fp32 [1], delayed scaling, else None), amax (fp32 [1] previous
    amax, delayed scaling, else None).
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    R, H = w.rows, w.hidden
    kw = dict(generator=g, dtype=torch.float32, device=device)

    def draw(*shape):
        t = torch.empty(*shape, dtype=torch.float32, device=device)
        return t.normal_(generator=g)

    x = draw(R, H).mul_(w.x_std).add_(w.x_mean)
    gamma = draw(H).mul_(w.gamma_std).add_(w.gamma_mean)
    beta = None
    if w.norm == "layernorm":
        beta = draw(H).mul_(w.beta_std)
    dz = draw(R, H)
    dres = draw(R, H) if w.dresidual else None
    if w.outlier_frac > 0:
        n_out = max(1, int(round(H * w.outlier_frac)))
        ch = torch.randperm(H, generator=g, device=device)[:n_out]
        x[:, ch] *= w.outlier_gain
    if w.row_log10_range is not None:
        lo, hi = w.row_log10_range
        u = torch.rand(R, **kw).to(torch.float64)
        mag = torch.pow(10.0, u * (hi - lo) + lo)
        x *= mag.to(torch.float32)[:, None]
    it, wt = _DT[w.in_dtype], _DT[w.w_dtype]
    out = {
        "x": x.to(it),
        "gamma": gamma.to(wt),
        "beta": None if beta is None else beta.to(wt),
        "dz": dz.to(it),
        "dresidual": None if dres is None else dres.to(it),
        "scale": None,
        "amax": None,
    }
    if w.scaling == "delayed":
        out["scale"] = torch.tensor([448.0 / w.amax_prev], dtype=torch.float32, device=device)
        out["amax"] = torch.tensor([w.amax_prev], dtype=torch.float32, device=device)
    return out


# ---------------------------------------------------------------- softmax

@dataclasses.dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    batches: int
    heads: int
    sq: int
    sk: int
    dtype: str                 # "f32" | "bf16" | "f16"
    mask: str = "none"         # "none" | "padding" | "causal" | "causal_aligned"
    scale: float = 0.125
    x_std: float = 4.0         # logits ~ x_std * N(0, 1)
    mask_batches: int = 1
    mask_frac: float = 0.25    # padding: fraction of masked positions

    def with_shape(self, batches, heads, sq, sk) -> "SoftmaxWorkload":
        return dataclasses.replace(self, batches=batches, heads=heads, sq=sq, sk=sk)


SOFTMAX_WORKLOADS = {
    # Causal (upper-triangular) attention probabilities, bf16, 8 x 16 heads x 2048 x 2048.
    "softmax_causal_bf16_8x16x2048x2048": SoftmaxWorkload(
        "softmax_causal_bf16_8x16x2048x2048", 8, 16, 2048, 2048, "bf16", mask="causal"),
    # Padding-masked attention probabilities, bf16, 8 x 16 x 1024 x 1024, one mask per batch.
    "softmax_padding_bf16_8x16x1024x1024": SoftmaxWorkload(
        "softmax_padding_bf16_8x16x1024x1024", 8, 16, 1024, 1024, "bf16", mask="padding",
        mask_batches=8),
}


def make_softmax_inputs(w: SoftmaxWorkload, seed: int = 0, device: str = "cpu") -> dict:
    """Seeded inputs of a softmax workload: x (logits), dy, and the padding
    mask (uint8, nonzero = masked) or None.  Draw order: x, dy, mask."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (w.batches, w.heads, w.sq, w.sk)
    x = torch.empty(shape, dtype=torch.float32, device=device).normal_(generator=g)
    x.mul_(w.x_std)
    dy = torch.empty(shape, dtype=torch.float32, device=device).normal_(generator=g)
    mask = None
    if w.mask == "padding":
        u = torch.rand((w.mask_batches, 1, w.sq, w.sk), generator=g, device=device)
        mask = (u < w.mask_frac).to(torch.uint8)
    dt = _DT[w.dtype]
    return {"x": x.to(dt), "dy": dy.to(dt), "mask": mask}
