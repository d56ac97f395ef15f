// Generic backward kernel (any size and alignment): dx (optionally +
// dresidual) and per-CTA partial dgamma/dbeta.  The fast path is the ring
// kernel (ring.cuh); the finalize pass is in finalize.cu.
//
// Operation: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Description (backward handler dispatching to the LayerNorm / RMSNorm
// backward), and "Implementation:NVIDIA TransformerEngine Ops Fused Backward
// Add RMSNorm", Description and I/O Contract (grad_input = RMSNorm backward +
// residual gradient in one kernel; grad_weight).  The bwd = row pass +
// finalize structure follows the dispatch flowchart of "Migrate norms and
// softmax kernels to NVRTC" ("For bwd: also launch finalize kernel").
#pragma once

#include "gbn_device.cuh"

namespace gbn {

// Generic backward: any hidden size and alignment.  Each CTA keeps its
// partial dgamma/dbeta directly in its own workspace row (columns owned by
// one thread each, so no synchronization is needed on them).
template <typename Tin>
__global__ void __launch_bounds__(256) bwd_generic_kernel(const BwdParams p) {
  pdl_begin();
  __shared__ __align__(16) float2 red[2][32];
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const int H = p.hidden;
  const bool ln = (p.norm == 0);
  const float gadd = p.zcg ? 1.f : 0.f;
  const float fH = static_cast<float>(H);
  const Tin* dzp = reinterpret_cast<const Tin*>(p.dz);
  const Tin* xp = reinterpret_cast<const Tin*>(p.x);
  const Tin* drp = reinterpret_cast<const Tin*>(p.dres);
  float* pg = p.part_dgamma + static_cast<int64_t>(blockIdx.x) * H;
  float* pb = ln ? p.part_dbeta + static_cast<int64_t>(blockIdx.x) * H : nullptr;
  for (int j = tid; j < H; j += T) {
    pg[j] = 0.f;
    if (ln) pb[j] = 0.f;
  }
  // slots past the warp count read as zero in the block sums; no warp writes them
  for (int i = nwarps + tid; i < 32; i += T) red[0][i] = red[1][i] = make_float2(0.f, 0.f);
  int rb = 0;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const int64_t base = row * H;
    const float mu = ln ? p.mu[row] : 0.f;
    const float rs = p.rsigma[row];
    float2 s = make_float2(0.f, 0.f);
    for (int j = tid; j < H; j += T) {
      const float fz = ld_scalar(dzp, base + j);
      const float xh = (ld_scalar(xp, base + j) - mu) * rs;
      const float dy = fz * (ld_weight_scalar(p.gamma, p.w_dt, j) + gadd);
      s.x += dy;
      s.y = fmaf(dy, xh, s.y);
      pg[j] = fmaf(fz, xh, pg[j]);
      if (ln) pb[j] += fz;
    }
    s = block_sum2(s, red[rb], lane, warp, nwarps);
    rb ^= 1;
    const float c1 = ln ? s.x / fH : 0.f;
    const float c2 = s.y / fH;
    for (int j = tid; j < H; j += T) {
      const float fz = ld_scalar(dzp, base + j);
      const float xh = (ld_scalar(xp, base + j) - mu) * rs;
      const float dy = fz * (ld_weight_scalar(p.gamma, p.w_dt, j) + gadd);
      float d = rs * (dy - c1 - xh * c2);
      if (drp) d += ld_scalar(drp, base + j);
      st_scalar(reinterpret_cast<Tin*>(p.dx), base + j, d);
    }
  }
}

}  // namespace gbn
