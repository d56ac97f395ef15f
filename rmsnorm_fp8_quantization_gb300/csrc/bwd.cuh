// Backward kernels: the row pass (dx, optionally + dresidual, and per-CTA
// partial dgamma/dbeta), its generic fallback, and the finalize pass.
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

// Row pass.  Persistent CTAs over rows (row = blockIdx.x + k*gridDim.x); each
// thread owns the NV vectors v = k*T + t of every row, so its dgamma/dbeta
// partials stay in registers across all rows of the CTA and are written once,
// as row blockIdx.x of the [P, hidden] fp32 workspace slabs.  The next row's
// dz, x (and dresidual) are prefetched into L2 while this row is reduced.
template <typename Tin, bool LN, bool ADD, int NV>
__global__ void __launch_bounds__(bwd_max_threads(NV)) bwd_row_kernel(const BwdParams p) {
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  __shared__ float2 red[2][32];
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const int H = p.hidden;
  const int nvec = H / VEC;
  constexpr bool ln = LN;
  const float gadd = p.zcg ? 1.f : 0.f;
  const float fH = static_cast<float>(H);
  const uint32_t row_bytes = static_cast<uint32_t>(H) * sizeof(Tin);
  const Tin* dzp = reinterpret_cast<const Tin*>(p.dz);
  const Tin* xp = reinterpret_cast<const Tin*>(p.x);
  const Tin* drp = reinterpret_cast<const Tin*>(p.dres);

  float dg[NV][VEC], db[LN ? NV : 1][VEC];
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      dg[k][e] = 0.f;
      if constexpr (LN) db[k][e] = 0.f;
    }
  int rb = 0;

  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const int64_t base = row * H;
    if (tid < (ADD ? 3 : 2) && row + gridDim.x < p.rows) {
      const int64_t nb = base + static_cast<int64_t>(gridDim.x) * H;
      const Tin* src = tid == 0 ? dzp : (tid == 1 ? xp : drp);
      prefetch_l2(src + nb, row_bytes);
    }
    uint32_t dzw[NV][NW], xw[NV][NW], rw[ADD ? NV : 1][NW];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v = k * T + tid;
      if (v < nvec) {
        ld_vec_raw<Tin, VEC, true>(dzp + base + v * VEC, dzw[k]);
        ld_vec_raw<Tin, VEC, true>(xp + base + v * VEC, xw[k]);
        if constexpr (ADD) ld_vec_raw<Tin, VEC, true>(drp + base + v * VEC, rw[k]);
      } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          dzw[k][i] = 0u;
          xw[k][i] = 0u;
          if constexpr (ADD) rw[k][i] = 0u;
        }
      }
    }
    const float mu = ln ? p.mu[row] : 0.f;
    const float rs = p.rsigma[row];

    float2 s = make_float2(0.f, 0.f);  // (sum dy, sum dy * xhat)
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v = k * T + tid;
      if (v < nvec) {
        float fz[VEC], fx[VEC], g[VEC];
        unpack<Tin, VEC>(dzw[k], fz);
        unpack<Tin, VEC>(xw[k], fx);
        ld_weights<VEC>(p.gamma, p.w_dt, v * VEC, g);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float xh = (fx[e] - mu) * rs;
          const float dy = fz[e] * (g[e] + gadd);
          s.x += dy;
          s.y = fmaf(dy, xh, s.y);
          dg[k][e] = fmaf(fz[e], xh, dg[k][e]);
          if constexpr (LN) db[k][e] += fz[e];
        }
      }
    }
    s = block_sum2(s, red[rb], lane, warp, nwarps);
    rb ^= 1;
    const float c1 = ln ? s.x / fH : 0.f;
    const float c2 = s.y / fH;

#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v = k * T + tid;
      if (v < nvec) {
        float fz[VEC], fx[VEC], g[VEC], o[VEC];
        unpack<Tin, VEC>(dzw[k], fz);
        unpack<Tin, VEC>(xw[k], fx);
        ld_weights<VEC>(p.gamma, p.w_dt, v * VEC, g);
        float fr[VEC];
        if constexpr (ADD) unpack<Tin, VEC>(rw[k], fr);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float xh = (fx[e] - mu) * rs;
          const float dy = fz[e] * (g[e] + gadd);
          float d = rs * (dy - c1 - xh * c2);
          if constexpr (ADD) d += fr[e];
          o[e] = d;
        }
        uint32_t w[NW];
        pack<Tin, VEC>(o, w);
        st_words<NW>(reinterpret_cast<Tin*>(p.dx) + base + v * VEC, w);
      }
    }
  }

  // Partials of this CTA (zeros for a CTA that saw no row).
  float* pg = p.part_dgamma + static_cast<int64_t>(blockIdx.x) * H;
  float* pb = ln ? p.part_dbeta + static_cast<int64_t>(blockIdx.x) * H : nullptr;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = k * T + tid;
    if (v < nvec) {
      uint32_t w[VEC];
      pack<float, VEC>(dg[k], w);
      st_words<VEC>(pg + v * VEC, w);
      if constexpr (LN) {
        pack<float, VEC>(db[k], w);
        st_words<VEC>(pb + v * VEC, w);
      }
    }
  }
}

// Generic backward: any hidden size and alignment.  Each CTA keeps its
// partial dgamma/dbeta directly in its own workspace row (columns owned by
// one thread each, so no synchronization is needed on them).
template <typename Tin>
__global__ void __launch_bounds__(256) bwd_generic_kernel(const BwdParams p) {
  __shared__ float2 red[2][32];
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
