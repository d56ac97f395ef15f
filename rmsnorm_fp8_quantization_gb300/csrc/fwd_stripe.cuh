// Forward kernel for the columnwise FP8 layouts (delayed scaling with a
// transposed [hidden, rows] copy, MXFP8 with 32x1 column blocks), optionally
// together with the rowwise outputs.
//
// Operation: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Description ("rowwise and optional columnwise (2x2x layout) FP8 output
// tensors with scale/amax/scale_inv") and I/O Contract.
//
// A columnwise output needs 32 finished rows before any column can be
// written, and 32 rows of a long row do not fit one SM.  So a thread-block
// cluster of C CTAs takes one 32-row stripe: CTA `rank` owns columns
// [rank*hc, (rank+1)*hc).  Each CTA loads its 32 x hc slice into registers
// once, reduces per-row partial statistics, and exchanges them with the other
// CTAs through distributed shared memory; the row statistics are combined in
// the same fixed order in every CTA.  Rowwise codes go straight to HBM;
// columnwise codes are staged in shared memory and written as 32-byte column
// segments (delayed) or after a column-block amax pass (MXFP8).  x is read
// from HBM exactly once.
#pragma once

#include "gbn_device.cuh"

namespace gbn {

constexpr int kStripeRows = 32;
constexpr int kStripeWarps = 8;
constexpr int kRowsPerWarp = kStripeRows / kStripeWarps;  // 4 consecutive rows per warp

// Dynamic shared memory bytes of the stripe kernel for a slice of hc columns.
__host__ __device__ inline int stripe_smem_bytes(int qm, int hc) {
  if (qm == Q_DELAYED) return kStripeRows * hc;  // codes tile [32][hc]
  return (kStripeWarps + 1) * hc * 4;            // column partial maxima + multipliers
}

template <typename Tin, int QM, int NVS>
__global__ void __launch_bounds__(256, 1) fwd_stripe_kernel(const FwdParams p, const int hc) {
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  constexpr int RPW = kRowsPerWarp;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float2 stat[2][kStripeRows];  // per row: (local mean, local M2) of this slice
  __shared__ float red[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int H = p.hidden;
  const int c0 = static_cast<int>(rank) * hc;
  const int nvs = hc / VEC;  // vectors per row in this slice
  const int64_t N = p.rows;
  const int64_t nstripes = N / kStripeRows;
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const bool ln = (p.norm == 0);
  const float gadd = p.zcg ? 1.f : 0.f;
  const float fH = static_cast<float>(H), fhc = static_cast<float>(hc);
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  float amax_t = 0.f;
  const Tin* x = reinterpret_cast<const Tin*>(p.x);
  int buf = 0;

  for (int64_t s = cid; s < nstripes; s += ncl) {
    const int64_t i0 = s * kStripeRows;
    const int r0 = warp * RPW;  // first stripe row of this warp

    // ---- load the warp's 4 rows of this CTA's slice
    uint32_t xw[RPW][NVS][NW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const Tin* xr = x + (i0 + r0 + r) * H + c0;
#pragma unroll
      for (int j = 0; j < NVS; ++j) {
        const int v = j * 32 + lane;
        if (v < nvs) {
          ld_vec_raw<Tin, VEC, true>(xr + v * VEC, xw[r][j]);
        } else {
#pragma unroll
          for (int i = 0; i < NW; ++i) xw[r][j][i] = 0u;
        }
      }
    }
    if (lane < RPW && s + ncl < nstripes)
      prefetch_l2(x + (i0 + ncl * kStripeRows + r0 + lane) * H + c0,
                  static_cast<uint32_t>(hc * sizeof(Tin)));

    // ---- per-row statistics of this slice (one warp owns whole row slices)
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      float m = 0.f;
      if (ln) {
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < NVS; ++j) {
          float f[VEC];
          unpack<Tin, VEC>(xw[r][j], f);
#pragma unroll
          for (int e = 0; e < VEC; ++e) sum += f[e];
        }
        m = warp_sum(sum) / fhc;
      }
      float q = 0.f;
#pragma unroll
      for (int j = 0; j < NVS; ++j) {
        if (j * 32 + lane < nvs) {
          float f[VEC];
          unpack<Tin, VEC>(xw[r][j], f);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float d = f[e] - m;
            q = fmaf(d, d, q);
          }
        }
      }
      q = warp_sum(q);
      if (lane == 0) stat[buf][r0 + r] = make_float2(m, q);
    }
    cluster_sync();

    // ---- combine the C slices of each row, in rank order (same in every CTA)
    float mean[RPW], rs[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      float2 mine = make_float2(0.f, 0.f);
      if (lane < static_cast<int>(C)) mine = dsmem_ld2(&stat[buf][r0 + r], lane);
      float msum = 0.f, qsum = 0.f;
      for (uint32_t c = 0; c < C; ++c) {
        const float mc = __shfl_sync(0xFFFFFFFFu, mine.x, c);
        msum += mc;
      }
      const float mu = ln ? msum / static_cast<float>(C) : 0.f;
      for (uint32_t c = 0; c < C; ++c) {
        const float mc = __shfl_sync(0xFFFFFFFFu, mine.x, c);
        const float qc = __shfl_sync(0xFFFFFFFFu, mine.y, c);
        const float d = mc - mu;
        qsum += ln ? fmaf(fhc * d, d, qc) : qc;
      }
      mean[r] = mu;
      rs[r] = 1.f / sqrtf(qsum / fH + p.eps);
      if (rank == 0 && lane == 0) {
        if (ln && p.mu) p.mu[i0 + r0 + r] = mu;
        if (p.rsigma) p.rsigma[i0 + r0 + r] = rs[r];
      }
    }
    buf ^= 1;

    // ---- normalize; rowwise codes to HBM, columnwise material to smem
#pragma unroll
    for (int j = 0; j < NVS; ++j) {
      const int v = j * 32 + lane;
      const bool act = v < nvs;
      const int col = c0 + v * VEC;  // global column of element 0 of this vector
      float g[VEC], b[VEC];
      if (act) {
        ld_weights<VEC>(p.gamma, p.w_dt, col, g);
        if (ln) ld_weights<VEC>(p.beta, p.w_dt, col, b);
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        if (!act) g[e] = 0.f;
        if (!ln || !act) b[e] = 0.f;
        g[e] += gadd;
      }
      float cmax[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) cmax[e] = 0.f;
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const int64_t row = i0 + r0 + r;
        float f[VEC], z[VEC];
        unpack<Tin, VEC>(xw[r][j], f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) z[e] = act ? (f[e] - mean[r]) * rs[r] * g[e] + b[e] : 0.f;
        if constexpr (QM == Q_DELAYED) {
          if (act) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) amax_t = fmax_nan(amax_t, fabsf(z[e]));
            uint32_t w[VEC / 4];
            e4m3_pack_scaled<VEC>(z, qscale, w);
            if (p.write_rowwise) st_words<VEC / 4>(reinterpret_cast<uint8_t*>(p.out) + row * H + col, w);
            st_words<VEC / 4>(smem + (r0 + r) * hc + v * VEC, w);  // colwise tile [32][hc]
          }
        } else {  // MXFP8
          if (p.write_rowwise) {
            constexpr int TPB = 32 / VEC;
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) a = fmax_nan(a, fabsf(z[e]));
#pragma unroll
            for (int o = 1; o < TPB; o <<= 1) a = fmax_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            if (act) {
              const uint32_t c = e8m0_code(a);
              uint32_t w[VEC / 4];
              e4m3_pack_scaled<VEC>(z, e8m0_mult(c), w);
              st_words<VEC / 4>(reinterpret_cast<uint8_t*>(p.out) + row * H + col, w);
              if ((lane & (TPB - 1)) == 0) p.mx_scale[row * (H / 32) + col / 32] = static_cast<uint8_t>(c);
            }
          }
#pragma unroll
          for (int e = 0; e < VEC; ++e) cmax[e] = fmax_nan(cmax[e], fabsf(z[e]));
        }
      }
      if constexpr (QM == Q_MXFP8) {
        if (act) {
          float* colmax = reinterpret_cast<float*>(smem);  // [8 warps][hc]
#pragma unroll
          for (int e = 0; e < VEC; ++e) colmax[warp * hc + v * VEC + e] = cmax[e];
        }
      }
    }
    __syncthreads();

    if constexpr (QM == Q_DELAYED) {
      // ---- transposed write: thread takes 4 adjacent columns, 32 rows each
      const uint32_t* tile = reinterpret_cast<const uint32_t*>(smem);
      const int ngrp = hc / 4;
      for (int cg = tid; cg < ngrp; cg += 256) {
        uint32_t w[kStripeRows];
#pragma unroll
        for (int r = 0; r < kStripeRows; ++r) w[r] = tile[r * ngrp + cg];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t sel = static_cast<uint32_t>(cc) | (static_cast<uint32_t>(cc + 4) << 4);
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t lo = __byte_perm(w[4 * q], w[4 * q + 1], sel);
            const uint32_t hi = __byte_perm(w[4 * q + 2], w[4 * q + 3], sel);
            o[q] = __byte_perm(lo, hi, 0x5410);
          }
          uint8_t* dst = p.colwise_out + static_cast<int64_t>(c0 + 4 * cg + cc) * N + i0;
          st_words<8>(dst, o);
        }
      }
    } else {
      // ---- column-block scales, then columnwise codes
      float* colmax = reinterpret_cast<float*>(smem);
      float* colmul = colmax + kStripeWarps * hc;
      for (int c = tid; c < hc; c += 256) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kStripeWarps; ++w) a = fmax_nan(a, colmax[w * hc + c]);
        const uint32_t code = e8m0_code(a);
        colmul[c] = e8m0_mult(code);
        p.mx_colwise_scale[s * H + c0 + c] = static_cast<uint8_t>(code);
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < NVS; ++j) {
        const int v = j * 32 + lane;
        if (v < nvs) {
          const int col = c0 + v * VEC;
          float g[VEC], b[VEC], m[VEC];
          ld_weights<VEC>(p.gamma, p.w_dt, col, g);
          if (ln) {
            ld_weights<VEC>(p.beta, p.w_dt, col, b);
          } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) b[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            g[e] += gadd;
            m[e] = colmul[v * VEC + e];
          }
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            float f[VEC], z[VEC];
            unpack<Tin, VEC>(xw[r][j], f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) z[e] = (f[e] - mean[r]) * rs[r] * g[e] + b[e];
            uint32_t w[VEC / 4];
            e4m3_pack_mul<VEC>(z, m, w);
            st_words<VEC / 4>(p.colwise_out + (i0 + r0 + r) * H + col, w);
          }
        }
      }
    }
    // The next stripe's smem writes happen after its cluster barrier, which
    // every thread of this CTA reaches only after finishing the reads above.
  }
  // Keep this CTA's shared memory alive until every peer has read its stats.
  cluster_sync();

  if constexpr (QM == Q_DELAYED) {
    block_amax_commit(amax_t, red, p.amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      const float inv = 1.f / qscale;
      if (p.scale_inv) *p.scale_inv = inv;
      if (p.colwise_scale_inv) *p.colwise_scale_inv = inv;
    }
  }
}

}  // namespace gbn
