// Generic forward kernel: any size, any alignment, every layout.  The fast
// paths are the ring kernels (ring.cuh) and the stripe kernel
// (fwd_stripe.cuh).
//
// Operation: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Description and I/O Contract -- per row, mean (LayerNorm only) and rsigma,
// z = (x - mu) * rsigma * g' (+ beta), stored unquantized, or as E4M3 with
// delayed per-tensor scaling (scale, updated amax, scale_inv), or as MXFP8
// with one E8M0 scale per 32 elements.
#pragma once

#include "gbn_device.cuh"

namespace gbn {

// z of element (row, j) for the generic path.
template <typename Tin>
__device__ __forceinline__ float z_at(const FwdParams& p, int64_t row, int j, float mean, float rs,
                                      float gadd, bool ln) {
  const float x = ld_scalar(reinterpret_cast<const Tin*>(p.x), row * p.hidden + j);
  const float g = ld_weight_scalar(p.gamma, p.w_dt, j) + gadd;
  const float t = (x - mean) * rs;
  return ln ? fmaf(t, g, ld_weight_scalar(p.beta, p.w_dt, j)) : t * g;
}

// Generic forward: any hidden size, any alignment, every layout.  One CTA of
// 256 threads per 32-row stripe (persistent); statistics by one warp per row,
// then outputs re-read x through L1/L2.  Correct for every shape the
// interface accepts; the vectorized kernels cover the fast cases.
template <typename Tin, int QM>
__global__ void __launch_bounds__(256) fwd_generic_kernel(const FwdParams p) {
  pdl_begin();
  __shared__ float s_mean[32], s_rs[32], red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.hidden;
  const bool ln = (p.norm == 0);
  const float gadd = p.zcg ? 1.f : 0.f;
  const int64_t N = p.rows;
  const int64_t nstripes = (N + 31) / 32;
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  float amax_t = 0.f;
  const Tin* x = reinterpret_cast<const Tin*>(p.x);

  for (int64_t s = blockIdx.x; s < nstripes; s += gridDim.x) {
    const int64_t i0 = s * 32;
    const int nr = static_cast<int>(N - i0 < 32 ? N - i0 : 32);
    for (int r = warp; r < nr; r += 8) {
      const int64_t row = i0 + r;
      float mean = 0.f;
      if (ln) {
        float sum = 0.f;
        for (int j = lane; j < H; j += 32) sum += ld_scalar(x, row * H + j);
        mean = warp_sum(sum) / static_cast<float>(H);
      }
      float ss = 0.f;
      for (int j = lane; j < H; j += 32) {
        const float d = ld_scalar(x, row * H + j) - mean;
        ss = fmaf(d, d, ss);
      }
      const float rs = 1.f / sqrtf(warp_sum(ss) / static_cast<float>(H) + p.eps);
      if (lane == 0) {
        s_mean[r] = mean;
        s_rs[r] = rs;
        if (ln && p.mu) p.mu[row] = mean;
        if (p.rsigma) p.rsigma[row] = rs;
      }
    }
    __syncthreads();

    if (p.write_rowwise) {
      if constexpr (QM == Q_MXFP8) {
        const int nb = H / 32;
        for (int idx = tid; idx < nr * nb; idx += 256) {
          const int r = idx / nb, blk = idx % nb;
          const int64_t row = i0 + r;
          float a = 0.f;
          for (int e = 0; e < 32; ++e)
            a = fmax_nan(a, fabsf(z_at<Tin>(p, row, blk * 32 + e, s_mean[r], s_rs[r], gadd, ln)));
          uint32_t c;
          float m;
          e8m0_scale(a, c, m);
          uint8_t* o = reinterpret_cast<uint8_t*>(p.out) + row * H + blk * 32;
          for (int e = 0; e < 32; ++e)
            o[e] = e4m3(z_at<Tin>(p, row, blk * 32 + e, s_mean[r], s_rs[r], gadd, ln) * m);
          p.mx_scale[mx_row_scale_at(p, row, blk)] = static_cast<uint8_t>(c);
        }
      } else {
        for (int64_t idx = tid; idx < static_cast<int64_t>(nr) * H; idx += 256) {
          const int r = static_cast<int>(idx / H), j = static_cast<int>(idx % H);
          const int64_t row = i0 + r;
          const float z = z_at<Tin>(p, row, j, s_mean[r], s_rs[r], gadd, ln);
          if constexpr (QM == Q_NONE) {
            st_scalar(reinterpret_cast<Tin*>(p.out), row * H + j, z);
          } else {
            amax_t = fmax_nan(amax_t, fabsf(z));
            reinterpret_cast<uint8_t*>(p.out)[row * H + j] = e4m3(z * qscale);
          }
        }
      }
    }
    if constexpr (QM == Q_DELAYED) {
      if (p.write_colwise) {
        // colwise_out [H, N]: consecutive threads take consecutive rows of one column.
        for (int64_t idx = tid; idx < static_cast<int64_t>(nr) * H; idx += 256) {
          const int j = static_cast<int>(idx / nr), r = static_cast<int>(idx % nr);
          const float z = z_at<Tin>(p, i0 + r, j, s_mean[r], s_rs[r], gadd, ln);
          if (!p.write_rowwise) amax_t = fmax_nan(amax_t, fabsf(z));
          p.colwise_out[static_cast<int64_t>(j) * N + i0 + r] = e4m3(z * qscale);
        }
      }
    }
    if constexpr (QM == Q_MXFP8) {
      if (p.write_colwise) {  // nr == 32 (rows % 32 == 0 is validated)
        for (int j = tid; j < H; j += 256) {
          float a = 0.f;
          for (int r = 0; r < 32; ++r)
            a = fmax_nan(a, fabsf(z_at<Tin>(p, i0 + r, j, s_mean[r], s_rs[r], gadd, ln)));
          uint32_t c;
          float m;
          e8m0_scale(a, c, m);
          for (int r = 0; r < 32; ++r)
            p.colwise_out[(i0 + r) * H + j] =
                e4m3(z_at<Tin>(p, i0 + r, j, s_mean[r], s_rs[r], gadd, ln) * m);
          p.mx_colwise_scale[mx_col_scale_at(p, s, j)] = static_cast<uint8_t>(c);
        }
      }
    }
    __syncthreads();
  }

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
