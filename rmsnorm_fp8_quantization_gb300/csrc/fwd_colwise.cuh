// Columnwise FP8 output of rows too long for a stripe slice in shared memory
// (the stripe kernel's limit: 32 rows x 2048 two-byte columns per CTA, 16
// CTAs per cluster).  The row statistics come from the long-row forward that
// ran just before (its mu / rsigma outputs, or scratch), which also wrote the
// rowwise output and, for delayed scaling, the amax; this kernel reads x again
// and writes the columnwise codes (and the MXFP8 32x1 block scales).
//
// Operation: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Description ("rowwise and optional columnwise (2x2x layout) FP8 output
// tensors") and I/O Contract.
//
// A tile is 32 rows x 512 columns; thread t owns columns c, c + 1 (c = tile
// column + 2t), loads its bf16/f16 pair (or fp32 pair) of every row -- a warp
// reads 128 (256) contiguous bytes of a row -- and keeps the 32 z pairs in
// registers.  z is evaluated in the same fp32 order as the row kernels:
// ((x - mu) * rsigma) * g' (+ beta).  Delayed scaling: a column's 32 codes
// leave as one 32-byte store of the transposed output; MXFP8: the column
// block's amax gives its E8M0 scale, and each row gets a 2-byte store.
#pragma once

#include "gbn_device.cuh"

namespace gbn {

template <typename Tin, int QM, bool LN>
__global__ void __launch_bounds__(kColTileThreads)
    fwd_colwise_kernel(const FwdParams p, const float* mu, const float* rsigma) {
  static_assert(QM == Q_DELAYED || QM == Q_MXFP8, "columnwise output is FP8");
  pdl_begin();
  __shared__ float2 rstat[32];  // (mu, rsigma) of the tile's rows
  const int tid = threadIdx.x;
  const int H = p.hidden;
  const int64_t N = p.rows;
  const int tiles_per_stripe = (H + kColTileCols - 1) / kColTileCols;
  const int64_t ntiles = (N / 32) * tiles_per_stripe;
  const Tin* x = reinterpret_cast<const Tin*>(p.x);
  const float gadd = p.zcg ? 1.f : 0.f;
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  const uint64_t q2 = p2(qscale, qscale);
  const uint64_t pol = l2_evict_last_policy();

  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t s = t / tiles_per_stripe;
    const int c = static_cast<int>(t - s * tiles_per_stripe) * kColTileCols + 2 * tid;
    const int64_t i0 = s * 32;
    __syncthreads();  // the previous tile's statistics are read
    if (tid < 32) rstat[tid] = make_float2(LN ? mu[i0 + tid] : 0.f, rsigma[i0 + tid]);
    __syncthreads();
    if (c >= H) continue;  // H is even, so c + 1 < H as well
    const uint64_t g2 = p2(ld_weight_scalar(p.gamma, p.w_dt, c) + gadd,
                           ld_weight_scalar(p.gamma, p.w_dt, c + 1) + gadd);
    uint64_t b2 = 0ull;
    if constexpr (LN)
      b2 = p2(ld_weight_scalar(p.beta, p.w_dt, c), ld_weight_scalar(p.beta, p.w_dt, c + 1));
    const Tin* xr = x + i0 * H + c;
    uint64_t z[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      uint64_t xp;
      if constexpr (sizeof(Tin) == 4) {
        const float2 f = *reinterpret_cast<const float2*>(xr + static_cast<int64_t>(r) * H);
        xp = p2(f.x, f.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(xr + static_cast<int64_t>(r) * H);
        widen_pairs<Tin, 2>(&w, &xp);
      }
      const float2 st = rstat[r];
      const uint64_t tt = mul2(LN ? sub2(xp, p2(st.x, st.x)) : xp, p2(st.y, st.y));
      z[r] = LN ? fma2(tt, g2, b2) : mul2(tt, g2);
    }
    if constexpr (QM == Q_DELAYED) {
      // codes of rows 4m..4m+3: column c in the low bytes, c + 1 in the high
      uint32_t o0[8], o1[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = u2(mul2(z[4 * m + j], q2));
          h[j] = e4m3x2(f.x, f.y);
        }
        const uint32_t a = h[0] | (h[1] << 16), b = h[2] | (h[3] << 16);
        o0[m] = __byte_perm(a, b, 0x6420);
        o1[m] = __byte_perm(a, b, 0x7531);
      }
      st_global_v8_policy(p.colwise_out + static_cast<int64_t>(c) * N + i0, o0, pol);
      st_global_v8_policy(p.colwise_out + static_cast<int64_t>(c + 1) * N + i0, o1, pol);
    } else {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float2 f = u2(z[r]);
        a0 = fmax_nan(a0, fabsf(f.x));
        a1 = fmax_nan(a1, fabsf(f.y));
      }
      uint32_t k0, k1;
      float m0, m1;
      e8m0_scale(a0, k0, m0);
      e8m0_scale(a1, k1, m1);
      const uint64_t m2 = p2(m0, m1);
      uint8_t* o = p.colwise_out + i0 * H + c;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float2 f = u2(mul2(z[r], m2));
        *reinterpret_cast<uint16_t*>(o + static_cast<int64_t>(r) * H) =
            static_cast<uint16_t>(e4m3x2(f.x, f.y));
      }
      p.mx_colwise_scale[mx_col_scale_at(p, s, c)] = static_cast<uint8_t>(k0);
      p.mx_colwise_scale[mx_col_scale_at(p, s, c + 1)] = static_cast<uint8_t>(k1);
    }
  }
}

}  // namespace gbn
