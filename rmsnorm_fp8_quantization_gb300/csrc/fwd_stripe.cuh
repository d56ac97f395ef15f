// Forward kernel for the columnwise FP8 layouts (delayed scaling with a
// transposed [hidden, rows] copy, MXFP8 with 32x1 column blocks), optionally
// together with the rowwise outputs.
//
// Operation: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Description ("rowwise and optional columnwise (2x2x layout) FP8 output
// tensors with scale/amax/scale_inv") and I/O Contract.
//
// A columnwise output needs 32 finished rows before any column can be
// written, and 32 rows of a long row do not fit one SM.  A thread-block
// cluster of C CTAs therefore takes one 32-row stripe: CTA `rank` owns
// columns [rank*hc, (rank+1)*hc).
//   1. The CTA's 32 x hc slice arrives in shared memory by bulk copies (with
//      two stages, the next slice is copied while this one is processed; with
//      one, the other CTAs on the SM keep it busy meanwhile).  No L2
//      prefetch of the next slice: measured, its lines were often evicted
//      before use and read twice.
//   2. One warp per four rows reduces the slice's per-row mean and M2; the 32
//      pairs are pushed to every CTA of the cluster with `st.async`, whose
//      bytes complete a transaction count on the receiver's mbarrier.  Every
//      CTA merges the C partials of a row in rank order (identical results in
//      all CTAs); no cluster-wide barrier per stripe.
//   3. Delayed scaling: a thread item is 4 adjacent columns x all 32 rows,
//      computed in packed fp32 pairs.  Rowwise codes go to HBM as 4-byte
//      words (a warp writes 128 contiguous bytes of a row); the codes are
//      transposed in registers (4x4 byte transposes) and each column's 32
//      codes leave as one 32-byte store, a whole sector.  MXFP8: a warp owns
//      a band of 16 16-byte vectors over the 32 rows, a lane one vector of
//      every other row.  A pass writes the rowwise codes (a 1x32 block is
//      32/VEC adjacent lanes) and keeps each column's amax; a second pass,
//      after one shuffle per column with the lane holding the other rows,
//      writes the colwise codes.
//   Slice rows sit 16 bytes apart beyond their length in shared memory, so
//   that the lanes of a tile, reading 8 rows at once, hit distinct banks.
// x is read from HBM once.
#pragma once

#include <type_traits>

#include "ring.cuh"

namespace gbn {

constexpr int kStripeWarps = kStripeThreads / 32;
constexpr int kRowsPerWarp = kStripeRows / kStripeWarps;  // 4
constexpr int kMaxCluster = 16;

// Four consecutive elements of a shared-memory row as two fp32 pairs.
template <typename Tin>
__device__ __forceinline__ void lds4_pairs(const Tin* p, uint64_t* pr) {
  if constexpr (sizeof(Tin) == 4) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    widen_pairs<Tin, 4>(w, pr);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {u.x, u.y};
    widen_pairs<Tin, 4>(w, pr);
  }
}

// In-register 4x4 byte transpose: out[c] byte r = in[r] byte c.
__device__ __forceinline__ void transpose4x4(const uint32_t* in, uint32_t* out) {
  const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140), t1 = __byte_perm(in[0], in[1], 0x7362);
  const uint32_t t2 = __byte_perm(in[2], in[3], 0x5140), t3 = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// x - mu (LayerNorm, neg_mu = -mu) or x (RMSNorm) of a 16-byte vector as
// VEC/2 fp32 pairs.
template <typename Tin, bool LN>
__device__ __forceinline__ void centered_pairs(const uint4& u, float neg_mu, uint64_t* z) {
  constexpr int VEC = 16 / (int)sizeof(Tin);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  widen_pairs<Tin, VEC>(w, z);
  if constexpr (LN) {
    const uint64_t c2 = p2(neg_mu, neg_mu);
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) z[i] = add2(z[i], c2);
  }
}

template <typename Tin, int QM, bool LN>
__global__ void __launch_bounds__(kStripeThreads, 3)
    fwd_stripe_kernel(const FwdParams p, const int hc, const int stages) {
  pdl_begin();
  constexpr int VEC = 16 / (int)sizeof(Tin);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[2];                          // x slice landed
  __shared__ uint64_t statbar[2];                       // all C stat pushes landed
  __shared__ float2 mystat[kStripeRows];
  // per row: delayed scaling (mean, rsigma); MXFP8 (-mean, -mean, rsigma, rsigma),
  // whose halves load as ready fp32 pairs
  using RowStat = typename std::conditional<QM == Q_MXFP8, float4, float2>::type;
  __shared__ RowStat rstat[kStripeRows];
  __shared__ float red[32];
  __shared__ int s_abort;
  __shared__ long long s_kfail;  // first stripe whose copy never landed

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int H = p.hidden;
  const int c0 = static_cast<int>(rank) * hc;
  const int nvs = hc / VEC;
  const int G = hc / 4;  // groups of 4 adjacent columns
  const int64_t N = p.rows;
  const int64_t nstripes = N / kStripeRows;
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t count = cid < nstripes ? (nstripes - 1 - cid) / ncl + 1 : 0;
  const float inv_h = 1.f / static_cast<float>(H), fhc = static_cast<float>(hc);
  const uint32_t row_bytes = static_cast<uint32_t>(hc) * sizeof(Tin);
  const uint32_t rstride = row_bytes + 16;  // shared-memory bytes between slice rows
  const uint32_t slice = kStripeRows * rstride;
  const Tin* x = reinterpret_cast<const Tin*>(p.x);
  uint8_t* xbuf = smem;
  // statistics pushed by the cluster's CTAs: [stripe parity][sender][row]
  float2* rbuf = reinterpret_cast<float2*>(smem + stages * slice);
  float* wg = reinterpret_cast<float*>(rbuf + 2 * C * kStripeRows);  // g' [hc]
  float* wb = wg + hc;                                              // beta [hc] (LayerNorm)
  auto rb_at = [&](int par, uint32_t sender, int row) -> float2& {
    return rbuf[(par * C + sender) * kStripeRows + row];
  };
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  float amax_t = 0.f;

  auto stripe_of = [&](int64_t k) { return cid + k * ncl; };
  auto issue = [&](int b, int64_t k) {
    const int64_t i0 = stripe_of(k) * kStripeRows;
    mbar_arrive_expect_tx(&full[b], kStripeRows * row_bytes);
    for (int r = 0; r < kStripeRows; ++r)
      bulk_g2s(xbuf + b * slice + r * rstride, x + (i0 + r) * H + c0, row_bytes, &full[b]);
  };
  // Bounded waits by one thread, the rest of the CTA blocked on the barrier
  // that follows (no spinning warps).  After the first timeout every later
  // wait gives up at once and no further copies are issued (the outputs are
  // then invalid and the device error flag is set).
  auto wait = [&](uint64_t* bar, uint32_t parity, int64_t k) {
    if (tid == 0 && !s_abort && !mbar_wait(bar, parity)) {
      s_kfail = k;
      s_abort = 1;
    }
    __syncthreads();
  };

  int64_t issued = 0;
  if (tid == 0) {
    s_abort = 0;
    s_kfail = -1;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&statbar[i], 1);
    }
    fence_mbar_init();
    for (; issued < stages && issued < count; ++issued) issue(static_cast<int>(issued), issued);
  }
  {
    const float gadd = p.zcg ? 1.f : 0.f;
    for (int c = tid; c < hc; c += kStripeThreads) {
      wg[c] = ld_weight_scalar(p.gamma, p.w_dt, c0 + c) + gadd;
      if constexpr (LN) wb[c] = ld_weight_scalar(p.beta, p.w_dt, c0 + c);
    }
  }
  // Peers push statistics into this CTA's mbarriers: they must be initialized
  // cluster-wide before the first push.
  cluster_sync();

  for (int64_t k = 0; k < count; ++k) {
    const int64_t i0 = stripe_of(k) * kStripeRows;
    const int b = stages == 2 ? static_cast<int>(k & 1) : 0;
    const uint32_t par = static_cast<uint32_t>(stages == 2 ? (k >> 1) & 1 : k & 1);
    const int sb = static_cast<int>(k & 1);  // stat buffer
    if (tid == 0) mbar_arrive_expect_tx(&statbar[sb], C * kStripeRows * sizeof(float2));
    wait(&full[b], par, k);
    const uint8_t* xsb = xbuf + b * slice;
    const Tin* xs = reinterpret_cast<const Tin*>(xsb);
    const int xrow = static_cast<int>(rstride / sizeof(Tin));  // elements between slice rows

    // ---- 1. slice statistics, warp w owns rows 4w .. 4w+3; the four rows
    // are walked together (independent loads and shuffles in flight).
    {
      constexpr int NP = VEC / 2;
      constexpr int RW4 = kRowsPerWarp;
      const uint8_t* xr = xsb + warp * RW4 * rstride;
      float m[RW4];
#pragma unroll
      for (int rr = 0; rr < RW4; ++rr) m[rr] = 0.f;
      if constexpr (LN) {
        uint64_t a[RW4];
#pragma unroll
        for (int rr = 0; rr < RW4; ++rr) a[rr] = 0ull;
        for (int v = lane; v < nvs; v += 32) {
#pragma unroll
          for (int rr = 0; rr < RW4; ++rr) {
            const uint4 u = reinterpret_cast<const uint4*>(xr + rr * rstride)[v];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint64_t pr[NP];
            widen_pairs<Tin, VEC>(w, pr);
#pragma unroll
            for (int i = 0; i < NP; ++i) a[rr] = add2(a[rr], pr[i]);
          }
        }
#pragma unroll
        for (int rr = 0; rr < RW4; ++rr) {
          const float2 af = u2(a[rr]);
          m[rr] = warp_sum(af.x + af.y) / fhc;
        }
      }
      uint64_t q2[RW4];
#pragma unroll
      for (int rr = 0; rr < RW4; ++rr) q2[rr] = 0ull;
      // (unrolled by four: delayed scaling on 32768 x 8192 bf16 191.5 -> 189.2 us)
#pragma unroll 4
      for (int v = lane; v < nvs; v += 32) {
#pragma unroll
        for (int rr = 0; rr < RW4; ++rr) {
          const uint4 u = reinterpret_cast<const uint4*>(xr + rr * rstride)[v];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
          uint64_t pr[NP];
          widen_pairs<Tin, VEC>(w, pr);
          const uint64_t m2 = p2(m[rr], m[rr]);
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            const uint64_t d = LN ? sub2(pr[i], m2) : pr[i];
            q2[rr] = fma2(d, d, q2[rr]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < RW4; ++rr) {
        const float2 qf = u2(q2[rr]);
        const float q = warp_sum(qf.x + qf.y);
        if (lane == 0) mystat[warp * RW4 + rr] = make_float2(m[rr], q);
      }
    }
    __syncthreads();
    if (warp == 0) {
      const float2 mine = mystat[lane];
#pragma unroll
      for (uint32_t c = 0; c < kMaxCluster; ++c)
        if (c < C) push_stat(&rb_at(sb, rank, lane), &statbar[sb], c, mine);
    }
    wait(&statbar[sb], static_cast<uint32_t>((k >> 1) & 1), -1);

    // ---- 2. merge the C partials of each row in rank order
    if (warp == 0) {
      const int r = lane;
      float mu = 0.f, qsum = 0.f;
      // (unrolled to the largest cluster, entries past C skipped)
      if constexpr (LN) {
        float msum = 0.f;
#pragma unroll
        for (uint32_t c = 0; c < kMaxCluster; ++c)
          if (c < C) msum += rb_at(sb, c, r).x;
        mu = msum / static_cast<float>(C);
      }
#pragma unroll
      for (uint32_t c = 0; c < kMaxCluster; ++c) {
        if (c < C) {
          const float2 v = rb_at(sb, c, r);
          const float d = v.x - mu;
          qsum += LN ? fmaf(fhc * d, d, v.y) : v.y;
        }
      }
      const float rs = rsqrtf(fmaf(qsum, inv_h, p.eps));
      if constexpr (QM == Q_MXFP8)
        rstat[r] = make_float4(-mu, -mu, rs, rs);
      else
        rstat[r] = make_float2(mu, rs);
      if (rank == 0) {
        if (LN && p.mu) p.mu[i0 + r] = mu;
        if (p.rsigma) p.rsigma[i0 + r] = rs;
      }
    }
    __syncthreads();

    // ---- 3, MXFP8: a warp owns a band of 16 vectors (16*VEC columns) over the
    // 32 rows; lane = (vector vl, row parity rp) walks rows rp, rp+2, ...
    // A 1x32 row block is 32/VEC adjacent lanes (shuffles); a 32x1 column
    // block is one lane's 16 rows plus its partner lane^16's.  Pass 1 writes
    // the rowwise codes and keeps the column amax; pass 2 the colwise codes.
    // Each step takes two rows (r, r + 2) for independent work in flight.
    if constexpr (QM == Q_MXFP8) {
      auto bands = [&](auto rw_tag, auto swz_tag) {
        constexpr bool RW = decltype(rw_tag)::value, SWZ = decltype(swz_tag)::value;
        constexpr int NPV = VEC / 2;
        constexpr int TPB = 32 / VEC;
        const int vl = lane & 15, rp = lane >> 4;
        const int nbands = nvs / 16;
        const int64_t sc_stride = H / 32;
        // row steps unrolled: RMSNorm four in pass 1, all eight in pass 2
        // (measured on 16384 x 5120 bf16: 77.8 us with two and two, 75.7 with
        // four and four, 73.9 with four and eight); LayerNorm two (more spill)
        constexpr int kBandUnroll = LN ? 2 : 4;
        constexpr int kColUnroll = LN ? 2 : 8;
        for (int band = warp; band < nbands; band += kStripeWarps) {
          const int v = band * 16 + vl;
          const int col = c0 + v * VEC;
          uint64_t gw[NPV], bw[NPV];
#pragma unroll
          for (int h = 0; h < NPV / 2; ++h) {
            const float4 g = reinterpret_cast<const float4*>(wg + v * VEC)[h];
            gw[2 * h] = p2(g.x, g.y);
            gw[2 * h + 1] = p2(g.z, g.w);
            if constexpr (LN) {
              const float4 bv = reinterpret_cast<const float4*>(wb + v * VEC)[h];
              bw[2 * h] = p2(bv.x, bv.y);
              bw[2 * h + 1] = p2(bv.z, bv.w);
            } else {
              bw[2 * h] = bw[2 * h + 1] = 0ull;
            }
          }
          const uint4* xv = reinterpret_cast<const uint4*>(xsb + rp * rstride) + v;
          const int xstep = 2 * static_cast<int>(rstride / 16);  // vectors between rows r and r + 2
          // z of the lane's vector in row r, as NPV pairs, with weights g, b
          auto zvec = [&](int r, const uint64_t* g, const uint64_t* bb, uint64_t* z) {
            float neg_mu = 0.f;
            uint64_t r2;
            if constexpr (LN) {
              const float4 st = rstat[r];
              neg_mu = st.x;
              r2 = p2(st.z, st.w);
            } else {
              const float2 st = reinterpret_cast<const float2*>(&rstat[r])[1];
              r2 = p2(st.x, st.y);
            }
            centered_pairs<Tin, LN>(xv[(r >> 1) * xstep], neg_mu, z);
#pragma unroll
            for (int i = 0; i < NPV; ++i) {
              const uint64_t t = mul2(z[i], r2);
              z[i] = LN ? fma2(t, g[i], bb[i]) : mul2(t, g[i]);
            }
          };
          float cm[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) cm[e] = 0.f;
          uint8_t* orow = RW ? reinterpret_cast<uint8_t*>(p.out) + (i0 + rp) * H + col : nullptr;
          int64_t srow = RW && !SWZ ? (i0 + rp) * sc_stride + col / 32 : 0;
          const bool sc_lane = (v & (TPB - 1)) == 0;
#pragma unroll kBandUnroll
          for (int r = rp; r < kStripeRows; r += 4) {
            uint64_t za[NPV], zb[NPV];
            zvec(r, gw, bw, za);
            zvec(r + 2, gw, bw, zb);
            float aa = 0.f, ab = 0.f;
#pragma unroll
            for (int i = 0; i < NPV; ++i) {
              const float2 fa = u2(za[i]), fb = u2(zb[i]);
              cm[2 * i] = fmax_nan(cm[2 * i], fmax_nan(fabsf(fa.x), fabsf(fb.x)));
              cm[2 * i + 1] = fmax_nan(cm[2 * i + 1], fmax_nan(fabsf(fa.y), fabsf(fb.y)));
              aa = fmax_nan(aa, fmax_nan(fabsf(fa.x), fabsf(fa.y)));
              ab = fmax_nan(ab, fmax_nan(fabsf(fb.x), fabsf(fb.y)));
            }
            if constexpr (RW) {
#pragma unroll
              for (int o = 1; o < TPB; o <<= 1) {
                aa = fmax_nan(aa, __shfl_xor_sync(0xFFFFFFFFu, aa, o));
                ab = fmax_nan(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, o));
              }
              uint32_t ka, kb;
              float ma, mb;
              e8m0_scale(aa, ka, ma);
              e8m0_scale(ab, kb, mb);
              const uint64_t sa = p2(ma, ma), sb = p2(mb, mb);
              uint32_t qa[VEC / 4], qb[VEC / 4];
#pragma unroll
              for (int i = 0; i < VEC / 4; ++i) {
                qa[i] = e4m3x4_pairs(za[2 * i], za[2 * i + 1], sa);
                qb[i] = e4m3x4_pairs(zb[2 * i], zb[2 * i + 1], sb);
              }
              st_words<VEC / 4>(orow, qa);
              st_words<VEC / 4>(orow + 2 * H, qb);
              if (sc_lane) {
                if constexpr (SWZ) {
                  p.mx_scale[mx_row_scale_at(p, i0 + r, col / 32)] = static_cast<uint8_t>(ka);
                  p.mx_scale[mx_row_scale_at(p, i0 + r + 2, col / 32)] = static_cast<uint8_t>(kb);
                } else {
                  p.mx_scale[srow] = static_cast<uint8_t>(ka);
                  p.mx_scale[srow + 2 * sc_stride] = static_cast<uint8_t>(kb);
                }
              }
              orow += 4 * H;
              srow += 4 * sc_stride;
            }
          }
          if (p.write_colwise) {
            uint32_t cw[VEC / 4];
            uint64_t gm[NPV], bm[NPV];
#pragma unroll
            for (int i = 0; i < NPV; ++i) {
              const float c0a = fmax_nan(cm[2 * i], __shfl_xor_sync(0xFFFFFFFFu, cm[2 * i], 16));
              const float c1a =
                  fmax_nan(cm[2 * i + 1], __shfl_xor_sync(0xFFFFFFFFu, cm[2 * i + 1], 16));
              uint32_t k0, k1;
              float m0, m1;
              e8m0_scale(c0a, k0, m0);
              e8m0_scale(c1a, k1, m1);
              if ((i & 1) == 0) cw[i / 2] = 0u;
              cw[i / 2] |= (k0 | (k1 << 8)) << (16 * (i & 1));
              // A power-of-two multiplier commutes exactly with the roundings
              // of (x - mu) * rs * g' + beta (while g' and beta times it stay
              // normal), so it is applied to g' and beta once.
              const uint64_t m01 = p2(m0, m1);
              gm[i] = mul2(gw[i], m01);
              bm[i] = mul2(bw[i], m01);
            }
            if (rp == 0) {
              if constexpr (SWZ) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                  p.mx_colwise_scale[mx_col_scale_at(p, stripe_of(k), col + e)] =
                      static_cast<uint8_t>(cw[e / 4] >> (8 * (e & 3)));
              } else {
                st_words<VEC / 4>(p.mx_colwise_scale + stripe_of(k) * H + col, cw);
              }
            }
            uint8_t* crow = p.colwise_out + (i0 + rp) * H + col;
#pragma unroll kColUnroll
            for (int r = rp; r < kStripeRows; r += 4) {
              uint64_t za[NPV], zb[NPV];
              zvec(r, gm, bm, za);
              zvec(r + 2, gm, bm, zb);
              uint32_t qa[VEC / 4], qb[VEC / 4];
#pragma unroll
              for (int i = 0; i < VEC / 4; ++i) {
                const float2 fa = u2(za[2 * i]), fb = u2(za[2 * i + 1]);
                qa[i] = e4m3x2(fa.x, fa.y) | (e4m3x2(fb.x, fb.y) << 16);
                const float2 ga = u2(zb[2 * i]), gb = u2(zb[2 * i + 1]);
                qb[i] = e4m3x2(ga.x, ga.y) | (e4m3x2(gb.x, gb.y) << 16);
              }
              st_words<VEC / 4>(crow, qa);
              st_words<VEC / 4>(crow + 2 * H, qb);
              crow += 4 * H;
            }
          }
        }
      };
      if (p.write_rowwise) {
        if (p.mx_swizzle)
          bands(std::true_type{}, std::true_type{});
        else
          bands(std::true_type{}, std::false_type{});
      } else {
        if (p.mx_swizzle)
          bands(std::false_type{}, std::true_type{});
        else
          bands(std::false_type{}, std::false_type{});
      }
    }

    // ---- 3, delayed scaling: items of 4 columns x 32 rows
    if constexpr (QM == Q_DELAYED)
    for (int cg = tid; cg < G; cg += kStripeThreads) {
      const float4 g4 = reinterpret_cast<const float4*>(wg)[cg];
      const uint64_t g01 = p2(g4.x, g4.y), g23 = p2(g4.z, g4.w);
      uint64_t b01 = 0ull, b23 = 0ull;
      if constexpr (LN) {
        const float4 b4 = reinterpret_cast<const float4*>(wb)[cg];
        b01 = p2(b4.x, b4.y);
        b23 = p2(b4.z, b4.w);
      }
      const int col = c0 + 4 * cg;
      const Tin* xcol = xs + 4 * cg;
      // z of row r as two pairs, with weights (ga, gb) and betas (ba, bb)
      auto zrow_w = [&](int r, uint64_t ga, uint64_t gb, uint64_t ba, uint64_t bb, uint64_t& z01,
                        uint64_t& z23) {
        const float2 st = rstat[r];
        const uint64_t m2 = p2(st.x, st.x), r2 = p2(st.y, st.y);
        uint64_t xp[2];
        lds4_pairs<Tin>(xcol + r * xrow, xp);
        const uint64_t t01 = mul2(LN ? sub2(xp[0], m2) : xp[0], r2);
        const uint64_t t23 = mul2(LN ? sub2(xp[1], m2) : xp[1], r2);
        z01 = LN ? fma2(t01, ga, ba) : mul2(t01, ga);
        z23 = LN ? fma2(t23, gb, bb) : mul2(t23, gb);
      };
      auto zrow = [&](int r, uint64_t& z01, uint64_t& z23) {
        zrow_w(r, g01, g23, b01, b23, z01, z23);
      };
      auto absmax4 = [](uint64_t a, uint64_t b) {
        const float2 x = u2(a), y = u2(b);
        return fmax_nan(fmax_nan(fabsf(x.x), fabsf(x.y)), fmax_nan(fabsf(y.x), fabsf(y.y)));
      };
      if constexpr (QM == Q_DELAYED) {
        uint8_t* orow = p.write_rowwise ? reinterpret_cast<uint8_t*>(p.out) + i0 * H + col : nullptr;
        const uint64_t s2 = p2(qscale, qscale);
        uint32_t w[kStripeRows];
#pragma unroll
        for (int r = 0; r < kStripeRows; ++r) {
          uint64_t z01, z23;
          zrow(r, z01, z23);
          amax_t = fmax_nan(amax_t, absmax4(z01, z23));
          w[r] = e4m3x4_pairs(z01, z23, s2);
          if (p.write_rowwise) *reinterpret_cast<uint32_t*>(orow + static_cast<int64_t>(r) * H) = w[r];
        }
        if (p.write_colwise) {
          uint32_t o[4][8];  // [column][rows 4m..4m+3]
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            uint32_t t[4];
            transpose4x4(&w[4 * m], t);
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c][m] = t[c];
          }
          // A column's 32 codes are one 32-byte sector of a 128-byte line
          // whose other sectors come from the three neighbouring stripes,
          // written by other clusters at about the same time: kept in L2
          // evict-last, a line is more often complete before it is written
          // back (measured: 32768 x 8192 bf16 195.5 -> 191.4 us; the same
          // hint on the rowwise codes or evict-first on x made it slower).
          const uint64_t pol = l2_evict_last_policy();
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_global_v8_policy(p.colwise_out + static_cast<int64_t>(col + c) * N + i0, o[c], pol);
        }
      }
    }
    __syncthreads();
    // Every thread is done with this stage and rstat.
    if (tid == 0 && issued < count && !s_abort) {
      issue(stages == 2 ? b : 0, issued);
      ++issued;
    }
  }

  if (tid == 0 && s_abort) {
    atomicOr(&g_gbn_device_error, 1u);
    // Let copies still in flight land before this CTA's shared memory goes.
    for (int64_t j = s_kfail < 0 ? issued : s_kfail; j < issued; ++j)
      mbar_wait(&full[stages == 2 ? static_cast<int>(j & 1) : 0],
                static_cast<uint32_t>(stages == 2 ? (j >> 1) & 1 : j & 1));
  }
  // No CTA leaves while a peer of its cluster may still push into it.
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
