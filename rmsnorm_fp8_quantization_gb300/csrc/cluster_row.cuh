// Long rows: a row too long for one CTA's ring is split over a thread-block
// cluster.  CTA `rank` of a cluster of C owns columns [rank*hc, (rank+1)*hc)
// of every row the cluster takes (rows cid, cid + nclusters, ...); its slice
// of a row arrives in its own bulk-copy ring, its weights stay in registers,
// and the row statistics are combined across the cluster: each CTA pushes
// its slice's statistics (forward: mean and M2, or the sum of squares;
// backward: sum dy and sum dy*xhat) into every CTA's shared memory with
// `st.async`, whose bytes complete a transaction count on the receiver's
// mbarrier, and every CTA merges the C entries the same way (forward: a tree
// of xor shuffles over 8 lanes; backward: all 8 entries in rank order, zeros
// past C) -- identical bits in every CTA, no cluster barrier per row.  For
// the columnwise FP8 layouts of such rows the forward runs first and writes
// the statistics, the amax and any rowwise codes (none for a columnwise-only
// layout); the columnwise tile kernel (fwd_colwise.cuh) follows.
//
// Operations: "Implementation:NVIDIA TransformerEngine JAX XLA
// Normalization" (Description, I/O Contract), rowwise outputs;
// "Implementation:NVIDIA TransformerEngine Ops Fused Backward Add RMSNorm"
// (Description, I/O Contract) for the residual add.
//
// Why the statistics buffers of two rows suffice: a peer pushes row k+2's
// statistics only after it merged row k+1, which needs this CTA's push of
// row k+1, which this CTA makes after it has read row k's entries.
#pragma once

#include "ring.cuh"

namespace gbn {

constexpr int kMaxRowCluster = 8;

// The statistics exchange of one row (buffer and mbarrier k & 1).  The wait
// is bounded; the caller turns a timeout into its abort flag.
struct RowExchange {
  uint64_t* bar;   // [2] mbarriers
  float2* buf;     // [2][kMaxRowCluster]
  uint32_t C, rank;

  // Arms row k's mbarrier for C pushes of 8 bytes (one thread).
  __device__ void arm(int64_t k) const {
    mbar_arrive_expect_tx(&bar[k & 1], C * static_cast<uint32_t>(sizeof(float2)));
  }
  // Pushes v to every CTA of the cluster (lanes 0..C-1 of one warp).
  __device__ void push(int64_t k, int lane, float2 v) const {
    if (lane < static_cast<int>(C)) push_stat(&buf[(k & 1) * kMaxRowCluster + rank], &bar[k & 1],
                                              static_cast<uint32_t>(lane), v);
  }
  __device__ bool wait(int64_t k) const {
    return mbar_wait(&bar[k & 1], static_cast<uint32_t>((k >> 1) & 1));
  }
  __device__ const float2* entries(int64_t k) const { return &buf[(k & 1) * kMaxRowCluster]; }

  // Two rows per exchange (pair pr): buf is [2 parities][2 rows][kMaxRowCluster].
  __device__ void arm2(int64_t pr) const {
    mbar_arrive_expect_tx(&bar[pr & 1], C * 2 * static_cast<uint32_t>(sizeof(float2)));
  }
  __device__ void push2(int64_t pr, int lane, float2 v0, float2 v1) const {
    if (lane < static_cast<int>(C)) {
      float2* b = &buf[(pr & 1) * 2 * kMaxRowCluster + rank];
      push_stat(b, &bar[pr & 1], static_cast<uint32_t>(lane), v0);
      push_stat(b + kMaxRowCluster, &bar[pr & 1], static_cast<uint32_t>(lane), v1);
    }
  }
  __device__ const float2* entries2(int64_t pr, int row) const {
    return &buf[((pr & 1) * 2 + row) * kMaxRowCluster];
  }
  // Zeroes the entries past C (no peer writes them) of a buffer of `n`
  // entries, so that a merge may add all kMaxRowCluster entries without a
  // test: adding +0 leaves a sum's bits unchanged.  Before the first cluster
  // barrier.
  __device__ void zero_unused(int tid, int T, int n) const {
    for (int i = tid; i < n; i += T)
      if (static_cast<uint32_t>(i % kMaxRowCluster) >= C) buf[i] = make_float2(0.f, 0.f);
  }
};

template <typename Tin, int QM, bool LN, int NV>
__global__ void __launch_bounds__(fwd_ring_max_threads(NV))
    fwd_cluster_kernel(const FwdParams p, const int stages, const int hc) {
  pdl_begin();
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  constexpr int NP = VEC / 2;
  using Tout = typename std::conditional<QM == Q_NONE, Tin, uint8_t>::type;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxRingStages];
  __shared__ uint64_t statbar[2];
  __shared__ float2 statbuf[2 * kMaxRowCluster];
  __shared__ __align__(16) float red[2][32];
  __shared__ int s_abort;
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
  const int H = p.hidden;
  const int c0 = static_cast<int>(rank) * hc;
  const int nvec = hc / VEC;
  const float inv_h = 1.f / static_cast<float>(H), inv_hc = 1.f / static_cast<float>(hc);
  const uint32_t row_bytes = static_cast<uint32_t>(hc) * sizeof(Tin);
  const uint32_t stage_bytes = static_cast<uint32_t>(ring_slot_bytes(NV, T));
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t count = cid < p.rows ? (p.rows - 1 - cid) / ncl + 1 : 0;
  const int64_t row_step = ncl * H;
  const RowExchange ex{statbar, statbuf, C, rank};
  const bool c_pow2 = (C & (C - 1)) == 0;
  const float inv_c = 1.f / static_cast<float>(C);
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  const uint64_t qscale2 = p2(qscale, qscale);
  float amax_t = 0.f;

  int64_t issued = 0;
  const Tin* src = reinterpret_cast<const Tin*>(p.x) + cid * H + c0;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    mbar_init(&statbar[0], 1);
    mbar_init(&statbar[1], 1);
    fence_mbar_init();
    for (; issued < stages && issued < count; ++issued, src += row_step) {
      const int s = static_cast<int>(issued);
      mbar_arrive_expect_tx(&full[s], row_bytes);
      bulk_g2s(ring + s * stage_bytes, src, row_bytes, &full[s]);
    }
  }
  for (int i = tid; i < 64; i += T) (&red[0][0])[i] = 0.f;
  zero_slot_tails(ring, stages, stage_bytes, row_bytes);
  uint64_t gw[NV][NP], bw[LN ? NV : 1][NP];
  {
    const float gadd = p.zcg ? 1.f : 0.f;
    const int wc = c0 / VEC;  // this CTA's first weight vector
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      load_weight_pairs<VEC>(p.gamma, p.w_dt, wc + v, v < nvec, gadd, gw[kk]);
      if constexpr (LN) load_weight_pairs<VEC>(p.beta, p.w_dt, wc + v, v < nvec, 0.f, bw[kk]);
    }
  }
  // Peers push into this CTA's statistics mbarriers: initialized cluster-wide
  // before the first push.
  cluster_sync();

  const uint8_t* xs = ring + tid * 16;
  Tout* orow = reinterpret_cast<Tout*>(p.out) + cid * H + c0 + tid * VEC;
  const int64_t vstep = static_cast<int64_t>(T) * VEC;
  int rb = 0;
  int st = 0;
  uint32_t phase = 0;
  int64_t k = 0;
  // LayerNorm with every thread holding NV full vectors and a power-of-two
  // warp count: one block reduction per row (Chan's merge of per-thread mean
  // and M2 over equal counts) instead of a sum, then the M2 about its mean.
  const bool one_pass = LN && nvec == NV * T && nwarps >= 2 && (nwarps & (nwarps - 1)) == 0;
  for (; k < count; ++k, orow += row_step) {
    if (tid == 0) ex.arm(k);
    if (!mbar_wait(&full[st], phase)) s_abort = 1;
    uint64_t xp[NV][NP];
    uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const uint4 r = *reinterpret_cast<const uint4*>(xs + kk * T * 16);
      const uint32_t w[NW] = {r.x, r.y, r.z, r.w};
      widen_pairs<Tin, VEC>(w, xp[kk]);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        uint64_t& a = (i & 1) ? acc1 : acc0;
        a = LN ? add2(a, xp[kk][i]) : fma2(xp[kk][i], xp[kk][i], a);
      }
    }
    float s1;
    {
      const float2 a = u2(add2(acc0, acc1));
      s1 = a.x + a.y;
    }
    float2 mine;
    if (LN && one_pass) {
      // Thread: mean and M2 of its NV * VEC elements (a power of two).  Then
      // equal halves merge as m = (m_a + m_b) / 2, M2 = M2_a + M2_b +
      // (m_b - m_a)^2 * n / 2 (n elements per half): lanes by xor shuffles,
      // then the warps through shared memory by the same tree, so every
      // thread gets the same bits (each step is commutative).
      constexpr int NE = NV * VEC;
      const float mt = s1 * (1.f / static_cast<float>(NE));
      const uint64_t mt2 = p2(mt, mt);
      uint64_t q0 = 0ull, q1 = 0ull;
#pragma unroll
      for (int kk = 0; kk < NV; ++kk) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const uint64_t d = sub2(xp[kk][i], mt2);
          uint64_t& q = (i & 1) ? q1 : q0;
          q = fma2(d, d, q);
        }
      }
      const float2 qq = u2(add2(q0, q1));
      float m = mt, q = qq.x + qq.y;
      auto merge = [](float& m, float& q, float mo, float qo, float half_n) {
        const float d = mo - m;
        q = (q + qo) + (d * d) * half_n;
        m = (m + mo) * 0.5f;
      };
#pragma unroll
      for (int o = 1; o < 32; o <<= 1)
        merge(m, q, __shfl_xor_sync(0xFFFFFFFFu, m, o), __shfl_xor_sync(0xFFFFFFFFu, q, o),
              0.5f * static_cast<float>(NE * o));
      float2* r2 = reinterpret_cast<float2*>(red[rb]);
      if (lane == 0) r2[warp] = make_float2(m, q);
      __syncthreads();
      const float2 v = r2[lane & (nwarps - 1)];
      m = v.x;
      q = v.y;
      for (int o = 1; o < nwarps; o <<= 1)
        merge(m, q, __shfl_xor_sync(0xFFFFFFFFu, m, o), __shfl_xor_sync(0xFFFFFFFFu, q, o),
              0.5f * static_cast<float>(NE * 32 * o));
      mine = make_float2(m, q);
    } else {
      if (nwarps == 1) __syncthreads();
      s1 = row_block_sum(s1, red[rb], lane, warp, nwarps);
      mine = make_float2(0.f, s1);
    }
    rb ^= 1;
    if (s_abort) break;
    if (tid == 0 && issued < count) {
      mbar_arrive_expect_tx(&full[st], row_bytes);
      bulk_g2s(ring + st * stage_bytes, src, row_bytes, &full[st]);
      ++issued;
      src += row_step;
    }
    if (++st == stages) {
      st = 0;
      phase ^= 1u;
      xs = ring + tid * 16;
    } else {
      xs += stage_bytes;
    }
    // This slice's statistics: LayerNorm (mean, M2) about the slice mean,
    // RMSNorm (0, sum of squares).
    if (LN && !one_pass) {
      const float ml = s1 * inv_hc;
      const uint64_t m2 = p2(ml, ml);
      uint64_t q0 = 0ull, q1 = 0ull;
#pragma unroll
      for (int kk = 0; kk < NV; ++kk) {
        const bool act = kk * T + tid < nvec;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const uint64_t d = sub2(xp[kk][i], m2);
          uint64_t& q = (i & 1) ? q1 : q0;
          if (act) q = fma2(d, d, q);
        }
      }
      const float2 qq = u2(add2(q0, q1));
      mine = make_float2(ml, row_block_sum(qq.x + qq.y, red[rb], lane, warp, nwarps));
      rb ^= 1;
    }
    if (warp == 0) ex.push(k, lane, mine);
    // Every thread waits for the C entries itself (no barrier: a warp goes on
    // as soon as they have landed); a timeout is acted on after the next
    // barrier, as the copy wait's is.
    if (!ex.wait(k)) s_abort = 1;
    // Merge: lane c of every group of 8 lanes takes entry c (zero past C) and
    // the C entries are added as a tree of xor shuffles.  Every lane, warp and
    // CTA of the cluster adds the same pairs (fp32 addition is commutative),
    // so all get the same bits; a warp needs no barrier and no other warp.
    const float2* e = ex.entries(k);
    float mean = 0.f, ss = 0.f;
    {
      const uint32_t c = static_cast<uint32_t>(lane) & (kMaxRowCluster - 1);
      const float2 v = c < C ? e[c] : make_float2(0.f, 0.f);
      float t;
      if constexpr (LN) {
        float msum = v.x;
#pragma unroll
        for (int o = 1; o < kMaxRowCluster; o <<= 1) msum += __shfl_xor_sync(0xFFFFFFFFu, msum, o);
        // (a multiply by 1/C where C is a power of two: the same bits, and no
        // division sequence per row)
        mean = c_pow2 ? msum * inv_c : msum / static_cast<float>(C);
        const float d = v.x - mean;
        t = c < C ? fmaf(static_cast<float>(hc) * d, d, v.y) : 0.f;
      } else {
        t = v.y;
      }
#pragma unroll
      for (int o = 1; o < kMaxRowCluster; o <<= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
      ss = t;
    }
    const float rs = rsqrtf(fmaf(ss, inv_h, p.eps));
    const uint64_t rs2 = p2(rs, rs), mean2 = p2(mean, mean);
    if (tid == 0 && rank == 0) {
      const int64_t row = cid + k * ncl;
      if (LN && p.mu) p.mu[row] = mean;
      if (p.rsigma) p.rsigma[row] = rs;
    }

#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      const bool act = v < nvec;
      uint64_t z[NP];
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint64_t t = mul2(LN ? sub2(xp[kk][i], mean2) : xp[kk][i], rs2);
        z[i] = LN ? fma2(t, gw[kk][i], bw[kk][i]) : mul2(t, gw[kk][i]);
      }
      Tout* o = orow + kk * vstep;
      if constexpr (QM == Q_NONE) {
        if (act) {
          uint32_t w[NW];
          narrow_pairs<Tin, VEC>(z, w);
          st_words<NW>(o, w);
        }
      } else {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const float2 f = u2(z[i]);
          a = fmax_nan(a, fmax_nan(fabsf(f.x), fabsf(f.y)));
        }
        uint64_t s2 = qscale2;
        uint32_t code = 0;
        if constexpr (QM == Q_DELAYED) {
          if (act) amax_t = fmax_nan(amax_t, a);
        } else {  // MXFP8 rowwise: 32-element blocks span 32/VEC adjacent threads
          constexpr int TPB = 32 / VEC;
#pragma unroll
          for (int o2 = 1; o2 < TPB; o2 <<= 1) a = fmax_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, o2));
          float m;
          e8m0_scale(a, code, m);
          s2 = p2(m, m);
        }
        if (act && p.write_rowwise) {  // (columnwise-only: statistics and amax only)
          uint32_t w[VEC / 4];
#pragma unroll
          for (int i = 0; i < VEC / 4; ++i) w[i] = e4m3x4_pairs(z[2 * i], z[2 * i + 1], s2);
          st_words<VEC / 4>(o, w);
          if constexpr (QM == Q_MXFP8) {
            constexpr int TPB = 32 / VEC;
            if ((tid & (TPB - 1)) == 0)
              p.mx_scale[mx_row_scale_at(p, cid + k * ncl, (c0 + v * VEC) / 32)] =
                  static_cast<uint8_t>(code);
          }
        }
      }
    }
  }

  __syncthreads();  // a timeout of the last row's waits is seen by thread 0
  if (s_abort && tid == 0) {
    atomicOr(&g_gbn_device_error, 1u);
    drain_ring(full, stages, k, issued);
  }
  // No CTA leaves while a peer of its cluster may still push into it.
  cluster_sync();
  if (s_abort) return;
  if constexpr (QM == Q_DELAYED) {
    block_amax_commit(amax_t, red[0], p.amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      const float inv = 1.f / qscale;
      if (p.scale_inv) *p.scale_inv = inv;
      if (p.colwise_scale_inv) *p.colwise_scale_inv = inv;
    }
  }
}

// Backward of a long row over a cluster: a stage holds this CTA's slices of
// dz, x (and dresidual) of one row; each CTA reduces its slice's (sum dy,
// sum dy*xhat), the C pairs are exchanged and added in rank order, and each
// CTA writes dx for its columns.  Rows go two at a time through one block
// reduction and one exchange (the exchange's round trip is the per-row cost
// that matters here), with at least four stages so that the next two rows
// are in flight meanwhile.  dgamma/dbeta partials stay in registers and go to
// workspace row `cluster id`, columns of this CTA.
template <typename Tin, bool LN, bool ADD, int NV>
__global__ void __launch_bounds__(bwd_max_threads(NV))
    bwd_cluster_kernel(const BwdParams p, const int stages, const int hc) {
  pdl_begin();
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  constexpr int NP = VEC / 2;
  constexpr int NS = ADD ? 3 : 2;  // slots per stage: dz, x, (dresidual)
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxRingStages];
  __shared__ uint64_t statbar[2];
  __shared__ float2 statbuf[4 * kMaxRowCluster];  // [parity][row of the pair][sender]
  __shared__ __align__(16) float2 red[2][32];
  __shared__ int s_abort;
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
  const int H = p.hidden;
  const int c0 = static_cast<int>(rank) * hc;
  const int nvec = hc / VEC;
  const float inv_h = 1.f / static_cast<float>(H);
  const uint32_t row_bytes = static_cast<uint32_t>(hc) * sizeof(Tin);
  const uint32_t slot = static_cast<uint32_t>(ring_slot_bytes(NV, T));
  const uint32_t stage_bytes = NS * slot;
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t count = cid < p.rows ? (p.rows - 1 - cid) / ncl + 1 : 0;
  const int64_t row_step = ncl * H;
  const RowExchange ex{statbar, statbuf, C, rank};
  int64_t src_off = cid * H + c0;  // element offset of the next slice to fetch

  auto issue = [&](int s) {
    mbar_arrive_expect_tx(&full[s], NS * row_bytes);
    uint8_t* dst = ring + s * stage_bytes;
    bulk_g2s(dst, reinterpret_cast<const Tin*>(p.dz) + src_off, row_bytes, &full[s]);
    bulk_g2s(dst + slot, reinterpret_cast<const Tin*>(p.x) + src_off, row_bytes, &full[s]);
    if constexpr (ADD)
      bulk_g2s(dst + 2 * slot, reinterpret_cast<const Tin*>(p.dres) + src_off, row_bytes,
               &full[s]);
    src_off += row_step;
  };

  int64_t issued = 0;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    mbar_init(&statbar[0], 1);
    mbar_init(&statbar[1], 1);
    fence_mbar_init();
    for (; issued < stages && issued < count; ++issued) issue(static_cast<int>(issued));
  }
  zero_slot_tails(ring, stages * NS, slot, row_bytes);
  uint64_t gw[NV][NP], dg[NV][NP], db[LN ? NV : 1][NP];
  {
    const float gadd = p.zcg ? 1.f : 0.f;
    const int wc = c0 / VEC;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      load_weight_pairs<VEC>(p.gamma, p.w_dt, wc + v, v < nvec, gadd, gw[kk]);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        dg[kk][i] = 0ull;
        if constexpr (LN) db[kk][i] = 0ull;
      }
    }
  }
  ex.zero_unused(tid, T, 4 * kMaxRowCluster);
  cluster_sync();

  int64_t k = 0;
  // Rows are taken in pairs (k, k + 1): one block reduction and one cluster
  // exchange per pair, which halves the per-row exchange latency (the
  // exchange alone costs about a quarter of the time).  Both rows are read
  // from their stages twice (sums, then dx), so no row is held in registers
  // across the exchange; their stages are refilled at the next pair's barrier.
  int rb = 0;
  const int64_t vstep = static_cast<int64_t>(T) * VEC;
  Tin* dx0 = reinterpret_cast<Tin*>(p.dx) + cid * H + c0 + tid * VEC;  // row r: + r * row_step
  const float* mup = LN ? p.mu + cid : nullptr;
  const float* rsp = p.rsigma + cid;
  auto row_stats = [&](int64_t r, float& mu, float& rs) {
    rs = rsp[r * ncl];
    mu = LN ? mup[r * ncl] : 0.f;
  };
  // stage and phase parity of a row, advanced row by row (no divisions)
  auto next_stage = [&](int& s, uint32_t& ph) {
    if (++s == stages) {
      s = 0;
      ph ^= 1u;
    }
  };
  int sa = 0;       // stage of row k
  uint32_t pa = 0;  // its phase parity
  int si = static_cast<int>(issued % stages);  // stage of the next row to issue (thread 0)
  // this thread's dz, x (and dresidual) vectors of the row in stage s
  auto load_row = [&](int s, uint32_t (&dzw)[NV][NW], uint32_t (&xw)[NV][NW],
                      uint32_t (&rw)[ADD ? NV : 1][NW]) {
    const uint8_t* sb = ring + s * stage_bytes + tid * 16;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      // No bounds test: past the slice the slots are zero, and zero dz and x
      // contribute nothing to any sum.
      const uint4 a = *reinterpret_cast<const uint4*>(sb + kk * T * 16);
      const uint4 b = *reinterpret_cast<const uint4*>(sb + slot + kk * T * 16);
      dzw[kk][0] = a.x; dzw[kk][1] = a.y; dzw[kk][2] = a.z; dzw[kk][3] = a.w;
      xw[kk][0] = b.x; xw[kk][1] = b.y; xw[kk][2] = b.z; xw[kk][3] = b.w;
      if constexpr (ADD) {
        const uint4 c = *reinterpret_cast<const uint4*>(sb + 2 * slot + kk * T * 16);
        rw[kk][0] = c.x; rw[kk][1] = c.y; rw[kk][2] = c.z; rw[kk][3] = c.w;
      }
    }
  };
  // (sum dy, sum dy * xhat) of the thread's part of a row; dgamma/dbeta
  // partials accumulate
  auto row_sums = [&](const uint32_t (&dzw)[NV][NW], const uint32_t (&xw)[NV][NW], uint64_t mu2,
                      uint64_t rs2) {
    uint64_t sx = 0ull, sy = 0ull;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      uint64_t fz[NP], fx[NP];
      widen_pairs<Tin, VEC>(dzw[kk], fz);
      widen_pairs<Tin, VEC>(xw[kk], fx);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint64_t xh = mul2(sub2(fx[i], mu2), rs2);
        const uint64_t dy = mul2(fz[i], gw[kk][i]);
        sx = add2(sx, dy);
        sy = fma2(dy, xh, sy);
        dg[kk][i] = fma2(fz[i], xh, dg[kk][i]);
        if constexpr (LN) db[kk][i] = add2(db[kk][i], fz[i]);
      }
    }
    const float2 a = u2(sx), b = u2(sy);
    return make_float2(a.x + a.y, b.x + b.y);
  };
  // dx = rs * (dy - c1 - xhat * c2) = rs * dy - rs * c1 - (rs * c2) * xhat
  auto write_dx = [&](int64_t r, const uint32_t (&dzw)[NV][NW], const uint32_t (&xw)[NV][NW],
                      const uint32_t (&rw)[ADD ? NV : 1][NW], float mu, float rs, float2 t) {
    const uint64_t mu2 = p2(mu, mu), rs2 = p2(rs, rs);
    const float b1 = LN ? rs * (t.x * inv_h) : 0.f;
    const float a2 = rs * (t.y * inv_h);
    const uint64_t nb1 = p2(-b1, -b1), na2 = p2(-a2, -a2);
    Tin* dxrow = dx0 + r * row_step;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      uint64_t o[NP], fr[NP], fz[NP], fx[NP];
      if constexpr (ADD) widen_pairs<Tin, VEC>(rw[kk], fr);
      widen_pairs<Tin, VEC>(dzw[kk], fz);
      widen_pairs<Tin, VEC>(xw[kk], fx);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint64_t xh = mul2(sub2(fx[i], mu2), rs2);
        const uint64_t dy = mul2(fz[i], gw[kk][i]);
        o[i] = fma2(na2, xh, fma2(rs2, dy, nb1));
        if constexpr (ADD) o[i] = add2(o[i], fr[i]);
      }
      if (v < nvec) {
        uint32_t w[NW];
        narrow_pairs<Tin, VEC>(o, w);
        st_words<NW>(dxrow + kk * vstep, w);
      }
    }
  };

  // Row statistics are loaded one pair ahead so their latency is hidden.
  float mu_a = 0.f, rs_a = 0.f, mu_b = 0.f, rs_b = 0.f;
  if (count > 0) row_stats(0, mu_a, rs_a);
  if (count > 1) row_stats(1, mu_b, rs_b);
  for (; k < count; k += 2) {
    const bool two = k + 1 < count;  // uniform over the cluster
    const int64_t pr = k >> 1;       // pair index
    if (tid == 0) ex.arm2(pr);
    const float mua = mu_a, rsa = rs_a, mub = mu_b, rsb = rs_b;
    if (k + 2 < count) row_stats(k + 2, mu_a, rs_a);
    if (k + 3 < count) row_stats(k + 3, mu_b, rs_b);
    int sb = sa;
    uint32_t pb = pa;
    next_stage(sb, pb);  // row k + 1
    float2 s0, s1 = make_float2(0.f, 0.f);
    {
      if (!mbar_wait(&full[sa], pa)) s_abort = 1;
      uint32_t dzw[NV][NW], xw[NV][NW], rw[ADD ? NV : 1][NW];
      load_row(sa, dzw, xw, rw);
      s0 = row_sums(dzw, xw, p2(mua, mua), p2(rsa, rsa));
    }
    if (two) {
      if (!mbar_wait(&full[sb], pb)) s_abort = 1;
      uint32_t dzb[NV][NW], xb[NV][NW], rwb[ADD ? NV : 1][NW];
      load_row(sb, dzb, xb, rwb);
      s1 = row_sums(dzb, xb, p2(mub, mub), p2(rsb, rsb));
    }
    const float4 s4 = block_sum4(make_float4(s0.x, s0.y, s1.x, s1.y),
                                 reinterpret_cast<float4*>(red[rb]), lane, warp, nwarps);
    rb ^= 1;
    if (s_abort) break;
    // The previous pair's rows are written: refill their stages, in row order.
    if (tid == 0) {
      for (; issued < count && issued < k + stages; ++issued) {
        issue(si);
        if (++si == stages) si = 0;
      }
    }
    if (warp == 0) ex.push2(pr, lane, make_float2(s4.x, s4.y), make_float2(s4.z, s4.w));
    // One waiter, the rest of the CTA held at the barrier (uniform exit).
    if (tid == 0 && !ex.wait(pr)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    // entries past C are zeros: every entry is added, in rank order
    const float2* e0 = ex.entries2(pr, 0);
    const float2* e1 = ex.entries2(pr, 1);
    float2 t0 = make_float2(0.f, 0.f), t1 = make_float2(0.f, 0.f);
#pragma unroll
    for (uint32_t c = 0; c < kMaxRowCluster; ++c) {
      t0.x += e0[c].x;
      t0.y += e0[c].y;
      t1.x += e1[c].x;
      t1.y += e1[c].y;
    }
    {
      uint32_t dzw[NV][NW], xw[NV][NW], rw[ADD ? NV : 1][NW];
      load_row(sa, dzw, xw, rw);
      write_dx(k, dzw, xw, rw, mua, rsa, t0);
    }
    if (two) {
      uint32_t dzb[NV][NW], xb[NV][NW], rwb[ADD ? NV : 1][NW];
      load_row(sb, dzb, xb, rwb);
      write_dx(k + 1, dzb, xb, rwb, mub, rsb, t1);
    }
    sa = sb;
    pa = pb;
    next_stage(sa, pa);
  }

  if (s_abort && tid == 0) {
    atomicOr(&g_gbn_device_error, 1u);
    drain_ring(full, stages, k, issued);
  }
  cluster_sync();
  if (s_abort) return;
  float* pg = p.part_dgamma + cid * H + c0;
  float* pb = LN ? p.part_dbeta + cid * H + c0 : nullptr;
#pragma unroll
  for (int kk = 0; kk < NV; ++kk) {
    const int v = kk * T + tid;
    if (v < nvec) {
      uint32_t w[VEC];
      narrow_pairs<float, VEC>(dg[kk], w);
      st_words<VEC>(pg + v * VEC, w);
      if constexpr (LN) {
        narrow_pairs<float, VEC>(db[kk], w);
        st_words<VEC>(pb + v * VEC, w);
      }
    }
  }
}

}  // namespace gbn
