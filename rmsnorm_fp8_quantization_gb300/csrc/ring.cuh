// Row-pass kernels fed by a bulk-copy ring: the forward (rowwise outputs)
// and the backward.  One elected thread streams whole rows (or, for the
// backward, the dz / x / dresidual rows of one row index) into a ring of
// shared-memory stages with `cp.async.bulk` and mbarrier transaction counts;
// all threads compute from shared memory.  A stage is refilled as soon as
// every thread has copied its vectors out of it (after the first block
// reduction of the row), so `stages - 1` rows stay in flight per CTA
// independently of the register budget.
//
// Operations: "Implementation:NVIDIA TransformerEngine JAX XLA
// Normalization" (Description, I/O Contract) for the forward and backward;
// "Implementation:NVIDIA TransformerEngine Ops Fused Backward Add RMSNorm"
// (Description, I/O Contract) for the residual add.
#pragma once

#include <type_traits>

#include "gbn_device.cuh"

namespace gbn {

constexpr int kMaxRingStages = 8;

// Sticky flag of this translation unit: bit 0 = a wait for this library's
// own bulk copies exceeded kWaitLimitNs and the kernel stopped early.
static __device__ unsigned int g_gbn_device_error;

// Self-test of the bounded wait: one thread waits for 16 bytes on an
// mbarrier that no copy will ever fill, gives up after limit_ns and records
// the timeout in the device error flag, as a real kernel would.
static __global__ void copy_timeout_probe_kernel(const unsigned long long limit_ns) {
  pdl_begin();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, 16u);
    if (!mbar_wait_for(&bar, 0u, limit_ns)) atomicOr(&g_gbn_device_error, 1u);
  }
}

// Per-CTA schedule: this CTA owns rows first, first + stride, ...
struct RowSchedule {
  int64_t first, stride, count;
  __device__ RowSchedule(int64_t rows) : first(blockIdx.x), stride(gridDim.x) {
    count = first < rows ? (rows - 1 - first) / stride + 1 : 0;
  }
  __device__ int64_t row(int64_t k) const { return first + k * stride; }
};

// Waits (bounded) for every stage that still has a copy in flight, so that
// no bulk copy targets this CTA's shared memory after it exits.
__device__ __forceinline__ void drain_ring(uint64_t* full, int stages, int64_t next_k,
                                          int64_t issued) {
  for (int64_t k = next_k; k < issued; ++k) {
    mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
  }
}

// Loads VEC weights of this thread's vector v as VEC/2 fp32 pairs (+add).
template <int VEC>
__device__ __forceinline__ void load_weight_pairs(const void* base, int wdt, int v, bool act,
                                                  float add, uint64_t* out) {
  float f[VEC];
  if (act) {
    ld_weights<VEC>(base, wdt, v * VEC, f);
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) f[e] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) out[i] = p2(f[2 * i] + add, f[2 * i + 1] + add);
}

// Zeroes bytes [from, slot) of each of the n slots (slot apart) starting at
// base, cooperatively over the CTA.  `from` and `slot` are multiples of 16.
__device__ __forceinline__ void zero_slot_tails(uint8_t* base, int n, uint32_t slot,
                                                uint32_t from) {
  for (int q = 0; q < n; ++q)
    for (uint32_t b = from + 16u * threadIdx.x; b < slot; b += 16u * blockDim.x)
      *reinterpret_cast<uint4*>(base + q * slot + b) = make_uint4(0u, 0u, 0u, 0u);
}

// Block sum for the row kernels.  buf: 32 floats whose entries at and past
// nwarps are zero.  Up to 8 warps, every thread adds the warp partials from
// shared memory in one fixed order (no second shuffle tree).
__device__ __forceinline__ float row_block_sum(float v, float* buf, int lane, int warp,
                                               int nwarps) {
  v = warp_sum(v);
  if (nwarps == 1) return v;
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  if (nwarps <= 8) {
    const float4 a = *reinterpret_cast<const float4*>(buf);
    float r = (a.x + a.y) + (a.z + a.w);
    if (nwarps > 4) {
      const float4 b = *reinterpret_cast<const float4*>(buf + 4);
      r += (b.x + b.y) + (b.z + b.w);
    }
    return r;
  }
  return warp_sum(lane < nwarps ? buf[lane] : 0.f);
}
// Forward row pass.  Thread t owns vectors v = k*T + t (k < NV) of every row;
// its g' / beta stay in registers for the whole kernel as fp32 pairs, the row
// is widened to pairs once and all arithmetic runs two lanes per instruction.
// A stage slot holds NV*T vectors; the part past the row is zero, so the
// loads need no bounds test (zeros add nothing to either sum).
// ONE (LayerNorm only; the host selects it when every thread holds NV whole
// vectors of the row and the CTA has 8 or 16 warps):
// one block reduction per row, a merge of per-thread mean and M2 over equal
// counts, instead of a sum and then the M2 about it.  A template flag, not a
// runtime test: the two-pass variant keeps its own code.
template <typename Tin, int QM, bool LN, int NV, bool ONE = false>
__global__ void __launch_bounds__(fwd_ring_max_threads(NV)) fwd_ring_kernel(const FwdParams p,
                                                                           const int stages) {
  static_assert(!ONE || LN, "the one-pass merge is LayerNorm's");
  pdl_begin();
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  constexpr int NP = VEC / 2;
  using Tout = typename std::conditional<QM == Q_NONE, Tin, uint8_t>::type;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxRingStages];
  __shared__ __align__(16) float red[2][32];
  __shared__ int s_abort;
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const int H = p.hidden;
  const int nvec = H / VEC;
  const float inv_h = 1.f / static_cast<float>(H);
  const uint32_t row_bytes = static_cast<uint32_t>(H) * sizeof(Tin);
  const uint32_t stage_bytes = static_cast<uint32_t>(ring_slot_bytes(NV, T));
  const RowSchedule sched(p.rows);
  const int64_t row_step = sched.stride * H;  // elements between this CTA's rows
  float qscale = 1.f;
  if constexpr (QM == Q_DELAYED) qscale = *p.scale;
  const uint64_t qscale2 = p2(qscale, qscale);
  float amax_t = 0.f;

  int64_t issued = 0;
  const Tin* src = reinterpret_cast<const Tin*>(p.x) + sched.first * H;  // next row to fetch
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    for (; issued < stages && issued < sched.count; ++issued, src += row_step) {
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
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      load_weight_pairs<VEC>(p.gamma, p.w_dt, v, v < nvec, gadd, gw[kk]);
      if constexpr (LN) load_weight_pairs<VEC>(p.beta, p.w_dt, v, v < nvec, 0.f, bw[kk]);
    }
  }
  __syncthreads();

  // This thread's first element in the current row, in the input stage and
  // in the output.
  const uint8_t* xs = ring + tid * 16;
  Tout* orow = reinterpret_cast<Tout*>(p.out) + sched.first * H + tid * VEC;
  const int64_t vstep = static_cast<int64_t>(T) * VEC;  // elements between k-vectors
  int rb = 0;
  int st = 0;          // stage of row k
  uint32_t phase = 0;  // its mbarrier phase parity
  int64_t k = 0;
  for (; k < sched.count; ++k, orow += row_step) {
    if (!mbar_wait(&full[st], phase)) s_abort = 1;
    uint64_t xp[NV][NP];
    uint64_t acc0 = 0ull, acc1 = 0ull;  // two chains of pairs
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
    float mean = 0.f, ss = 0.f;
    if constexpr (ONE) {
      // Thread: mean and M2 of its NV * VEC elements; equal halves merge as
      // m = (m_a + m_b) / 2, M2 = M2_a + M2_b + (m_b - m_a)^2 * n / 2 (n per
      // half), lanes by xor shuffles, then the warps through shared memory
      // by the same tree: one block reduction per row, and every thread gets
      // the same bits (each step is commutative).
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
      __syncthreads();  // also: every thread has copied its vectors out of this stage
      const float2 v = r2[lane & (nwarps - 1)];
      m = v.x;
      q = v.y;
      for (int o = 1; o < nwarps; o <<= 1)
        merge(m, q, __shfl_xor_sync(0xFFFFFFFFu, m, o), __shfl_xor_sync(0xFFFFFFFFu, q, o),
              0.5f * static_cast<float>(NE * 32 * o));
      mean = m;
      ss = q;
    } else {
      // The barrier of the first reduction also tells thread 0 that every
      // thread has copied its vectors out of this stage.
      if (nwarps == 1) __syncthreads();
      s1 = row_block_sum(s1, red[rb], lane, warp, nwarps);
      ss = s1;
    }
    rb ^= 1;
    if (s_abort) break;
    if (tid == 0 && issued < sched.count) {
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
    if constexpr (ONE) {
      const uint64_t m2 = p2(mean, mean);
#pragma unroll
      for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int i = 0; i < NP; ++i) xp[kk][i] = sub2(xp[kk][i], m2);
    } else if constexpr (LN) {
      mean = s1 * inv_h;
      const uint64_t m2 = p2(mean, mean);
      uint64_t q0 = 0ull, q1 = 0ull;
#pragma unroll
      for (int kk = 0; kk < NV; ++kk) {
        const bool act = kk * T + tid < nvec;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          xp[kk][i] = sub2(xp[kk][i], m2);
          uint64_t& q = (i & 1) ? q1 : q0;
          if (act) q = fma2(xp[kk][i], xp[kk][i], q);
        }
      }
      const float2 qq = u2(add2(q0, q1));
      ss = row_block_sum(qq.x + qq.y, red[rb], lane, warp, nwarps);
      rb ^= 1;
    }
    const float rs = rsqrtf(fmaf(ss, inv_h, p.eps));
    const uint64_t rs2 = p2(rs, rs);
    if (tid == 0) {
      const int64_t row = sched.row(k);
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
        const uint64_t t = mul2(xp[kk][i], rs2);
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
        if (act) {
          uint32_t w[VEC / 4];
#pragma unroll
          for (int i = 0; i < VEC / 4; ++i) w[i] = e4m3x4_pairs(z[2 * i], z[2 * i + 1], s2);
          st_words<VEC / 4>(o, w);
          if constexpr (QM == Q_MXFP8) {
            constexpr int TPB = 32 / VEC;
            if ((tid & (TPB - 1)) == 0)
              p.mx_scale[mx_row_scale_at(p, sched.row(k), (v * VEC) / 32)] =
                  static_cast<uint8_t>(code);
          }
        }
      }
    }
  }

  if (s_abort) {
    if (tid == 0) {
      atomicOr(&g_gbn_device_error, 1u);
      drain_ring(full, stages, k, issued);
    }
    return;
  }
  if constexpr (QM == Q_DELAYED) {
    block_amax_commit(amax_t, red[0], p.amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      const float inv = 1.f / qscale;
      if (p.scale_inv) *p.scale_inv = inv;
      if (p.colwise_scale_inv) *p.colwise_scale_inv = inv;
    }
  }
}

// Backward row pass fed by the ring: a stage holds the dz, x (and
// dresidual) rows of one row index.  g' and the dgamma/dbeta partials stay in
// registers (fp32 pairs) across all rows of the CTA; the partials are written
// once to the CTA's workspace row.  When the register budget allows (KEEP)
// dy and xhat are kept between the two passes, otherwise recomputed from the
// packed inputs.
template <typename Tin, bool LN, bool ADD, int NV>
__global__ void __launch_bounds__(bwd_max_threads(NV)) bwd_ring_kernel(const BwdParams p,
                                                                      const int stages) {
  pdl_begin();
  constexpr int VEC = 16 / (int)sizeof(Tin);
  constexpr int NW = Words<Tin, VEC>::n;
  constexpr int NP = VEC / 2;
  constexpr int NS = ADD ? 3 : 2;  // streams per stage: dz, x, (dresidual)
  constexpr bool KEEP = (NV == 1) || (NV == 2 && !LN);
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxRingStages];
  __shared__ __align__(16) float2 red[2][32];
  __shared__ int s_abort;
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  const int H = p.hidden;
  const int nvec = H / VEC;
  const float inv_h = 1.f / static_cast<float>(H);
  const uint32_t row_bytes = static_cast<uint32_t>(H) * sizeof(Tin);
  const uint32_t slot = (row_bytes + 127u) & ~127u;
  const uint32_t stage_bytes = NS * slot;
  const Tin* srcs[3] = {reinterpret_cast<const Tin*>(p.dz), reinterpret_cast<const Tin*>(p.x),
                        reinterpret_cast<const Tin*>(p.dres)};
  const RowSchedule sched(p.rows);

  auto issue = [&](int s, int64_t row) {
    mbar_arrive_expect_tx(&full[s], NS * row_bytes);
#pragma unroll
    for (int q = 0; q < NS; ++q)
      bulk_g2s(ring + s * stage_bytes + q * slot, srcs[q] + row * H, row_bytes, &full[s]);
  };

  int64_t issued = 0;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    for (; issued < stages && issued < sched.count; ++issued)
      issue(static_cast<int>(issued), sched.row(issued));
  }

  uint64_t gw[NV][NP], dg[NV][NP], db[LN ? NV : 1][NP];
  {
    const float gadd = p.zcg ? 1.f : 0.f;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      load_weight_pairs<VEC>(p.gamma, p.w_dt, v, v < nvec, gadd, gw[kk]);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        dg[kk][i] = 0ull;
        if constexpr (LN) db[kk][i] = 0ull;
      }
    }
  }
  __syncthreads();

  // slots past the warp count read as zero in the block sums; no warp writes them
  for (int i = nwarps + tid; i < 32; i += T) red[0][i] = red[1][i] = make_float2(0.f, 0.f);
  int rb = 0;
  int st = 0;          // stage of row k
  uint32_t phase = 0;  // its mbarrier phase parity
  int64_t k = 0;
  // Row statistics are loaded one row ahead so their latency is hidden.
  float mu_next = 0.f, rs_next = 0.f;
  if (sched.count > 0) {
    if constexpr (LN) mu_next = p.mu[sched.row(0)];
    rs_next = p.rsigma[sched.row(0)];
  }
  for (; k < sched.count; ++k, st = st + 1 == stages ? 0 : st + 1, phase ^= (st == 0)) {
    const int64_t row = sched.row(k);
    const float mu = mu_next, rs = rs_next;
    if (k + 1 < sched.count) {
      if constexpr (LN) mu_next = p.mu[row + sched.stride];
      rs_next = p.rsigma[row + sched.stride];
    }
    if (!mbar_wait(&full[st], phase)) s_abort = 1;
    const uint8_t* sb = ring + st * stage_bytes;
    uint32_t dzw[NV][NW], xw[NV][NW], rw[ADD ? NV : 1][NW];
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      // Branch-free: a thread past the row's end reads the last vector and
      // zeroes it (zero dz and x contribute nothing to any sum).
      const int v = kk * T + tid;
      const bool act = v < nvec;
      const int vl = act ? v : nvec - 1;
      const uint4 a = *reinterpret_cast<const uint4*>(sb + vl * 16);
      const uint4 b = *reinterpret_cast<const uint4*>(sb + slot + vl * 16);
      dzw[kk][0] = act ? a.x : 0u; dzw[kk][1] = act ? a.y : 0u;
      dzw[kk][2] = act ? a.z : 0u; dzw[kk][3] = act ? a.w : 0u;
      xw[kk][0] = act ? b.x : 0u; xw[kk][1] = act ? b.y : 0u;
      xw[kk][2] = act ? b.z : 0u; xw[kk][3] = act ? b.w : 0u;
      if constexpr (ADD) {
        const uint4 c = *reinterpret_cast<const uint4*>(sb + 2 * slot + vl * 16);
        rw[kk][0] = c.x; rw[kk][1] = c.y; rw[kk][2] = c.z; rw[kk][3] = c.w;
      }
    }
    const uint64_t mu2 = p2(mu, mu), rs2 = p2(rs, rs);

    uint64_t sx = 0ull, sy = 0ull;  // pairs of (sum dy), (sum dy * xhat)
    uint64_t kdy[KEEP ? NV : 1][NP], kxh[KEEP ? NV : 1][NP];
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
        if constexpr (KEEP) {
          kdy[kk][i] = dy;
          kxh[kk][i] = xh;
        }
      }
    }
    float2 s;
    {
      const float2 a = u2(sx), b = u2(sy);
      s = make_float2(a.x + a.y, b.x + b.y);
    }
    if (nwarps == 1) __syncthreads();
    s = block_sum2(s, red[rb], lane, warp, nwarps);
    rb ^= 1;
    if (s_abort) break;
    if (tid == 0 && issued < sched.count) {
      issue(st, sched.row(issued));
      ++issued;
    }
    // dx = rs * (dy - c1 - xhat * c2) = rs * dy - rs * c1 - (rs * c2) * xhat
    const float b1 = LN ? rs * (s.x * inv_h) : 0.f;
    const float a2 = rs * (s.y * inv_h);
    const uint64_t nb1 = p2(-b1, -b1), na2 = p2(-a2, -a2);

#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
      const int v = kk * T + tid;
      uint64_t o[NP], fr[NP];
      if constexpr (ADD) widen_pairs<Tin, VEC>(rw[kk], fr);
      if constexpr (KEEP) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          o[i] = fma2(na2, kxh[kk][i], fma2(rs2, kdy[kk][i], nb1));
          if constexpr (ADD) o[i] = add2(o[i], fr[i]);
        }
      } else {
        uint64_t fz[NP], fx[NP];
        widen_pairs<Tin, VEC>(dzw[kk], fz);
        widen_pairs<Tin, VEC>(xw[kk], fx);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const uint64_t xh = mul2(sub2(fx[i], mu2), rs2);
          const uint64_t dy = mul2(fz[i], gw[kk][i]);
          o[i] = fma2(na2, xh, fma2(rs2, dy, nb1));
          if constexpr (ADD) o[i] = add2(o[i], fr[i]);
        }
      }
      if (v < nvec) {
        uint32_t w[NW];
        narrow_pairs<Tin, VEC>(o, w);
        st_words<NW>(reinterpret_cast<Tin*>(p.dx) + row * H + v * VEC, w);
      }
    }
  }

  if (s_abort) {
    if (tid == 0) {
      atomicOr(&g_gbn_device_error, 1u);
      drain_ring(full, stages, k, issued);
    }
    return;
  }
  float* pg = p.part_dgamma + static_cast<int64_t>(blockIdx.x) * H;
  float* pb = LN ? p.part_dbeta + static_cast<int64_t>(blockIdx.x) * H : nullptr;
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
