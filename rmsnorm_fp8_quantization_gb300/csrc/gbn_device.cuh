// Device-side helpers: typed vector loads/stores, conversions, reductions,
// FP8/E8M0 encoding through the hardware conversion, cluster primitives.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gbn_internal.h"

namespace gbn {

// ---------------------------------------------------------------- raw loads

// 16-byte streaming load: read-only path, no L1 allocation (the row is used
// once by this CTA).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Cached read-only loads (weights: reused by every row of the CTA).
__device__ __forceinline__ uint4 ld_cached16(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_cached8(const void* p) {
  uint2 r;
  asm("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// ---------------------------------------------------------------- element types

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kDt = DT_F32;
  __device__ __forceinline__ static float to_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kDt = DT_BF16;
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};
template <> struct Elem<__half> {
  static constexpr int kDt = DT_F16;
  __device__ __forceinline__ static float to_f(__half v) { return __half2float(v); }
};

// Unpacks 32-bit words holding packed elements of T into floats.
template <typename T, int N>
__device__ __forceinline__ void unpack(const uint32_t* w, float* f) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < N; ++i) f[i] = __uint_as_float(w[i]);
  } else if constexpr (Elem<T>::kDt == DT_BF16) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 v = __half22float2(h);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
}

// Number of 32-bit words in a vector of VEC elements of T.
template <typename T, int VEC>
struct Words {
  static constexpr int n = (VEC * (int)sizeof(T)) / 4;
};

// Loads VEC elements of T (16-byte aligned group) as raw words.
template <typename T, int VEC, bool STREAM>
__device__ __forceinline__ void ld_vec_raw(const T* p, uint32_t* w) {
  constexpr int B = VEC * (int)sizeof(T);
  static_assert(B % 8 == 0, "vector must be a multiple of 8 bytes");
  if constexpr (B % 16 == 0) {
#pragma unroll
    for (int c = 0; c < B / 16; ++c) {
      uint4 r = STREAM ? ld_stream16(reinterpret_cast<const uint8_t*>(p) + 16 * c)
                       : ld_cached16(reinterpret_cast<const uint8_t*>(p) + 16 * c);
      w[4 * c] = r.x; w[4 * c + 1] = r.y; w[4 * c + 2] = r.z; w[4 * c + 3] = r.w;
    }
  } else {
    uint2 r = ld_cached8(p);
    w[0] = r.x; w[1] = r.y;
  }
}

// Loads VEC weights of runtime dtype `wdt` starting at element `idx` as floats.
template <int VEC>
__device__ __forceinline__ void ld_weights(const void* base, int wdt, int idx, float* f) {
  if (wdt == DT_F32) {
    uint32_t w[VEC];
    ld_vec_raw<float, VEC, false>(reinterpret_cast<const float*>(base) + idx, w);
    unpack<float, VEC>(w, f);
  } else if (wdt == DT_BF16) {
    uint32_t w[VEC / 2];
    ld_vec_raw<__nv_bfloat16, VEC, false>(reinterpret_cast<const __nv_bfloat16*>(base) + idx, w);
    unpack<__nv_bfloat16, VEC>(w, f);
  } else {
    uint32_t w[VEC / 2];
    ld_vec_raw<__half, VEC, false>(reinterpret_cast<const __half*>(base) + idx, w);
    unpack<__half, VEC>(w, f);
  }
}

// Scalar element access for the generic (any alignment, any size) path.
template <typename T>
__device__ __forceinline__ float ld_scalar(const T* p, int64_t i) {
  return Elem<T>::to_f(p[i]);
}
__device__ __forceinline__ float ld_weight_scalar(const void* base, int wdt, int64_t i) {
  if (wdt == DT_F32) return reinterpret_cast<const float*>(base)[i];
  if (wdt == DT_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  return __half2float(reinterpret_cast<const __half*>(base)[i]);
}
template <typename T>
__device__ __forceinline__ void st_scalar(T* p, int64_t i, float v);
template <> __device__ __forceinline__ void st_scalar<float>(float* p, int64_t i, float v) {
  p[i] = v;
}
template <>
__device__ __forceinline__ void st_scalar<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ void st_scalar<__half>(__half* p, int64_t i, float v) {
  p[i] = __float2half_rn(v);
}
__device__ __forceinline__ void st_weight_scalar(void* base, int wdt, int64_t i, float v) {
  if (wdt == DT_F32) reinterpret_cast<float*>(base)[i] = v;
  else if (wdt == DT_BF16) reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
}

// An L2 access policy that marks every line it touches evict-last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 32-byte store (32-byte aligned): one full sector per instruction, under
// the L2 cache policy `pol`.
__device__ __forceinline__ void st_global_v8_policy(void* p, const uint32_t* w, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
               "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
               "r"(w[7]), "l"(pol)
               : "memory");
}

// Stores a packed vector (16 or 32 bytes of words; 16-byte aligned).
template <int NW>
__device__ __forceinline__ void st_words(void* p, const uint32_t* w) {
  static_assert(NW % 4 == 0 || NW == 2 || NW == 1, "");
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int c = 0; c < NW / 4; ++c)
      reinterpret_cast<uint4*>(p)[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  } else if constexpr (NW == 2) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint32_t*>(p) = w[0];
  }
}

// ---------------------------------------------------------------- packed fp32 pairs
//
// Blackwell executes two fp32 lanes per instruction (add/mul/fma .f32x2,
// round to nearest even per lane, identical to the scalar forms).  A pair is
// held as one 64-bit register pair: .x in the low half.

__device__ __forceinline__ uint64_t p2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 u2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// A 32-bit word of two packed elements of T as a pair of floats.
template <typename T>
__device__ __forceinline__ uint64_t widen2(uint32_t w) {
  if constexpr (Elem<T>::kDt == DT_BF16) {
    return p2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w));
    return p2(v.x, v.y);
  }
}
// A pair of floats rounded (RNE) into one word of two packed elements of T.
template <typename T>
__device__ __forceinline__ uint32_t narrow2(uint64_t v) {
  const float2 f = u2(v);
  if constexpr (Elem<T>::kDt == DT_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
// N elements of T held in N/2 pairs, from raw words (N*sizeof(T)/4 words).
template <typename T, int N>
__device__ __forceinline__ void widen_pairs(const uint32_t* w, uint64_t* pr) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) pr[i] = p2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) pr[i] = widen2<T>(w[i]);
  }
}
template <typename T, int N>
__device__ __forceinline__ void narrow_pairs(const uint64_t* pr, uint32_t* w) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float2 f = u2(pr[i]);
      w[2 * i] = __float_as_uint(f.x);
      w[2 * i + 1] = __float_as_uint(f.y);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) w[i] = narrow2<T>(pr[i]);
  }
}

// ---------------------------------------------------------------- FP8 / E8M0

// Two floats to two E4M3 codes (hardware cvt, RNE, satfinite); `lo` lands in
// the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ uint8_t e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}


// Four E4M3 codes of the pairs a = (v0, v1), b = (v2, v3), each scaled by s.
__device__ __forceinline__ uint32_t e4m3x4_pairs(uint64_t a, uint64_t b, uint64_t s) {
  const float2 x = u2(mul2(a, s)), y = u2(mul2(b, s));
  return e4m3x2(x.x, x.y) | (e4m3x2(y.x, y.y) << 16);
}

// NaN-propagating maximum.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Code and multiplier of the MX block scale for block amax A >= 0 (or NaN):
// the code is the biased exponent of 2^(floor(log2 A) - 8), 8 being the
// largest exponent of E4M3 -- A's exponent field minus 8 for normal A,
// clamped at 0 (zero and subnormal A give 0); Inf/NaN give code 255.  The
// multiplier is 2^(127 - code) as fp32 (always normal: code <= 246 for
// finite A), NaN for code 255.
__device__ __forceinline__ void e8m0_scale(float A, uint32_t& code, float& mult) {
  const uint32_t e = __float_as_uint(A) >> 23;  // sign is 0 for A >= 0
  const uint32_t t = max(e, 8u);
  code = e == 255u ? 255u : t - 8u;
  mult = e == 255u ? __uint_as_float(0x7FFFFFFFu) : __uint_as_float((262u - t) << 23);
}

// Byte offset of scale (r, c) in the tiled GEMM order: 512-byte tiles of
// 128 x 4 scales, `tiles_per_row` tiles (of 4 columns) per 128 rows, scale
// (r, c) of a tile at 16 * (r % 32) + 4 * (r / 32) + c.
__device__ __forceinline__ int64_t mx_tiled_offset(int64_t r, int64_t c, int64_t tiles_per_row) {
  return ((r >> 7) * tiles_per_row + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}
// Index of the rowwise MXFP8 scale of (row, block) in p.mx_scale.
__device__ __forceinline__ int64_t mx_row_scale_at(const FwdParams& p, int64_t row, int64_t blk) {
  const int64_t nb = p.hidden / 32;
  return p.mx_swizzle ? mx_tiled_offset(row, blk, (nb + 3) / 4) : row * nb + blk;
}
// Index of the columnwise MXFP8 scale of (32-row stripe, column) in
// p.mx_colwise_scale; the tiled order treats the operand as transposed.
__device__ __forceinline__ int64_t mx_col_scale_at(const FwdParams& p, int64_t stripe,
                                                   int64_t col) {
  const int64_t ns = p.rows / 32;
  return p.mx_swizzle ? mx_tiled_offset(col, stripe, (ns + 3) / 4)
                      : stripe * p.hidden + col;
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xFFFFFFFFu, v.x, o);
    v.y += __shfl_xor_sync(0xFFFFFFFFu, v.y, o);
  }
  return v;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Block-wide sum of a pair; every thread gets the same bits.  `buf` holds 32
// pairs (16-byte aligned) and must alternate between two buffers on
// consecutive calls (one barrier per call suffices then).  Up to 16 warps,
// every thread reads the warp partials from shared memory and adds them in
// one fixed order (entries at and past nwarps read as zero) instead of a
// second shuffle tree.
__device__ __forceinline__ float2 block_sum2(float2 v, float2* buf, int lane, int warp,
                                             int nwarps) {
  v = warp_sum2(v);
  if (nwarps == 1) return v;
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  if (nwarps <= 8) {
    const float4* b4 = reinterpret_cast<const float4*>(buf);
    const float4 a = b4[0];
    const float4 b = nwarps > 2 ? b4[1] : make_float4(0.f, 0.f, 0.f, 0.f);
    float2 r = make_float2((a.x + a.z) + (b.x + b.z), (a.y + a.w) + (b.y + b.w));
    if (nwarps > 4) {
      const float4 c = b4[2];
      const float4 d = nwarps > 6 ? b4[3] : make_float4(0.f, 0.f, 0.f, 0.f);
      r.x += (c.x + c.z) + (d.x + d.z);
      r.y += (c.y + c.w) + (d.y + d.w);
    }
    return r;
  }
  if (nwarps <= 16) {
    const float4* b4 = reinterpret_cast<const float4*>(buf);
    float2 r = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 a = b4[2 * q], b = b4[2 * q + 1];
      r.x += (a.x + a.z) + (b.x + b.z);
      r.y += (a.y + a.w) + (b.y + b.w);
    }
    return r;
  }
  float2 r = lane < nwarps ? buf[lane] : make_float2(0.f, 0.f);
  return warp_sum2(r);
}

// Block-wide sum of four values (two pairs); every thread gets the same
// bits.  `buf` holds one float4 per warp (up to 32 warps, 16-byte aligned)
// and must alternate between two buffers on consecutive calls.  The warp
// partials are added in warp order.
__device__ __forceinline__ float4 block_sum4(float4 v, float4* buf, int lane, int warp,
                                             int nwarps) {
  const float2 a = warp_sum2(make_float2(v.x, v.y)), b = warp_sum2(make_float2(v.z, v.w));
  v = make_float4(a.x, a.y, b.x, b.y);
  if (nwarps == 1) return v;
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  float4 r = buf[0];
  for (int w = 1; w < nwarps; ++w) {
    const float4 u = buf[w];
    r.x += u.x;
    r.y += u.y;
    r.z += u.z;
    r.w += u.w;
  }
  return r;
}

// Final amax of a CTA into *amax (float bits as int: valid for values >= 0,
// NaN compares above every finite value and Inf).  `buf` needs 32 floats and
// must not be in use by other threads.
__device__ __forceinline__ void block_amax_commit(float v, float* buf, float* amax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
  v = warp_max_nan(v);
  __syncthreads();
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float r = lane < nwarps ? buf[lane] : 0.f;
    r = warp_max_nan(r);
    if (lane == 0) atomicMax(reinterpret_cast<int*>(amax), static_cast<int>(__float_as_uint(r)));
  }
}

// ---------------------------------------------------------------- bulk copies + mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Programmatic dependent launch.  Every kernel of the library first lets the
// next kernel of the stream begin launching (its CTAs take SMs as this
// grid's CTAs leave), then waits until the previous kernel has completed and
// its writes are visible, before touching global memory.  Without the launch
// attribute both are no-ops.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Makes initialized mbarriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrives once on `bar` and adds `bytes` to the transaction count of its
// current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of
// 16) whose completion is reported as transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// One bounded wait for phase `parity`: the thread is suspended in hardware
// until the phase completes or about `hint_ns` pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Upper bound on any wait for this kernel's own bulk copies.  A copy that
// has not landed after this long means something is wrong; the kernel then
// records the fact in `err` and stops instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Waits for phase `parity` of `bar` to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity, 1000000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity, 1000000u)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Barrier over every thread of every CTA in the cluster, with release /
// acquire ordering of shared-memory writes (a hardware barrier, not a spin).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Pushes v into element `buf` of CTA `rank` of this cluster and reports
// 8 bytes on that CTA's mbarrier `bar` (same offsets in every CTA).
__device__ __forceinline__ void push_stat(float2* buf, uint64_t* bar, uint32_t rank, float2 v) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(buf)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(ra), "f"(v.x), "f"(v.y), "r"(rb)
               : "memory");
}



}  // namespace gbn
