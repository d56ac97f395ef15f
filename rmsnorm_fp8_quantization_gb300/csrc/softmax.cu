// Scaled (masked) softmax, forward and backward: the softmax kernels named
// on "Migrate norms and softmax kernels to NVRTC" (Description:
// scaled_masked_softmax, scaled_upper_triang_masked_softmax,
// scaled_aligned_causal_masked_softmax; forward and backward).  The page
// gives no formulas; these follow the plain definitions:
//   y  = softmax over the last axis of scale * x, over the kept positions
//        (masked ones are 0; a row with nothing kept is all 0);
//   dx = scale * y * (dy - sum_j dy * y).
//
// A row of sk elements is handled by a group of G = 32 * WPR threads (WPR
// warps, one to eight), each holding NV loads of V elements in registers, so a
// row is read once and written once.  The reductions (max, then sum; or
// sum dy * y) run over the group: warp shuffles, then shared memory when
// WPR > 1.  exp is taken as 2^(x * scale * log2(e) - (max - 64)): the
// hardware ex2 (flush-to-zero) on arguments at most 64, whose results stay
// normal for every term above 2^-190; the common factor 2^64 cancels in the
// normalization, and the final multiply by 1/sum (in full fp32, subnormal
// results included) rounds each output once from its normal-range term.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>

#include "gbnorm.h"
#include "gbn_device.cuh"

namespace gbn {
namespace {

constexpr int kSmThreads = 256;
constexpr int64_t kMaxSoftmaxKeys = GBN_SOFTMAX_MAX_KEYS;
constexpr float kLog2e = 1.4426950408889634f;

// 2^a by the hardware approximation, subnormal results flushed to zero.
__device__ __forceinline__ float ex2_ftz(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

template <typename T>
struct SmElem;
template <>
struct SmElem<float> {
  static __device__ float get(const float* p) { return *p; }
  static __device__ void put(float* p, float v) { *p = v; }
};
template <>
struct SmElem<__nv_bfloat16> {
  static __device__ float get(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ void put(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <>
struct SmElem<__half> {
  static __device__ float get(const __half* p) { return __half2float(*p); }
  static __device__ void put(__half* p, float v) { *p = __float2half_rn(v); }
};

template <typename T, int V>
__device__ __forceinline__ void store_v(T* p, const float* f) {
  if constexpr (V == 1) {
    SmElem<T>::put(p, f[0]);
  } else {
    uint64_t pr[V / 2];
#pragma unroll
    for (int i = 0; i < V / 2; ++i) pr[i] = p2(f[2 * i], f[2 * i + 1]);
    uint32_t w[Words<T, V>::n];
    narrow_pairs<T, V>(pr, w);
    st_words<Words<T, V>::n>(p, w);
  }
}

// Group-wide reduction (max or sum) over the WPR warps of one row.  `buf`:
// kSmThreads / 32 floats; all rows of the CTA call it together.
template <bool MAX>
__device__ __forceinline__ float group_reduce(float v, float* buf, int wpr) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = MAX ? fmaxf(v, u) : v + u;
  }
  if (wpr == 1) return v;
  const int warp = threadIdx.x >> 5, first = warp - warp % wpr;
  if ((threadIdx.x & 31) == 0) buf[warp] = v;
  __syncthreads();
  float r = buf[first];
  for (int w = 1; w < wpr; ++w) r = MAX ? fmaxf(r, buf[first + w]) : r + buf[first + w];
  __syncthreads();
  return r;
}

struct SmFwdParams {
  const void* x;
  const uint8_t* mask;
  void* y;
  int64_t rows;        // batches * heads * sq
  int64_t heads_sq;    // heads * sq
  int64_t sq;
  int64_t mask_batches;
  int sk;
  int wpr;             // warps per row
  float scale_log2e;
};

// Loads V consecutive elements as raw 32-bit words (V >= 2: 16 bytes).
template <typename T, int V>
__device__ __forceinline__ void load_words(const T* p, uint32_t* w) {
  if constexpr (V == 1) {
    w[0] = __float_as_uint(SmElem<T>::get(p));
  } else {
    const uint4 u = ld_stream16(p);
    w[0] = u.x;
    w[1] = u.y;
    w[2] = u.z;
    w[3] = u.w;
  }
}
template <typename T, int V>
__device__ __forceinline__ void words_to_floats(const uint32_t* w, float* f) {
  if constexpr (V == 1) {
    f[0] = __uint_as_float(w[0]);
  } else {
    uint64_t pr[V / 2];
    widen_pairs<T, V>(w, pr);
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      const float2 t = u2(pr[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// Forward.  MASK: 0 none, 1 padding mask, 2 upper-triangular, 3 aligned
// causal.  The CTA walks blocks of rows_per_cta rows (blockIdx, blockIdx +
// gridDim, ...).  With the most loads per thread (NV = 8) the grid is
// persistent and the next block's packed row (and mask bytes) is loaded into
// registers while the current one is computed; with fewer, one block per CTA
// and more CTAs resident (fewer registers) keep enough bytes in flight.
template <typename T, int V, int NV, int MASK>
__global__ void __launch_bounds__(kSmThreads, NV == 8 ? 2 : 4)
    softmax_fwd_kernel(const SmFwdParams p) {
  pdl_begin();
  constexpr int NW = V == 1 ? 1 : 4;
  __shared__ float buf[kSmThreads / 32];
  const int gthreads = 32 * p.wpr;
  const int rows_per_cta = kSmThreads / gthreads;
  const int g = threadIdx.x / gthreads, t = threadIdx.x % gthreads;
  const int sk = p.sk;
  const int64_t nblocks = (p.rows + rows_per_cta - 1) / rows_per_cta;

  // Index arithmetic in 32 bits when every operand fits (a 64-bit division
  // is a long instruction sequence, taken per row).
  const bool narrow = p.rows <= INT32_MAX && p.heads_sq <= INT32_MAX && p.mask_batches <= INT32_MAX;
  auto mod_sq = [&](int64_t row) -> int64_t {
    return narrow ? static_cast<int64_t>(static_cast<uint32_t>(row) % static_cast<uint32_t>(p.sq))
                  : row % p.sq;
  };
  // Positions j < limit of row `row` may be kept (causal rows end early).
  auto row_limit = [&](int64_t row) {
    int limit = sk;
    const int64_t i = mod_sq(row);
    if constexpr (MASK == 2) limit = static_cast<int>(i) + 1;
    if constexpr (MASK == 3) {
      const int64_t l = i + 1 + (sk - p.sq);
      limit = l < 0 ? 0 : (l > sk ? sk : static_cast<int>(l));
    }
    return limit;
  };
  // Loads the block's row; `limit` is kept for compute().
  auto fetch = [&](int64_t blk, uint32_t (&w)[NV][NW], uint64_t (&mb)[NV], int& limit) {
    const int64_t row = blk * rows_per_cta + g;
    const bool live = blk < nblocks && row < p.rows;
    limit = live ? row_limit(row) : 0;
    const T* xr = reinterpret_cast<const T*>(p.x) + (live ? row : 0) * sk;
    const uint8_t* mr = nullptr;
    if constexpr (MASK == 1) {
      const int64_t r = live ? row : 0;
      const int64_t b = narrow ? static_cast<int64_t>(static_cast<uint32_t>(r) /
                                                      static_cast<uint32_t>(p.heads_sq) %
                                                      static_cast<uint32_t>(p.mask_batches))
                               : r / p.heads_sq % p.mask_batches;
      mr = p.mask + (b * p.sq + mod_sq(r)) * static_cast<int64_t>(sk);
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j0 = (k * gthreads + t) * V;
      mb[k] = 0;
      if (j0 < limit) {
        load_words<T, V>(xr + j0, w[k]);
        if constexpr (MASK == 1) {
          if constexpr (V == 8) {
            mb[k] = *reinterpret_cast<const uint64_t*>(mr + j0);
          } else if constexpr (V == 4) {
            mb[k] = *reinterpret_cast<const uint32_t*>(mr + j0);
          } else {
            mb[k] = mr[j0];
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < NW; ++e) w[k][e] = 0u;
      }
    }
  };

  // Softmax of the block's row from its packed loads w and mask bytes mb.
  auto compute = [&](int64_t blk, const uint32_t (&w)[NV][NW], const uint64_t (&mb)[NV],
                     const int limit) {
    const int64_t row = blk * rows_per_cta + g;
    const bool live = row < p.rows;
    float u[NV][V];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j0 = (k * gthreads + t) * V;
      words_to_floats<T, V>(w[k], u[k]);
      if (MASK != 1 && j0 + V <= limit) {  // the whole vector is kept
        if constexpr (V >= 2) {  // two lanes per instruction
          const uint64_t sc2 = p2(p.scale_log2e, p.scale_log2e);
#pragma unroll
          for (int e = 0; e < V; e += 2) {
            const float2 f = u2(mul2(p2(u[k][e], u[k][e + 1]), sc2));
            u[k][e] = f.x;
            u[k][e + 1] = f.y;
          }
        } else {
          u[k][0] *= p.scale_log2e;
        }
#pragma unroll
        for (int e = 0; e < V; ++e) m = fmaxf(m, u[k][e]);
      } else if (MASK != 1 && j0 >= limit) {
        // nothing of this vector is kept: no part in the max or the sum
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) {
          bool keep = j0 + e < limit;
          if constexpr (MASK == 1) keep = keep && ((mb[k] >> (8 * e)) & 0xFFu) == 0;
          u[k][e] = keep ? u[k][e] * p.scale_log2e : -INFINITY;
          m = fmaxf(m, u[k][e]);
        }
      }
    }
    m = group_reduce<true>(m, buf, p.wpr);
    // nothing kept: every term is 2^-inf = 0
    const float mo = (m == -INFINITY ? 0.f : m) - 64.f;
    float s = 0.f;
    uint64_t s2 = 0ull;  // (even, odd) partial sums, V >= 2
    const uint64_t mo2 = p2(mo, mo);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j0 = (k * gthreads + t) * V;
      if (MASK != 1 && j0 >= limit) {
#pragma unroll
        for (int e = 0; e < V; ++e) u[k][e] = 0.f;
      } else if constexpr (V >= 2) {
#pragma unroll
        for (int e = 0; e < V; e += 2) {
          const float2 d = u2(sub2(p2(u[k][e], u[k][e + 1]), mo2));
          u[k][e] = ex2_ftz(d.x);
          u[k][e + 1] = ex2_ftz(d.y);
          s2 = add2(s2, p2(u[k][e], u[k][e + 1]));
        }
      } else {
        u[k][0] = ex2_ftz(u[k][0] - mo);
        s += u[k][0];
      }
    }
    if constexpr (V >= 2) {
      const float2 f = u2(s2);
      s = f.x + f.y;
    }
    s = group_reduce<false>(s, buf, p.wpr);
    const float inv = s > 0.f ? 1.f / s : 0.f;
    T* yr = reinterpret_cast<T*>(p.y) + (live ? row : 0) * sk;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j0 = (k * gthreads + t) * V;
      if (live && j0 < sk) {
        if constexpr (V >= 2) {
          const uint64_t inv2 = p2(inv, inv);
#pragma unroll
          for (int e = 0; e < V; e += 2) {
            const float2 f = u2(mul2(p2(u[k][e], u[k][e + 1]), inv2));
            u[k][e] = f.x;
            u[k][e + 1] = f.y;
          }
        } else {
          u[k][0] *= inv;
        }
        store_v<T, V>(yr + j0, u[k]);
      }
    }
  };

  uint32_t cw[NV][NW];
  uint64_t cm[NV];
  int cl = 0;
  if constexpr (NV < 8) {
    // One block per CTA.
    fetch(blockIdx.x, cw, cm, cl);
    compute(blockIdx.x, cw, cm, cl);
  } else {
    // Persistent, the next block's loads in flight during this one.
    int64_t blk = blockIdx.x;
    fetch(blk, cw, cm, cl);
    for (; blk < nblocks; blk += gridDim.x) {
      uint32_t nw[NV][NW];
      uint64_t nm[NV];
      int nl = 0;
      fetch(blk + gridDim.x, nw, nm, nl);
      compute(blk, cw, cm, cl);
#pragma unroll
      for (int k = 0; k < NV; ++k) {
#pragma unroll
        for (int e = 0; e < NW; ++e) cw[k][e] = nw[k][e];
        cm[k] = nm[k];
      }
      cl = nl;
    }
  }
}

struct SmBwdParams {
  const void* dy;
  const void* y;
  void* dx;
  int64_t rows;
  int sk;
  int wpr;
  float scale;
};

// Backward: y and dy stay packed in registers between the dot product and
// the output pass (widened twice), which keeps the register count low.
template <typename T, int V, int NV>
__global__ void __launch_bounds__(kSmThreads, 3) softmax_bwd_kernel(const SmBwdParams p) {
  pdl_begin();
  constexpr int NW = V == 1 ? 1 : 4;
  __shared__ float buf[kSmThreads / 32];
  const int gthreads = 32 * p.wpr;
  const int rows_per_cta = kSmThreads / gthreads;
  const int g = threadIdx.x / gthreads, t = threadIdx.x % gthreads;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rows_per_cta + g;
  const bool live = row < p.rows;
  const int sk = p.sk;
  const int64_t rr = live ? row : 0;
  const T* yr = reinterpret_cast<const T*>(p.y) + rr * sk;
  const T* dr = reinterpret_cast<const T*>(p.dy) + rr * sk;
  uint32_t yw[NV][NW], dw[NV][NW];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j0 = (k * gthreads + t) * V;
    if (live && j0 < sk) {
      load_words<T, V>(yr + j0, yw[k]);
      load_words<T, V>(dr + j0, dw[k]);
    } else {
#pragma unroll
      for (int e = 0; e < NW; ++e) yw[k][e] = dw[k][e] = 0u;
    }
  }
  float c = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    float yv[V], dv[V];
    words_to_floats<T, V>(yw[k], yv);
    words_to_floats<T, V>(dw[k], dv);
#pragma unroll
    for (int e = 0; e < V; ++e) c = fmaf(yv[e], dv[e], c);
  }
  c = group_reduce<false>(c, buf, p.wpr);
  T* xr = reinterpret_cast<T*>(p.dx) + rr * sk;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j0 = (k * gthreads + t) * V;
    if (live && j0 < sk) {
      float yv[V], dv[V], o[V];
      words_to_floats<T, V>(yw[k], yv);
      words_to_floats<T, V>(dw[k], dv);
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] = p.scale * yv[e] * (dv[e] - c);
      store_v<T, V>(xr + j0, o);
    }
  }
}

// ---- host side

// Loads per thread (NV) and warps per row (WPR) for a row of sk elements in
// loads of V: the smallest WPR (1..8) with NV <= 8, then the smallest NV.
bool sm_geom(int sk, int v, int* nv, int* wpr) {
  for (int w = 1; w <= kSmThreads / 32; w *= 2) {
    for (int n = 1; n <= 8; n *= 2) {
      if (static_cast<int64_t>(32) * w * n * v >= sk) {
        *nv = n;
        *wpr = w;
        return true;
      }
    }
  }
  return false;
}

using SmFwdKernel = void (*)(const SmFwdParams);

template <typename T, int V, int NV>
SmFwdKernel fwd_kernel_nv(int mask) {
  switch (mask) {
    case 0: return softmax_fwd_kernel<T, V, NV, 0>;
    case 1: return softmax_fwd_kernel<T, V, NV, 1>;
    case 2: return softmax_fwd_kernel<T, V, NV, 2>;
    default: return softmax_fwd_kernel<T, V, NV, 3>;
  }
}

template <typename T, int V>
SmFwdKernel fwd_kernel(int mask, int nv) {
  switch (nv) {
    case 1: return fwd_kernel_nv<T, V, 1>(mask);
    case 2: return fwd_kernel_nv<T, V, 2>(mask);
    case 4: return fwd_kernel_nv<T, V, 4>(mask);
    default: return fwd_kernel_nv<T, V, 8>(mask);
  }
}

// Resident CTAs per SM of a forward kernel (cached per device and kernel).
int fwd_ctas_per_sm(SmFwdKernel k) {
  static std::mutex mu;
  static std::map<std::pair<int, SmFwdKernel>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find({dev, k});
  if (it != cache.end()) return it->second;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kSmThreads, 0) != cudaSuccess)
    occ = 0;
  if (occ < 1) occ = 1;
  cache[{dev, k}] = occ;
  return occ;
}

template <typename T, int V>
cudaError_t launch_bwd(const SmBwdParams& p, int nv, int grid, cudaStream_t st) {
  const dim3 g(grid), b(kSmThreads);
  switch (nv) {
    case 1: return launch_pdl(softmax_bwd_kernel<T, V, 1>, g, b, 0, st, p);
    case 2: return launch_pdl(softmax_bwd_kernel<T, V, 2>, g, b, 0, st, p);
    case 4: return launch_pdl(softmax_bwd_kernel<T, V, 4>, g, b, 0, st, p);
    default: return launch_pdl(softmax_bwd_kernel<T, V, 8>, g, b, 0, st, p);
  }
}

int sm_esize(gbn_dtype d) { return d == GBN_F32 ? 4 : 2; }


bool sm_aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gbn

using namespace gbn;

extern "C" {

gbn_status gbn_softmax_fwd(const void* x, const uint8_t* mask, void* y, int64_t batches,
                           int64_t heads, int64_t sq, int64_t sk, int64_t mask_batches,
                           gbn_dtype dtype, gbn_softmax_mask mask_kind, float scale,
                           cudaStream_t stream) {
  if (dtype != GBN_F32 && dtype != GBN_BF16 && dtype != GBN_F16) return GBN_ERR_DTYPE;
  if (mask_kind < GBN_SOFTMAX_NO_MASK || mask_kind > GBN_SOFTMAX_CAUSAL_ALIGNED) return GBN_ERR_ENUM;
  if (batches < 0 || heads < 0 || sq < 0 || sk < 1 || sk > kMaxSoftmaxKeys) return GBN_ERR_SHAPE;
  if (mask_kind == GBN_SOFTMAX_CAUSAL_UPPER && sq != sk) return GBN_ERR_SHAPE;
  const int64_t rows = batches * heads * sq;
  if (rows == 0) return GBN_OK;
  if (!x || !y) return GBN_ERR_NULL;
  if (mask_kind == GBN_SOFTMAX_PADDING && (!mask || mask_batches < 1)) return GBN_ERR_NULL;
  const int vec = 16 / sm_esize(dtype);
  const bool vok = sk % vec == 0 && sm_aligned(x) && sm_aligned(y) &&
                   (mask_kind != GBN_SOFTMAX_PADDING || sm_aligned(mask));
  int nv = 0, wpr = 0;
  if (!sm_geom(static_cast<int>(sk), vok ? vec : 1, &nv, &wpr)) return GBN_ERR_SHAPE;
  SmFwdParams p{x, mask, y, rows, heads * sq, sq, mask_batches, static_cast<int>(sk), wpr,
                scale * kLog2e};
  const int m = static_cast<int>(mask_kind);
  SmFwdKernel k;
  if (dtype == GBN_F32)
    k = vok ? fwd_kernel<float, 4>(m, nv) : fwd_kernel<float, 1>(m, nv);
  else if (dtype == GBN_BF16)
    k = vok ? fwd_kernel<__nv_bfloat16, 8>(m, nv) : fwd_kernel<__nv_bfloat16, 1>(m, nv);
  else
    k = vok ? fwd_kernel<__half, 8>(m, nv) : fwd_kernel<__half, 1>(m, nv);
  const int64_t rows_per_cta = kSmThreads / (32 * wpr);
  int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  // NV = 8: persistent, at most the CTAs that are resident at once.
  if (nv == 8) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GBN_ERR_CUDA;
    const int64_t resident = static_cast<int64_t>(sms) * fwd_ctas_per_sm(k);
    if (grid > resident) grid = resident;
  }
  if (grid > 0x7FFFFFFF) return GBN_ERR_SHAPE;
  const cudaError_t e =
      launch_pdl(k, dim3(static_cast<unsigned>(grid)), dim3(kSmThreads), 0, stream, p);
  return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
}

gbn_status gbn_softmax_bwd(const void* dy, const void* y, void* dx, int64_t rows, int64_t sk,
                           gbn_dtype dtype, float scale, cudaStream_t stream) {
  if (dtype != GBN_F32 && dtype != GBN_BF16 && dtype != GBN_F16) return GBN_ERR_DTYPE;
  if (rows < 0 || sk < 1 || sk > kMaxSoftmaxKeys) return GBN_ERR_SHAPE;
  if (rows == 0) return GBN_OK;
  if (!dy || !y || !dx) return GBN_ERR_NULL;
  const int vec = 16 / sm_esize(dtype);
  const bool vok = sk % vec == 0 && sm_aligned(dy) && sm_aligned(y) && sm_aligned(dx);
  int nv = 0, wpr = 0;
  if (!sm_geom(static_cast<int>(sk), vok ? vec : 1, &nv, &wpr)) return GBN_ERR_SHAPE;
  // Two packed rows per load stay in registers: at most 4 loads per thread
  // (more warps per row instead), so the kernel keeps three CTAs per SM.
  if (nv == 8 && wpr < kSmThreads / 32) {
    nv = 4;
    wpr *= 2;
  }
  SmBwdParams p{dy, y, dx, rows, static_cast<int>(sk), wpr, scale};
  const int64_t rows_per_cta = kSmThreads / (32 * wpr);
  const int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7FFFFFFF) return GBN_ERR_SHAPE;
  const int g = static_cast<int>(grid);
  cudaError_t e;
  if (dtype == GBN_F32)
    e = vok ? launch_bwd<float, 4>(p, nv, g, stream) : launch_bwd<float, 1>(p, nv, g, stream);
  else if (dtype == GBN_BF16)
    e = vok ? launch_bwd<__nv_bfloat16, 8>(p, nv, g, stream)
            : launch_bwd<__nv_bfloat16, 1>(p, nv, g, stream);
  else
    e = vok ? launch_bwd<__half, 8>(p, nv, g, stream) : launch_bwd<__half, 1>(p, nv, g, stream);
  return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
}

}  // extern "C"
