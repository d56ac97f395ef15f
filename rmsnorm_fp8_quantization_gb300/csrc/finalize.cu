// Backward finalize launch.
#include "bwd.cuh"

namespace gbn {

// Finalize: dgamma[j] = sum_{b < P} part[b][j] in a fixed order, cast to the
// weight dtype (blockIdx.y = 0: dgamma, 1: dbeta).  A CTA takes 64 columns
// (a float2 per lane); warp w sums parts w, w + 16, ... with four loads in
// flight (four accumulators, combined in a fixed order), and the 16 warp sums
// are added in warp order.
constexpr int kFinWarps = 16;

__global__ void __launch_bounds__(kFinWarps * 32) bwd_finalize_kernel(const FinalizeParams p) {
  __shared__ float2 acc[kFinWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* part = blockIdx.y == 0 ? p.part_dgamma : p.part_dbeta;
  void* outp = blockIdx.y == 0 ? p.dgamma : p.dbeta;
  const int H = p.hidden;
  const int col = blockIdx.x * 64 + 2 * lane;
  const bool pair = (H % 2 == 0);
  auto load = [&](int b) -> float2 {
    const float* r = part + static_cast<int64_t>(b) * H;
    if (pair) {
      return col < H ? *reinterpret_cast<const float2*>(r + col) : make_float2(0.f, 0.f);
    }
    return make_float2(col < H ? r[col] : 0.f, col + 1 < H ? r[col + 1] : 0.f);
  };
  float2 a[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                 make_float2(0.f, 0.f)};
  int b = warp;
  for (; b + 3 * kFinWarps < p.parts; b += 4 * kFinWarps) {
    float2 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = load(b + u * kFinWarps);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u].x += v[u].x;
      a[u].y += v[u].y;
    }
  }
  for (; b < p.parts; b += kFinWarps) {
    const float2 v = load(b);
    a[0].x += v.x;
    a[0].y += v.y;
  }
  acc[warp][lane] = make_float2((a[0].x + a[1].x) + (a[2].x + a[3].x),
                                (a[0].y + a[1].y) + (a[2].y + a[3].y));
  __syncthreads();
  if (warp == 0) {
    float2 t = acc[0][lane];
#pragma unroll
    for (int w = 1; w < kFinWarps; ++w) {
      t.x += acc[w][lane].x;
      t.y += acc[w][lane].y;
    }
    if (col < H) st_weight_scalar(outp, p.w_dt, col, t.x);
    if (col + 1 < H) st_weight_scalar(outp, p.w_dt, col + 1, t.y);
  }
}

cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream) {
  const dim3 grid((p.hidden + 63) / 64, p.part_dbeta ? 2 : 1, 1);
  bwd_finalize_kernel<<<grid, kFinWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gbn
