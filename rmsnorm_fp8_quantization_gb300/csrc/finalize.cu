// Backward finalize launch.
#include "bwd.cuh"

namespace gbn {

// Finalize: dgamma[j] = sum_{b < P} part[b][j] in a fixed order, cast to the
// weight dtype (blockIdx.y = 0: dgamma, 1: dbeta).  A CTA takes 64 columns;
// warp w sums parts w, w+8, ... and the 8 warp sums are added in warp order.
__global__ void __launch_bounds__(256) bwd_finalize_kernel(const FinalizeParams p) {
  __shared__ float2 acc[8][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* part = blockIdx.y == 0 ? p.part_dgamma : p.part_dbeta;
  void* outp = blockIdx.y == 0 ? p.dgamma : p.dbeta;
  const int H = p.hidden;
  const int col = blockIdx.x * 64 + 2 * lane;
  const bool pair = (H % 2 == 0);
  float2 a = make_float2(0.f, 0.f);
  for (int b = warp; b < p.parts; b += 8) {
    const float* r = part + static_cast<int64_t>(b) * H;
    if (pair) {
      if (col < H) {
        const float2 v = *reinterpret_cast<const float2*>(r + col);
        a.x += v.x;
        a.y += v.y;
      }
    } else {
      if (col < H) a.x += r[col];
      if (col + 1 < H) a.y += r[col + 1];
    }
  }
  acc[warp][lane] = a;
  __syncthreads();
  if (warp == 0) {
    float2 t = acc[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      t.x += acc[w][lane].x;
      t.y += acc[w][lane].y;
    }
    if (col < H) st_weight_scalar(outp, p.w_dt, col, t.x);
    if (col + 1 < H) st_weight_scalar(outp, p.w_dt, col + 1, t.y);
  }
}

cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream) {
  const dim3 grid((p.hidden + 63) / 64, p.part_dbeta ? 2 : 1, 1);
  bwd_finalize_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gbn
