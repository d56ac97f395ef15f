// Backward finalize launch.
#include "bwd.cuh"

namespace gbn {

// Finalize: dgamma[j] = sum_{b < P} part[b][j] in a fixed order, cast to the
// weight dtype (blockIdx.y = 0: dgamma, 1: dbeta).  A CTA takes 32 columns
// (one per lane) with W = clamp(ceil(P / 8), 1, 32) warps, so that each warp
// has about eight partial rows to add: warp w sums parts w, w + W, ... with
// eight loads in flight (eight accumulators, combined in a fixed order), and
// the W warp sums are added in warp order.  W depends on P only: the same
// call always adds in the same order.
constexpr int kFinWarps = 32;
constexpr int kFinCols = 32;

__global__ void __launch_bounds__(kFinWarps * 32) bwd_finalize_kernel(const FinalizeParams p) {
  pdl_begin();
  __shared__ float acc[kFinWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const float* part = blockIdx.y == 0 ? p.part_dgamma : p.part_dbeta;
  void* outp = blockIdx.y == 0 ? p.dgamma : p.dbeta;
  const int H = p.hidden;
  const int col = blockIdx.x * kFinCols + lane;
  const bool in = col < H;
  const float* base = part + (in ? col : 0);
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int b = warp;
  for (; b + 7 * nw < p.parts; b += 8 * nw) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = base[static_cast<int64_t>(b + u * nw) * H];
#pragma unroll
    for (int u = 0; u < 8; ++u) a[u] += v[u];
  }
  for (; b < p.parts; b += nw) a[0] += base[static_cast<int64_t>(b) * H];
  acc[warp][lane] = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  __syncthreads();
  if (warp == 0) {
    float t = acc[0][lane];
    for (int w = 1; w < nw; ++w) t += acc[w][lane];
    if (in) st_weight_scalar(outp, p.w_dt, col, t);
  }
}

cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream) {
  int warps = (p.parts + 7) / 8;
  warps = warps < 1 ? 1 : (warps > kFinWarps ? kFinWarps : warps);
  const dim3 grid((p.hidden + kFinCols - 1) / kFinCols, p.part_dbeta ? 2 : 1, 1);
  return launch_pdl(bwd_finalize_kernel, grid, dim3(warps * 32), 0, stream, p);
}

}  // namespace gbn
