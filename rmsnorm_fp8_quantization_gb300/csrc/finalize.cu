// Backward finalize launch.
#include "bwd.cuh"

namespace gbn {

// Finalize: dgamma[j] = sum_{b < P} part[b][j] in a fixed order, cast to the
// weight dtype (blockIdx.y = 0: dgamma, 1: dbeta).  A CTA takes 32 columns
// (one per lane) with W = clamp(ceil(P / 16), 1, 32) warps: warp w loads
// parts w, w + W, ..., w + 15W at once (16 loads in flight, predicated past
// P), so that one round of loads covers up to 16W parts; the 16 sums of a
// warp combine as a tree, the W warp sums in warp order over four running
// sums.  W depends on P only: the same call always adds in the same order.
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
  constexpr int U = 16;
  float a[U];
#pragma unroll
  for (int u = 0; u < U; ++u) a[u] = 0.f;
  for (int b = warp; b < p.parts; b += U * nw) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = b + u * nw;
      v[u] = r < p.parts ? base[static_cast<int64_t>(r) * H] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] += v[u];
  }
#pragma unroll
  for (int s2 = U / 2; s2 > 0; s2 >>= 1) {
#pragma unroll
    for (int u = 0; u < s2; ++u) a[u] += a[u + s2];
  }
  acc[warp][lane] = a[0];
  __syncthreads();
  if (warp == 0) {
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    int w = 0;
    for (; w + 3 < nw; w += 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) t[j] += acc[w + j][lane];
    }
    for (; w < nw; ++w) t[0] += acc[w][lane];
    if (in) st_weight_scalar(outp, p.w_dt, col, (t[0] + t[1]) + (t[2] + t[3]));
  }
}

cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream) {
  int warps = (p.parts + 15) / 16;
  warps = warps < 1 ? 1 : (warps > kFinWarps ? kFinWarps : warps);
  const dim3 grid((p.hidden + kFinCols - 1) / kFinCols, p.part_dbeta ? 2 : 1, 1);
  return launch_pdl(bwd_finalize_kernel, grid, dim3(warps * 32), 0, stream, p);
}

}  // namespace gbn
