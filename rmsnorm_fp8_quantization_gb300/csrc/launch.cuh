// Host-side launch templates, explicitly instantiated once per input dtype
// (kernels_f32.cu, kernels_bf16.cu, kernels_f16.cu) so the three translation
// units compile in parallel.
#pragma once

#include "bwd.cuh"
#include "fwd_row.cuh"
#include "fwd_stripe.cuh"

namespace gbn {

template <typename Tin>
struct Launch {
  using Kfwd = void (*)(const FwdParams);
  using Kbwd = void (*)(const BwdParams);
  using Kstripe = void (*)(const FwdParams, const int);

  template <int QM>
  static Kfwd fwd_row_kernel_for(const RowGeom& g) {
    if (g.vec == 1) return fwd_generic_kernel<Tin, QM>;
    switch (g.nv) {
      case 1: return fwd_row_kernel<Tin, QM, 1>;
      case 2: return fwd_row_kernel<Tin, QM, 2>;
      case 4: return fwd_row_kernel<Tin, QM, 4>;
      case 8: return fwd_row_kernel<Tin, QM, 8>;
      default: return nullptr;
    }
  }
  static Kfwd fwd_kernel(int qm, const RowGeom& g) {
    switch (qm) {
      case Q_NONE: return fwd_row_kernel_for<Q_NONE>(g);
      case Q_DELAYED: return fwd_row_kernel_for<Q_DELAYED>(g);
      case Q_MXFP8: return fwd_row_kernel_for<Q_MXFP8>(g);
      default: return nullptr;
    }
  }

  template <int QM>
  static Kstripe stripe_kernel_for(int nvs) {
    switch (nvs) {
      case 1: return fwd_stripe_kernel<Tin, QM, 1>;
      case 2: return fwd_stripe_kernel<Tin, QM, 2>;
      case 4: return fwd_stripe_kernel<Tin, QM, 4>;
      case 8: return fwd_stripe_kernel<Tin, QM, 8>;
      default: return nullptr;
    }
  }
  static Kstripe stripe_kernel(int qm, int nvs) {
    if (qm == Q_DELAYED) return stripe_kernel_for<Q_DELAYED>(nvs);
    if (qm == Q_MXFP8) return stripe_kernel_for<Q_MXFP8>(nvs);
    return nullptr;
  }

  template <bool LN, bool ADD>
  static Kbwd bwd_kernel_for(const RowGeom& g) {
    if (g.vec == 1) return bwd_generic_kernel<Tin>;
    switch (g.nv) {
      case 1: return bwd_row_kernel<Tin, LN, ADD, 1>;
      case 2: return bwd_row_kernel<Tin, LN, ADD, 2>;
      case 4: return bwd_row_kernel<Tin, LN, ADD, 4>;
      case 8: return bwd_row_kernel<Tin, LN, ADD, 8>;
      default: return nullptr;
    }
  }
  static Kbwd bwd_kernel(bool ln, bool add, const RowGeom& g) {
    if (ln) return add ? bwd_kernel_for<true, true>(g) : bwd_kernel_for<true, false>(g);
    return add ? bwd_kernel_for<false, true>(g) : bwd_kernel_for<false, false>(g);
  }

  static cudaError_t fwd_occupancy(int qm, const RowGeom& g, int* occ) {
    Kfwd k = fwd_kernel(qm, g);
    if (!k) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, g.vec == 1 ? 256 : g.threads, 0);
  }
  static cudaError_t fwd_launch(int qm, const RowGeom& g, const FwdParams& p, int grid,
                                cudaStream_t st) {
    Kfwd k = fwd_kernel(qm, g);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, g.vec == 1 ? 256 : g.threads, 0, st>>>(p);
    return cudaGetLastError();
  }

  static cudaError_t stripe_launch(int qm, const StripeGeom& g, const FwdParams& p,
                                   double sm_fraction, cudaStream_t st) {
    Kstripe k = stripe_kernel(qm, g.nvs);
    if (!k) return cudaErrorInvalidValue;
    const int smem = stripe_smem_bytes(qm, g.hc);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t nstripes = p.rows / kStripeRows;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(g.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kStripeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent grid: as many clusters as fit at once (scaled by the SM share
    // left after sm_margin), never more than there are stripes.
    cfg.gridDim = dim3(static_cast<unsigned>(g.cluster) * 152u, 1, 1);
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg);
    if (e != cudaSuccess) return e;
    int64_t ncl = static_cast<int64_t>(max_clusters * sm_fraction);
    if (ncl < 1) ncl = 1;
    if (ncl > nstripes) ncl = nstripes > 0 ? nstripes : 1;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * g.cluster), 1, 1);
    e = cudaLaunchKernelEx(&cfg, k, p, g.hc);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }

  static cudaError_t bwd_occupancy(bool ln, bool add, const RowGeom& g, int* occ) {
    Kbwd k = bwd_kernel(ln, add, g);
    if (!k) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, g.vec == 1 ? 256 : g.threads, 0);
  }
  static cudaError_t bwd_launch(bool ln, bool add, const RowGeom& g, const BwdParams& p, int grid,
                                cudaStream_t st) {
    Kbwd k = bwd_kernel(ln, add, g);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, g.vec == 1 ? 256 : g.threads, 0, st>>>(p);
    return cudaGetLastError();
  }
};

}  // namespace gbn
