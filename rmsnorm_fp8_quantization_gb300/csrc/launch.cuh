// Host-side launch templates, explicitly instantiated once per input dtype
// (kernels_f32.cu, kernels_bf16.cu, kernels_f16.cu) so the three translation
// units compile in parallel.
#pragma once

#include "bwd.cuh"
#include "cluster_row.cuh"
#include "fwd_colwise.cuh"
#include "fwd_row.cuh"
#include "fwd_stripe.cuh"
#include "ring.cuh"

namespace gbn {

template <typename Tin>
struct Launch {
  using Kfwd = void (*)(const FwdParams);
  using Kbwd = void (*)(const BwdParams);

  static Kfwd fwd_generic(int qm) {
    if (qm == Q_NONE) return fwd_generic_kernel<Tin, Q_NONE>;
    if (qm == Q_DELAYED) return fwd_generic_kernel<Tin, Q_DELAYED>;
    if (qm == Q_MXFP8) return fwd_generic_kernel<Tin, Q_MXFP8>;
    return nullptr;
  }
  static cudaError_t fwd_generic_occupancy(int qm, int* occ) {
    Kfwd k = fwd_generic(qm);
    return k ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, 256, 0) : cudaErrorInvalidValue;
  }
  static cudaError_t fwd_generic_launch(int qm, const FwdParams& p, int grid, cudaStream_t st) {
    Kfwd k = fwd_generic(qm);
    if (!k) return cudaErrorInvalidValue;
    return launch_pdl(k, dim3(grid), dim3(256), 0, st, p);
  }
  using Kcol = void (*)(const FwdParams, const float*, const float*);
  static Kcol colwise(int qm, bool ln) {
    if (qm == Q_DELAYED) return ln ? fwd_colwise_kernel<Tin, Q_DELAYED, true>
                                   : fwd_colwise_kernel<Tin, Q_DELAYED, false>;
    if (qm == Q_MXFP8) return ln ? fwd_colwise_kernel<Tin, Q_MXFP8, true>
                                 : fwd_colwise_kernel<Tin, Q_MXFP8, false>;
    return nullptr;
  }
  static cudaError_t colwise_occupancy(int qm, bool ln, int* occ) {
    Kcol k = colwise(qm, ln);
    return k ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kColTileThreads, 0)
             : cudaErrorInvalidValue;
  }
  static cudaError_t colwise_launch(int qm, bool ln, const FwdParams& p, const float* mu,
                                    const float* rs, int grid, cudaStream_t st) {
    Kcol k = colwise(qm, ln);
    if (!k) return cudaErrorInvalidValue;
    return launch_pdl(k, dim3(grid), dim3(kColTileThreads), 0, st, p, mu, rs);
  }
  static cudaError_t bwd_generic_occupancy(int* occ) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, bwd_generic_kernel<Tin>, 256, 0);
  }
  static cudaError_t bwd_generic_launch(const BwdParams& p, int grid, cudaStream_t st) {
    return launch_pdl(bwd_generic_kernel<Tin>, dim3(grid), dim3(256), 0, st, p);
  }

  using Kstripe3 = void (*)(const FwdParams, const int, const int);
  static Kstripe3 stripe_kernel(int qm, bool ln) {
    if (qm == Q_DELAYED) return ln ? fwd_stripe_kernel<Tin, Q_DELAYED, true>
                                   : fwd_stripe_kernel<Tin, Q_DELAYED, false>;
    if (qm == Q_MXFP8) return ln ? fwd_stripe_kernel<Tin, Q_MXFP8, true>
                                 : fwd_stripe_kernel<Tin, Q_MXFP8, false>;
    return nullptr;
  }
  // attr[0]: cluster shape; attr[1] (launches only): programmatic dependent launch
  static void stripe_config(const StripeGeom& g, int nclusters, cudaLaunchConfig_t* cfg,
                            cudaLaunchAttribute* attr) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(g.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(nclusters * g.cluster), 1, 1);
    cfg->blockDim = dim3(kStripeThreads, 1, 1);
    cfg->dynamicSmemBytes = static_cast<size_t>(g.smem);
    cfg->attrs = attr;
    cfg->numAttrs = 1;
  }
  static cudaError_t stripe_max_clusters(int qm, bool ln, const StripeGeom& g, int* n) {
    Kstripe3 k = stripe_kernel(qm, ln);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    stripe_config(g, 960 / g.cluster, &cfg, attr);
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
  }
  static cudaError_t stripe_launch(int qm, bool ln, const StripeGeom& g, const FwdParams& p,
                                   int nclusters, cudaStream_t st) {
    Kstripe3 k = stripe_kernel(qm, ln);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    stripe_config(g, nclusters, &cfg, attr);
    cfg.numAttrs = 2;
    cfg.stream = st;
    e = cudaLaunchKernelEx(&cfg, k, p, g.hc, g.stages);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }

  // ---- bulk-copy ring variants
  using Kring = void (*)(const FwdParams, const int);
  using Kbring = void (*)(const BwdParams, const int);

  template <int QM, bool LN>
  static Kring fwd_ring_for(int nv) {
    switch (nv) {
      case 1: return fwd_ring_kernel<Tin, QM, LN, 1>;
      case 2: return fwd_ring_kernel<Tin, QM, LN, 2>;
      case 3: return fwd_ring_kernel<Tin, QM, LN, 3>;
      case 4: return fwd_ring_kernel<Tin, QM, LN, 4>;
      case 6: return fwd_ring_kernel<Tin, QM, LN, 6>;
      case 8: return fwd_ring_kernel<Tin, QM, LN, 8>;
      default: return nullptr;
    }
  }
  // kind = qm * 2 + (layernorm ? 1 : 0)
  // kinds 7, 9, 11: LayerNorm with the one-pass merge (NV = 4 only: the
  // one geometry of the forward ring where it applies)
  static Kring fwd_ring(int kind, int nv) {
    if (kind >= 6) {
      if (nv != 4) return nullptr;
      switch (kind) {
        case 7: return fwd_ring_kernel<Tin, Q_NONE, true, 4, true>;
        case 9: return fwd_ring_kernel<Tin, Q_DELAYED, true, 4, true>;
        case 11: return fwd_ring_kernel<Tin, Q_MXFP8, true, 4, true>;
        default: return nullptr;
      }
    }
    switch (kind) {
      case 0: return fwd_ring_for<Q_NONE, false>(nv);
      case 1: return fwd_ring_for<Q_NONE, true>(nv);
      case 2: return fwd_ring_for<Q_DELAYED, false>(nv);
      case 3: return fwd_ring_for<Q_DELAYED, true>(nv);
      case 4: return fwd_ring_for<Q_MXFP8, false>(nv);
      case 5: return fwd_ring_for<Q_MXFP8, true>(nv);
      default: return nullptr;
    }
  }
  template <bool LN, bool ADD>
  static Kbring bwd_ring_for(int nv) {
    switch (nv) {
      case 1: return bwd_ring_kernel<Tin, LN, ADD, 1>;
      case 2: return bwd_ring_kernel<Tin, LN, ADD, 2>;
      case 3: return bwd_ring_kernel<Tin, LN, ADD, 3>;
      case 4: return bwd_ring_kernel<Tin, LN, ADD, 4>;
      case 6: return bwd_ring_kernel<Tin, LN, ADD, 6>;
      case 8: return bwd_ring_kernel<Tin, LN, ADD, 8>;
      default: return nullptr;
    }
  }
  static Kbring bwd_ring(bool ln, bool add, int nv) {
    if (ln) return add ? bwd_ring_for<true, true>(nv) : bwd_ring_for<true, false>(nv);
    return add ? bwd_ring_for<false, true>(nv) : bwd_ring_for<false, false>(nv);
  }
  template <typename K>
  static cudaError_t occ_smem(K k, int threads, int smem, int* occ) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, threads, smem);
  }
  static cudaError_t fwd_ring_occupancy(int qm, const RowGeom& g, int smem, int* occ) {
    Kring k = fwd_ring(qm, g.nv);
    return k ? occ_smem(k, g.threads, smem, occ) : cudaErrorInvalidValue;
  }
  static cudaError_t fwd_ring_launch(int qm, const RowGeom& g, int stages, int smem,
                                     const FwdParams& p, int grid, cudaStream_t st) {
    Kring k = fwd_ring(qm, g.nv);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(g.threads), smem, st, p, stages);
  }
  static cudaError_t bwd_ring_occupancy(bool ln, bool add, const RowGeom& g, int smem, int* occ) {
    Kbring k = bwd_ring(ln, add, g.nv);
    return k ? occ_smem(k, g.threads, smem, occ) : cudaErrorInvalidValue;
  }
  static cudaError_t bwd_ring_launch(bool ln, bool add, const RowGeom& g, int stages, int smem,
                                     const BwdParams& p, int grid, cudaStream_t st) {
    Kbring k = bwd_ring(ln, add, g.nv);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(g.threads), smem, st, p, stages);
  }
  // ---- long rows: a row split over a thread-block cluster
  using Kcl = void (*)(const FwdParams, const int, const int);
  static Kcl fwd_cluster(int kind) {
    constexpr int NV = kClusterFwdNv;
    switch (kind) {
      case 0: return fwd_cluster_kernel<Tin, Q_NONE, false, NV>;
      case 1: return fwd_cluster_kernel<Tin, Q_NONE, true, NV>;
      case 2: return fwd_cluster_kernel<Tin, Q_DELAYED, false, NV>;
      case 3: return fwd_cluster_kernel<Tin, Q_DELAYED, true, NV>;
      case 4: return fwd_cluster_kernel<Tin, Q_MXFP8, false, NV>;
      case 5: return fwd_cluster_kernel<Tin, Q_MXFP8, true, NV>;
      default: return nullptr;
    }
  }
  // attr[0]: cluster shape; attr[1] (launches only): programmatic dependent launch
  static void cluster_config(int cluster, int nclusters, int threads, int smem,
                             cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(nclusters * cluster), 1, 1);
    cfg->blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg->dynamicSmemBytes = static_cast<size_t>(smem);
    cfg->attrs = attr;
    cfg->numAttrs = 1;
  }
  static cudaError_t fwd_cluster_max_clusters(int kind, int cluster, int threads, int smem,
                                              int* n) {
    Kcl k = fwd_cluster(kind);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cluster, 1024 / cluster, threads, smem, &cfg, attr);
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
  }
  static cudaError_t fwd_cluster_launch(int kind, int cluster, int threads, int stages, int smem,
                                        int hc, const FwdParams& p, int nclusters,
                                        cudaStream_t st) {
    Kcl k = fwd_cluster(kind);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cluster, nclusters, threads, smem, &cfg, attr);
    cfg.numAttrs = 2;
    cfg.stream = st;
    e = cudaLaunchKernelEx(&cfg, k, p, stages, hc);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }

  using Kbcl = void (*)(const BwdParams, const int, const int);
  static Kbcl bwd_cluster(bool ln, bool add) {
    constexpr int NV = kClusterBwdNv;
    if (ln) return add ? bwd_cluster_kernel<Tin, true, true, NV> : bwd_cluster_kernel<Tin, true, false, NV>;
    return add ? bwd_cluster_kernel<Tin, false, true, NV> : bwd_cluster_kernel<Tin, false, false, NV>;
  }
  static cudaError_t bwd_cluster_max_clusters(bool ln, bool add, int cluster, int threads,
                                              int smem, int* n) {
    Kbcl k = bwd_cluster(ln, add);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cluster, 1024 / cluster, threads, smem, &cfg, attr);
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
  }
  static cudaError_t bwd_cluster_launch(bool ln, bool add, int cluster, int threads, int stages,
                                        int smem, int hc, const BwdParams& p, int nclusters,
                                        cudaStream_t st) {
    Kbcl k = bwd_cluster(ln, add);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cluster, nclusters, threads, smem, &cfg, attr);
    cfg.numAttrs = 2;
    cfg.stream = st;
    e = cudaLaunchKernelEx(&cfg, k, p, stages, hc);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }

  static cudaError_t probe_copy_timeout(unsigned long long limit_ns, cudaStream_t st) {
    return launch_pdl(copy_timeout_probe_kernel, dim3(1), dim3(32), 0, st, limit_ns);
  }

  static cudaError_t read_device_error(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_gbn_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_gbn_device_error, &zero, sizeof(unsigned int));
  }

};

}  // namespace gbn
