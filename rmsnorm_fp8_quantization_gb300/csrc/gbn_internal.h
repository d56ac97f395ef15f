// Internal parameter blocks and launcher declarations shared by the C-ABI
// layer (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gbn {

enum Dt : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum Qm : int { Q_NONE = 0, Q_DELAYED = 1, Q_MXFP8 = 2 };

struct FwdParams {
  const void* x;
  const void* gamma;
  const void* beta;          // LayerNorm only
  const float* scale;        // delayed
  void* out;                 // rowwise output (in dtype or E4M3), may be null for colwise-only
  uint8_t* colwise_out;      // delayed: [hidden, rows]; MXFP8: [rows, hidden]
  float* mu;                 // may be null
  float* rsigma;             // may be null
  float* scale_inv;          // delayed rowwise 1/scale
  float* colwise_scale_inv;  // delayed colwise 1/scale
  uint8_t* mx_scale;         // MXFP8 rowwise E8M0 [rows, hidden/32]
  uint8_t* mx_colwise_scale; // MXFP8 colwise E8M0 [rows/32, hidden]
  float* amax;               // delayed updated amax (zeroed before the launch)
  int64_t rows;
  int hidden;
  float eps;
  int norm;                  // 0 LayerNorm, 1 RMSNorm
  int zcg;                   // zero-centered gamma
  int w_dt;                  // weight dtype (Dt)
  int write_rowwise;
  int write_colwise;
};

struct BwdParams {
  const void* dz;
  const void* x;
  const float* mu;           // LayerNorm
  const float* rsigma;
  const void* gamma;
  const void* dres;          // null: no add
  void* dx;
  float* part_dgamma;        // workspace [P, hidden]
  float* part_dbeta;         // workspace [P, hidden] (LayerNorm)
  int64_t rows;
  int hidden;
  int norm;
  int zcg;
  int w_dt;
};

struct FinalizeParams {
  const float* part_dgamma;
  const float* part_dbeta;   // null for RMSNorm
  void* dgamma;
  void* dbeta;
  int parts;
  int hidden;
  int w_dt;
};

// Launch geometry chosen by the host layer.
struct RowGeom {
  int vec;      // elements per vector: 16 bytes of the input type, or 1 (scalar path)
  int nv;       // vectors per thread per row (1, 2, 4, 8)
  int threads;  // CTA size (multiple of 32, <= 1024)
};

struct StripeGeom {
  int vec;      // as above
  int nvs;      // vectors per lane per row slice (1, 2, 4, 8)
  int cluster;  // CTAs per cluster (1..8); each takes hidden/cluster columns
  int hc;       // columns per CTA
};

// Largest CTA of the backward row pass with NV vectors per thread: the
// register budget per thread grows with NV (dgamma/dbeta partials live in
// registers), so the CTA shrinks.
constexpr int bwd_max_threads(int nv) {
  return nv <= 1 ? 1024 : (nv == 2 ? 768 : (nv == 4 ? 512 : 256));
}

// Launchers of one input dtype (one translation unit each).  Every function
// returns the cudaError_t of the CUDA calls it made.
struct KernelTable {
  // Occupancy (CTAs per SM) of the rowwise forward variant for geometry g.
  cudaError_t (*fwd_occupancy)(int qm, const RowGeom& g, int* blocks_per_sm);
  // Rowwise forward (vectorized row pass, or the generic kernel when g.vec == 1;
  // the generic kernel also writes every columnwise layout).
  cudaError_t (*fwd_launch)(int qm, const RowGeom& g, const FwdParams& p, int grid,
                            cudaStream_t stream);
  // Columnwise (and rowwise) forward over 32-row stripes split across a
  // thread-block cluster; sm_fraction scales the co-resident cluster count.
  cudaError_t (*stripe_launch)(int qm, const StripeGeom& g, const FwdParams& p,
                               double sm_fraction, cudaStream_t stream);
  cudaError_t (*bwd_occupancy)(bool layernorm, bool add, const RowGeom& g, int* blocks_per_sm);
  cudaError_t (*bwd_launch)(bool layernorm, bool add, const RowGeom& g, const BwdParams& p,
                            int grid, cudaStream_t stream);
};

const KernelTable& kernels_f32();
const KernelTable& kernels_bf16();
const KernelTable& kernels_f16();

// Finalize pass of the backward (sums the per-CTA partials).
cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream);

}  // namespace gbn
