// Internal parameter blocks and launcher declarations shared by the C-ABI
// layer (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gbn {

// Launches `k` with programmatic dependent launch allowed: it may begin
// launching while the previous kernel of the stream finishes; the kernels
// order their global-memory accesses with griddepcontrol (pdl_begin).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

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
  int mx_swizzle;            // MXFP8 scales in the padded 128x4-tiled GEMM order
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
  int vec;      // elements per vector: 16 bytes of the input type, or 1 (generic path)
  int nv;       // vectors per thread per row (1, 2, 3, 4, 6, 8)
  int threads;  // CTA size (multiple of 32, <= 1024)
};

struct StripeGeom {
  int cluster;  // CTAs per cluster (1..8); each takes hidden/cluster columns
  int hc;       // columns per CTA
  int stages;   // 32-row slices of x in shared memory (1 or 2)
  int smem;     // dynamic shared memory bytes
  int max_clusters;  // co-resident clusters of this geometry on the device
};

// Largest CTA of the backward row pass with NV vectors per thread: the
// register budget per thread grows with NV (dgamma/dbeta partials live in
// registers), so the CTA shrinks.
constexpr int bwd_max_threads(int nv) {
  return nv <= 1 ? 1024 : nv <= 3 ? 512 : nv == 4 ? 384 : 256;
}

// Largest CTA of the forward ring kernel with NV vectors per thread.
constexpr int fwd_ring_max_threads(int nv) {
  return nv <= 1 ? 1024 : nv == 2 ? 768 : nv == 3 ? 640 : nv == 4 ? 512 : nv == 6 ? 384 : 256;
}

// Bytes of one stage of the forward ring: the NV * threads vectors a CTA
// covers, rounded up to 128 bytes.  The tail past the row stays zero, so the
// row loop reads every vector without a bounds test.
__host__ __device__ constexpr int ring_slot_bytes(int nv, int threads) { return (nv * threads * 16 + 127) / 128 * 128; }

constexpr int kStripeRows = 32;
constexpr int kStripeThreads = 256;

// Dynamic shared memory of the stripe kernel: `stages` x 32-row slices of x
// (rows 16 bytes apart beyond their length), the statistics pushed by the
// cluster's CTAs (two stripes x `cluster` senders x 32 rows of float2),
// then the CTA's weights (g' and, for LayerNorm, beta; fp32).
inline int stripe_smem_bytes(int qm, bool ln, int hc, int esize, int stages, int cluster) {
  (void)qm;
  return stages * kStripeRows * (hc * esize + 16) + 2 * cluster * kStripeRows * 8 +
         (ln ? 8 : 4) * hc;
}

// Launchers of one input dtype (one translation unit each).  Every function
// returns the cudaError_t of the CUDA calls it made.
struct KernelTable {
  // Occupancy (CTAs per SM) and launch of the generic forward kernel (any
  // size and alignment, every layout; 256 threads per 32-row stripe).
  cudaError_t (*fwd_generic_occupancy)(int qm, int* blocks_per_sm);
  cudaError_t (*fwd_generic_launch)(int qm, const FwdParams& p, int grid, cudaStream_t stream);
  // Columnwise (and rowwise) forward over 32-row stripes split across a
  // thread-block cluster of g.cluster CTAs, `clusters` of them (persistent).
  cudaError_t (*stripe_max_clusters)(int qm, bool layernorm, const StripeGeom& g, int* clusters);
  cudaError_t (*stripe_launch)(int qm, bool layernorm, const StripeGeom& g, const FwdParams& p,
                               int clusters, cudaStream_t stream);
  // Columnwise FP8 output of rows too long for the stripe kernel, from x and
  // row statistics written by the long-row forward before it (mu: LayerNorm).
  cudaError_t (*colwise_occupancy)(int qm, bool layernorm, int* blocks_per_sm);
  cudaError_t (*colwise_launch)(int qm, bool layernorm, const FwdParams& p, const float* mu,
                                const float* rsigma, int grid, cudaStream_t stream);
  // Generic backward (any size and alignment, 256 threads).
  cudaError_t (*bwd_generic_occupancy)(int* blocks_per_sm);
  cudaError_t (*bwd_generic_launch)(const BwdParams& p, int grid, cudaStream_t stream);
  // Ring variants (rows streamed through shared memory by bulk copies);
  // `smem` = stages * stage bytes of dynamic shared memory.
  // kind = qm * 2 + (LayerNorm ? 1 : 0)
  cudaError_t (*fwd_ring_occupancy)(int kind, const RowGeom& g, int smem, int* blocks_per_sm);
  cudaError_t (*fwd_ring_launch)(int kind, const RowGeom& g, int stages, int smem,
                                 const FwdParams& p, int grid, cudaStream_t stream);
  cudaError_t (*bwd_ring_occupancy)(bool layernorm, bool add, const RowGeom& g, int smem,
                                    int* blocks_per_sm);
  cudaError_t (*bwd_ring_launch)(bool layernorm, bool add, const RowGeom& g, int stages, int smem,
                                 const BwdParams& p, int grid, cudaStream_t stream);
  // Long rows: forward with each row split over a cluster of `cluster` CTAs
  // of `threads` threads (4 vectors per thread), each owning hc columns.
  cudaError_t (*fwd_cluster_max_clusters)(int kind, int cluster, int threads, int smem,
                                          int* clusters);
  cudaError_t (*fwd_cluster_launch)(int kind, int cluster, int threads, int stages, int smem,
                                    int hc, const FwdParams& p, int clusters,
                                    cudaStream_t stream);
  // Long rows: backward with each row split over a cluster (2 vectors per
  // thread); partials go to workspace row `cluster id`.
  cudaError_t (*bwd_cluster_max_clusters)(bool layernorm, bool add, int cluster, int threads,
                                          int smem, int* clusters);
  cudaError_t (*bwd_cluster_launch)(bool layernorm, bool add, int cluster, int threads,
                                    int stages, int smem, int hc, const BwdParams& p,
                                    int clusters, cudaStream_t stream);
  // Self-test: a kernel whose wait for a copy that is never issued gives up
  // after limit_ns and sets this translation unit's device error flag.
  cudaError_t (*probe_copy_timeout)(unsigned long long limit_ns, cudaStream_t stream);
  // Sticky device-side error bits of this translation unit's kernels.
  cudaError_t (*read_device_error)(unsigned int* value, bool clear);
};

// Columnwise tile kernel: 256 threads of 2 columns, 32 rows per tile.
constexpr int kColTileThreads = 256;
constexpr int kColTileCols = 2 * kColTileThreads;

// Vectors per thread of the long-row (cluster) kernels.
constexpr int kClusterFwdNv = 4;
constexpr int kClusterBwdNv = 2;

const KernelTable& kernels_f32();
const KernelTable& kernels_bf16();
const KernelTable& kernels_f16();

// Finalize pass of the backward (sums the per-CTA partials).
cudaError_t launch_bwd_finalize(const FinalizeParams& p, cudaStream_t stream);

}  // namespace gbn
