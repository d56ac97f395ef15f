// C-ABI layer of libgbnorm.so: argument validation, path and geometry
// selection, persistent-grid sizing with the SM margin, and the launches.
//
// Interface: "Implementation:NVIDIA TransformerEngine JAX XLA Normalization",
// Signature and I/O Contract (NormForwardFFI, NormBackwardFFI,
// GetNormForwardWorkspaceSizes, GetNormBackwardWorkspaceSizes; "SM margin is
// subtracted from the device's multiprocessor count"), and
// "Implementation:NVIDIA TransformerEngine Ops Fused Backward Add RMSNorm",
// I/O Contract (the residual gradient added to grad_input).
#include <cstdint>

#include "gbn_internal.h"
#include "gbnorm.h"

namespace {

using namespace gbn;

constexpr int64_t kMaxHidden = int64_t(1) << 24;

bool io_dtype(gbn_dtype d) { return d == GBN_F32 || d == GBN_BF16 || d == GBN_F16; }
int esize(gbn_dtype d) { return d == GBN_F32 ? 4 : 2; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

const KernelTable& table(gbn_dtype in) {
  if (in == GBN_F32) return kernels_f32();
  if (in == GBN_BF16) return kernels_bf16();
  return kernels_f16();
}

// Vectors per thread and CTA size for a row of nvec 16-byte vectors.  Short
// rows shrink the per-thread count so a warp stays busy; long rows grow it
// until the CTA fits 1024 threads.  Returns false if even 8 do not fit.
// `max_threads(nv)` is the largest CTA the kernel variant was compiled for.
bool row_geom(int64_t nvec, int vec, int prefer_nv, int (*max_threads)(int), RowGeom* g) {
  int nv = prefer_nv;
  while (nv > 1 && (nvec + nv - 1) / nv < 32) nv /= 2;
  int64_t t = ((nvec + nv - 1) / nv + 31) / 32 * 32;
  while (t > max_threads(nv) && nv < 8) {
    nv *= 2;
    t = ((nvec + nv - 1) / nv + 31) / 32 * 32;
  }
  if (t > max_threads(nv)) return false;
  g->vec = vec;
  g->nv = nv;
  g->threads = static_cast<int>(t);
  return true;
}

RowGeom generic_geom() { return RowGeom{1, 1, 256}; }

int fwd_max_threads(int) { return 1024; }
int bwd_threads_cap(int nv) { return bwd_max_threads(nv); }

// Cluster split of a 32-row stripe: the smallest cluster (<= 8 CTAs) whose
// column slice gives every lane the same number (<= 4) of 16-byte vectors per
// row; otherwise the smallest one with <= 4, then <= 8, per lane.
bool stripe_geom(int64_t hidden, int vec, bool mxfp8, StripeGeom* g) {
  for (int pass = 0; pass < 3; ++pass) {
    for (int c = 1; c <= 8; ++c) {
      if (hidden % c) continue;
      const int64_t hc = hidden / c;
      if (hc % vec) continue;
      if (mxfp8 && hc % 32) continue;
      if (hc % 8) continue;  // 4-column transpose groups and 8-byte code vectors
      const int64_t nv_row = hc / vec;
      const int64_t nvs = (nv_row + 31) / 32;
      const bool exact = (nv_row % 32) == 0;
      const int64_t cap = pass == 2 ? 8 : 4;
      if (nvs > cap || (pass == 0 && !exact)) continue;
      int t = 1;
      while (t < nvs) t *= 2;
      g->vec = vec;
      g->nvs = t;
      g->cluster = c;
      g->hc = static_cast<int>(hc);
      return true;
    }
  }
  return false;
}

gbn_status device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GBN_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GBN_ERR_CUDA;
  return GBN_OK;
}

int effective_sms(int sms, int sm_margin) {
  const int e = sms - (sm_margin > 0 ? sm_margin : 0);
  return e < 1 ? 1 : e;
}

gbn_status check_fwd_args(int64_t rows, int64_t hidden, gbn_dtype in, gbn_dtype w, gbn_dtype out,
                          gbn_norm_type norm, gbn_scaling_mode sc, gbn_quantize_layout lay) {
  if (norm != GBN_LAYERNORM && norm != GBN_RMSNORM) return GBN_ERR_ENUM;
  if (sc < GBN_SCALING_NONE || sc > GBN_SCALING_MXFP8_1D) return GBN_ERR_ENUM;
  if (lay < GBN_LAYOUT_ROWWISE || lay > GBN_LAYOUT_ROWWISE_COLWISE) return GBN_ERR_ENUM;
  if (!io_dtype(in) || !io_dtype(w)) return GBN_ERR_DTYPE;
  if (sc == GBN_SCALING_NONE ? out != in : out != GBN_E4M3) return GBN_ERR_DTYPE;
  if (rows < 0 || hidden < 1 || hidden > kMaxHidden) return GBN_ERR_SHAPE;
  if (sc == GBN_SCALING_MXFP8_1D) {
    if (hidden % 32) return GBN_ERR_SHAPE;
    if (lay != GBN_LAYOUT_ROWWISE && rows % 32) return GBN_ERR_SHAPE;
  }
  return GBN_OK;
}

struct BwdPlan {
  RowGeom geom;       // geometry of the vector path (or generic)
  int parts;          // P: CTAs of the persistent grid = partial rows in the workspace
  size_t ws_bytes;
};

gbn_status plan_bwd(int64_t rows, int64_t hidden, gbn_dtype in, gbn_norm_type norm,
                    int sm_margin, BwdPlan* plan) {
  int sms = 0;
  gbn_status st = device_sms(&sms);
  if (st != GBN_OK) return st;
  const int vec = 16 / esize(in);
  RowGeom g = generic_geom();
  if (hidden % vec != 0 || !row_geom(hidden / vec, vec, 2, bwd_threads_cap, &g)) g = generic_geom();
  const bool ln = norm == GBN_LAYERNORM;
  int occ_a = 0, occ_b = 0;
  const KernelTable& kt = table(in);
  if (kt.bwd_occupancy(ln, false, g, &occ_a) != cudaSuccess) return GBN_ERR_CUDA;
  if (kt.bwd_occupancy(ln, true, g, &occ_b) != cudaSuccess) return GBN_ERR_CUDA;
  const int occ = occ_a > occ_b ? occ_a : occ_b;
  int64_t parts = static_cast<int64_t>(effective_sms(sms, sm_margin)) * (occ > 0 ? occ : 1);
  if (parts > rows) parts = rows;
  if (parts < 1) parts = 1;
  plan->geom = g;
  plan->parts = static_cast<int>(parts);
  plan->ws_bytes = static_cast<size_t>(parts) * static_cast<size_t>(hidden) * 4u * (ln ? 2u : 1u);
  return GBN_OK;
}

}  // namespace

extern "C" {

const char* gbn_status_string(gbn_status s) {
  switch (s) {
    case GBN_OK: return "GBN_OK";
    case GBN_ERR_NULL: return "GBN_ERR_NULL: a required pointer is NULL";
    case GBN_ERR_DTYPE: return "GBN_ERR_DTYPE: unsupported dtype combination";
    case GBN_ERR_SHAPE: return "GBN_ERR_SHAPE: unsupported rows/hidden";
    case GBN_ERR_ALIGNMENT: return "GBN_ERR_ALIGNMENT: misaligned pointer";
    case GBN_ERR_WORKSPACE: return "GBN_ERR_WORKSPACE: workspace missing or too small";
    case GBN_ERR_ENUM: return "GBN_ERR_ENUM: enum value out of range";
    case GBN_ERR_CUDA: return "GBN_ERR_CUDA: CUDA runtime error";
  }
  return "GBN_ERR_UNKNOWN";
}

gbn_status gbn_norm_fwd_workspace_size(int64_t rows, int64_t hidden, gbn_dtype in_dtype,
                                       gbn_dtype w_dtype, gbn_dtype out_dtype,
                                       gbn_norm_type norm_type, gbn_scaling_mode scaling_mode,
                                       gbn_quantize_layout quantize_layout,
                                       int zero_centered_gamma, int sm_margin, int is_training,
                                       size_t* bytes) {
  (void)zero_centered_gamma;
  (void)sm_margin;
  (void)is_training;
  if (!bytes) return GBN_ERR_NULL;
  const gbn_status st = check_fwd_args(rows, hidden, in_dtype, w_dtype, out_dtype, norm_type,
                                       scaling_mode, quantize_layout);
  if (st != GBN_OK) return st;
  *bytes = 0;
  return GBN_OK;
}

gbn_status gbn_norm_fwd(const void* x, const void* gamma, const void* beta, const float* scale,
                        const float* amax, void* out, void* colwise_out, float* mu,
                        float* rsigma, void* scale_inv, void* colwise_scale_inv,
                        float* updated_amax, void* workspace, size_t workspace_bytes,
                        int64_t rows, int64_t hidden, gbn_dtype in_dtype, gbn_dtype w_dtype,
                        gbn_dtype out_dtype, gbn_norm_type norm_type,
                        gbn_scaling_mode scaling_mode, gbn_quantize_layout quantize_layout,
                        int zero_centered_gamma, float eps, int sm_margin, cudaStream_t stream) {
  (void)amax;
  (void)workspace;
  (void)workspace_bytes;
  gbn_status st = check_fwd_args(rows, hidden, in_dtype, w_dtype, out_dtype, norm_type,
                                 scaling_mode, quantize_layout);
  if (st != GBN_OK) return st;
  const bool ln = norm_type == GBN_LAYERNORM;
  const int qm = scaling_mode == GBN_SCALING_NONE ? Q_NONE
                 : scaling_mode == GBN_SCALING_DELAYED_TENSOR ? Q_DELAYED : Q_MXFP8;
  const bool rowwise = qm == Q_NONE || quantize_layout != GBN_LAYOUT_COLWISE;
  const bool colwise = qm != Q_NONE && quantize_layout != GBN_LAYOUT_ROWWISE;
  // Row-sized buffers may be NULL only when there are no rows.
  const bool any = rows > 0;
  if (!gamma || (ln && !beta)) return GBN_ERR_NULL;
  if (any && (!x || (rowwise && !out) || (colwise && !colwise_out))) return GBN_ERR_NULL;
  if (qm == Q_DELAYED && (!scale || !updated_amax)) return GBN_ERR_NULL;
  if (any && qm == Q_MXFP8 && ((rowwise && !scale_inv) || (colwise && !colwise_scale_inv)))
    return GBN_ERR_NULL;

  int sms = 0;
  st = device_sms(&sms);
  if (st != GBN_OK) return st;
  const int esms = effective_sms(sms, sm_margin);

  FwdParams p = {};
  p.x = x;
  p.gamma = gamma;
  p.beta = ln ? beta : nullptr;
  p.scale = scale;
  p.out = rowwise ? out : nullptr;
  p.colwise_out = colwise ? static_cast<uint8_t*>(colwise_out) : nullptr;
  p.mu = ln ? mu : nullptr;
  p.rsigma = rsigma;
  if (qm == Q_DELAYED) {
    p.scale_inv = rowwise ? static_cast<float*>(scale_inv) : nullptr;
    p.colwise_scale_inv = colwise ? static_cast<float*>(colwise_scale_inv) : nullptr;
    p.amax = updated_amax;
  } else if (qm == Q_MXFP8) {
    p.mx_scale = rowwise ? static_cast<uint8_t*>(scale_inv) : nullptr;
    p.mx_colwise_scale = colwise ? static_cast<uint8_t*>(colwise_scale_inv) : nullptr;
  }
  p.rows = rows;
  p.hidden = static_cast<int>(hidden);
  p.eps = eps;
  p.norm = ln ? 0 : 1;
  p.zcg = zero_centered_gamma ? 1 : 0;
  p.w_dt = w_dtype == GBN_F32 ? DT_F32 : (w_dtype == GBN_BF16 ? DT_BF16 : DT_F16);
  p.write_rowwise = rowwise ? 1 : 0;
  p.write_colwise = colwise ? 1 : 0;

  const int vec = 16 / esize(in_dtype);
  const uintptr_t walign = static_cast<uintptr_t>(vec * esize(w_dtype) < 16 ? vec * esize(w_dtype) : 16);
  const uintptr_t oalign = qm == Q_NONE ? 16u : static_cast<uintptr_t>(vec);
  bool vec_ok = hidden % vec == 0 && aligned(x, 16) && aligned(gamma, walign) &&
                (!ln || aligned(beta, walign)) && (!rowwise || aligned(out, oalign));

  const KernelTable& kt = table(in_dtype);
  if (qm == Q_DELAYED && cudaMemsetAsync(updated_amax, 0, sizeof(float), stream) != cudaSuccess)
    return GBN_ERR_CUDA;

  if (colwise) {
    StripeGeom sg;
    const bool stripe_ok = vec_ok && rows % 32 == 0 && aligned(colwise_out, 16) &&
                           stripe_geom(hidden, vec, qm == Q_MXFP8, &sg);
    if (stripe_ok) {
      const cudaError_t e = kt.stripe_launch(qm, sg, p, static_cast<double>(esms) / sms, stream);
      return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
    }
    vec_ok = false;  // generic kernel writes every layout
  }

  RowGeom g = generic_geom();
  if (vec_ok && !row_geom(hidden / vec, vec, 4, fwd_max_threads, &g)) g = generic_geom();
  int occ = 0;
  if (kt.fwd_occupancy(qm, g, &occ) != cudaSuccess) return GBN_ERR_CUDA;
  const int64_t units = g.vec == 1 ? (rows + 31) / 32 : rows;  // generic: 32-row stripes
  int64_t grid = static_cast<int64_t>(esms) * (occ > 0 ? occ : 1);
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  const cudaError_t e = kt.fwd_launch(qm, g, p, static_cast<int>(grid), stream);
  return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
}

gbn_status gbn_norm_bwd_workspace_size(int64_t rows, int64_t hidden, gbn_dtype in_dtype,
                                       gbn_dtype w_dtype, gbn_norm_type norm_type,
                                       int zero_centered_gamma, int sm_margin, size_t* bytes) {
  (void)zero_centered_gamma;
  if (!bytes) return GBN_ERR_NULL;
  if (norm_type != GBN_LAYERNORM && norm_type != GBN_RMSNORM) return GBN_ERR_ENUM;
  if (!io_dtype(in_dtype) || !io_dtype(w_dtype)) return GBN_ERR_DTYPE;
  if (rows < 0 || hidden < 1 || hidden > kMaxHidden) return GBN_ERR_SHAPE;
  BwdPlan plan;
  const gbn_status st = plan_bwd(rows, hidden, in_dtype, norm_type, sm_margin, &plan);
  if (st != GBN_OK) return st;
  *bytes = plan.ws_bytes;
  return GBN_OK;
}

gbn_status gbn_norm_bwd(const void* dz, const void* x, const float* mu, const float* rsigma,
                        const void* gamma, const void* dresidual, void* dx, void* dgamma,
                        void* dbeta, void* workspace, size_t workspace_bytes, int64_t rows,
                        int64_t hidden, gbn_dtype in_dtype, gbn_dtype w_dtype,
                        gbn_norm_type norm_type, int zero_centered_gamma, int sm_margin,
                        cudaStream_t stream) {
  if (norm_type != GBN_LAYERNORM && norm_type != GBN_RMSNORM) return GBN_ERR_ENUM;
  if (!io_dtype(in_dtype) || !io_dtype(w_dtype)) return GBN_ERR_DTYPE;
  if (rows < 0 || hidden < 1 || hidden > kMaxHidden) return GBN_ERR_SHAPE;
  const bool ln = norm_type == GBN_LAYERNORM;
  // Row-sized buffers may be NULL only when there are no rows.
  if (!gamma || !dgamma || (ln && !dbeta)) return GBN_ERR_NULL;
  if (rows > 0 && (!dz || !x || !rsigma || !dx || (ln && !mu))) return GBN_ERR_NULL;
  if (!workspace || !aligned(workspace, 16)) return GBN_ERR_WORKSPACE;

  BwdPlan plan;
  gbn_status st = plan_bwd(rows, hidden, in_dtype, norm_type, sm_margin, &plan);
  if (st != GBN_OK) return st;
  if (workspace_bytes < plan.ws_bytes) return GBN_ERR_WORKSPACE;

  const int vec = 16 / esize(in_dtype);
  const uintptr_t walign = static_cast<uintptr_t>(vec * esize(w_dtype) < 16 ? vec * esize(w_dtype) : 16);
  RowGeom g = plan.geom;
  const bool vec_ok = g.vec != 1 && aligned(dz, 16) && aligned(x, 16) && aligned(dx, 16) &&
                      (!dresidual || aligned(dresidual, 16)) && aligned(gamma, walign);
  if (!vec_ok) g = generic_geom();
  const bool add = dresidual != nullptr;
  const KernelTable& kt = table(in_dtype);
  int occ = 0;
  if (kt.bwd_occupancy(ln, add, g, &occ) != cudaSuccess) return GBN_ERR_CUDA;
  int sms = 0;
  st = device_sms(&sms);
  if (st != GBN_OK) return st;
  int64_t grid = static_cast<int64_t>(effective_sms(sms, sm_margin)) * (occ > 0 ? occ : 1);
  if (grid > plan.parts) grid = plan.parts;
  if (grid < 1) grid = 1;

  float* ws = static_cast<float*>(workspace);
  BwdParams p = {};
  p.dz = dz;
  p.x = x;
  p.mu = ln ? mu : nullptr;
  p.rsigma = rsigma;
  p.gamma = gamma;
  p.dres = dresidual;
  p.dx = dx;
  p.part_dgamma = ws;
  p.part_dbeta = ln ? ws + grid * hidden : nullptr;
  p.rows = rows;
  p.hidden = static_cast<int>(hidden);
  p.norm = ln ? 0 : 1;
  p.zcg = zero_centered_gamma ? 1 : 0;
  p.w_dt = w_dtype == GBN_F32 ? DT_F32 : (w_dtype == GBN_BF16 ? DT_BF16 : DT_F16);
  if (kt.bwd_launch(ln, add, g, p, static_cast<int>(grid), stream) != cudaSuccess)
    return GBN_ERR_CUDA;

  FinalizeParams f = {};
  f.part_dgamma = p.part_dgamma;
  f.part_dbeta = p.part_dbeta;
  f.dgamma = dgamma;
  f.dbeta = ln ? dbeta : nullptr;
  f.parts = static_cast<int>(grid);
  f.hidden = static_cast<int>(hidden);
  f.w_dt = p.w_dt;
  return launch_bwd_finalize(f, stream) == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
}

}  // extern "C"
