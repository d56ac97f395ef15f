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
#include <map>
#include <mutex>
#include <tuple>

#include "gbn_internal.h"
#include "gbnorm.h"

namespace {

using namespace gbn;

constexpr int64_t kMaxHidden = int64_t(1) << 24;
constexpr int kMaxRingStagesHost = 8;  // matches the kernels' mbarrier array
constexpr int kMaxSmemPerCta = 220 * 1024;

bool io_dtype(gbn_dtype d) { return d == GBN_F32 || d == GBN_BF16 || d == GBN_F16; }
int esize(gbn_dtype d) { return d == GBN_F32 ? 4 : 2; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

const KernelTable& table(gbn_dtype in) {
  if (in == GBN_F32) return kernels_f32();
  if (in == GBN_BF16) return kernels_bf16();
  return kernels_f16();
}

// Vectors per thread (NV) and CTA size for a row of nvec 16-byte vectors:
// the first NV in {1, 2, 3, 4, 6, 8}, starting at `prefer_nv`, whose CTA
// (nvec / NV threads, rounded up to a warp) fits max_threads(NV), the
// largest CTA the kernel variant was compiled for; short rows take fewer
// vectors per thread so that a warp stays busy.  False if none fits.
bool row_geom(int64_t nvec, int vec, int prefer_nv, int (*max_threads)(int), RowGeom* g) {
  static const int kNv[] = {1, 2, 3, 4, 6, 8};
  for (int nv : kNv) {
    if (nv < prefer_nv && nvec > 32 * nv) continue;
    const int64_t t = ((nvec + nv - 1) / nv + 31) / 32 * 32;
    if (t > max_threads(nv)) continue;
    g->vec = vec;
    g->nv = nv;
    g->threads = static_cast<int>(t);
    return true;
  }
  return false;
}

RowGeom generic_geom() { return RowGeom{1, 1, 256}; }

int fwd_ring_cap(int nv) { return fwd_ring_max_threads(nv); }
int bwd_threads_cap(int nv) { return bwd_max_threads(nv); }

// Cluster split of a 32-row stripe for the columnwise layouts.  Candidates:
// C <= 16 CTAs per cluster (above 8 as a non-portable cluster size), each
// taking hc = hidden / C columns (a multiple of 8 and of the 16-byte vector;
// of 128 for MXFP8), at most 2048 two-byte or
// 1024 four-byte columns, with the slice (or two, when they fit) in shared
// memory.  Among them the one with the most co-resident CTAs (clusters x C;
// packing differs per C, and small slices fit several CTAs per SM), weighted
// by the share of threads that have work, wins; ties go to two stages, then to
// the smaller cluster.  Cached per (device, dtype, mode, hidden).
bool stripe_geom(const KernelTable& kt, int in, int qm, bool ln, int64_t hidden, int esize,
                 int sms, StripeGeom* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int64_t>, std::pair<bool, StripeGeom>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, in, qm, ln ? 1 : 0, hidden);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second.second;
      return it->second.first;
    }
  }
  const int vec = 16 / esize;
  const int64_t hc_max = esize == 2 ? 2048 : 1024;
  bool found = false;
  StripeGeom best{};
  int best_active = -1;
  for (int c = 1; c <= 16; ++c) {
    if (hidden % c) continue;
    const int64_t hc = hidden / c;
    // 16-byte vectors; MXFP8 in whole bands of 16 vectors (hc % 128 for 2- and 4-byte inputs).
    if (hc % vec || hc % 8 || (qm == Q_MXFP8 && hc % 128) || hc > hc_max) continue;
    for (int stages = 2; stages >= 1; --stages) {
      const int smem = stripe_smem_bytes(qm, ln, static_cast<int>(hc), esize, stages, c);
      if (smem > kMaxSmemPerCta) continue;
      StripeGeom g{c, static_cast<int>(hc), stages, smem, 0};
      int n = 0;
      if (kt.stripe_max_clusters(qm, ln, g, &n) != cudaSuccess || n < 1) continue;
      // co-resident CTAs, weighted by the share of each CTA's threads that
      // have work: delayed scaling gives a thread a 4-column item (hc/4 items
      // over kStripeThreads threads), MXFP8 a warp a band of 16 vectors.
      const int64_t workers = qm == Q_MXFP8 ? hc / vec / 16 : hc / 4;
      const int64_t slots = qm == Q_MXFP8 ? kStripeThreads / 32 : kStripeThreads;
      const int64_t waves = (workers + slots - 1) / slots;
      const int active = static_cast<int>(static_cast<int64_t>(n) * c * 1024 * workers /
                                          (waves * slots) / 1024);
      if (active > best_active) {  // strict: earlier (2 stages, smaller C) wins ties
        best_active = active;
        best = g;
        best.max_clusters = n;
        found = true;
      }
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = std::make_pair(found, best);
  *out = best;
  return found;
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

// ---- bulk-copy ring sizing


// Stage count (1..max_stages) for the ring kernels: CTAs per SM (occupancy
// with the ring's shared memory) times the stages being filled gives the
// bytes in flight per SM.  Occupancy answers are cached per (device, kernel
// choice).
struct RingChoice {
  int stages = 0;
  int occ = 0;
};

template <typename OccFn>
RingChoice choose_ring(int key_kind, int in, const RowGeom& g, int stage_bytes, int max_stages,
                       OccFn occ_fn) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, RingChoice> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, key_kind, in, g.nv, g.threads, stage_bytes);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  // Bytes in flight per SM up to kRingTarget count first, then resident
  // threads (latency hiding), then fewer stages.  Measured on the 16384 x
  // 4096 bf16 LayerNorm forward: 4 CTAs x 6 stages (160 KB in flight) 47.4
  // us, 3 x 8 (168 KB) 51.3 us, 3 x 3 to 3 x 6 about 49.2 us; more bytes in
  // flight than this only deepen the memory queue.
  constexpr int64_t kRingTarget = 160 * 1024;
  RingChoice best;
  int64_t best_inflight = -1;
  int best_occ = 0;
  for (int s = 1; s <= max_stages; ++s) {
    const int smem = s * stage_bytes;
    if (smem > kMaxSmemPerCta) break;
    int occ = 0;
    if (occ_fn(smem, &occ) != cudaSuccess || occ < 1) continue;
    int64_t inflight = static_cast<int64_t>(occ) * (s > 1 ? s - 1 : 1) * stage_bytes;
    if (inflight > kRingTarget) inflight = kRingTarget;
    if (inflight > best_inflight || (inflight == best_inflight && occ > best_occ)) {
      best_inflight = inflight;
      best_occ = occ;
      best.stages = s;
      best.occ = occ;
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = best;
  return best;
}

// Long rows: over the clusters C (2..8) whose per-CTA slice hc = H / C fits
// the cluster forward kernel (kClusterFwdNv vectors per thread, at most
// fwd_ring_max_threads(kClusterFwdNv) threads; MXFP8 slices whole
// 32-blocks) and their stage counts, the one that puts the most bytes in
// flight (up to the ring target per SM), ties to more resident CTAs.  A
// larger cluster of smaller CTAs can win: two CTAs on an SM hide each
// other's per-row statistics exchange (measured: 65536-wide bf16 LayerNorm
// 312 -> 287 us with C = 8 of 256 threads instead of C = 4 of 512).
// LayerNorm first considers only the clusters whose CTAs take the kernel's
// one-pass mean/M2 merge (whole vectors for every thread, a power-of-two
// warp count of at least 2; one block reduction per row instead of two):
// bf16 rows of 20480 123 us at C = 5 against 137 at C = 4, 28672 129 at
// C = 7 against 144 at C = 4.  Cached.
struct ClusterChoice {
  int cluster = 0, threads = 0, hc = 0, stages = 0, stage_bytes = 0, max_clusters = 0;
};

bool cluster_fwd_geom(const KernelTable& kt, int in, int kind, int qm, int64_t hidden, int vec,
                      int sms, ClusterChoice* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int64_t>, std::pair<bool, ClusterChoice>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, in, kind, hidden);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second.second;
      return it->second.first;
    }
  }
  constexpr int64_t kTarget = 224 * 1024;
  ClusterChoice best;
  bool found = false;
  int64_t best_inflight = -1;
  const bool ln = (kind & 1) != 0;
  for (int pass = ln ? 0 : 1; pass < 2 && !found; ++pass)
  for (int c = 2; c <= 8; ++c) {
    if (hidden % (static_cast<int64_t>(c) * vec)) continue;
    const int64_t hc = hidden / c;
    if (qm == Q_MXFP8 && hc % 32) continue;
    const int64_t nvc = hc / vec;
    const int64_t t = ((nvc + kClusterFwdNv - 1) / kClusterFwdNv + 31) / 32 * 32;
    if (t > fwd_ring_max_threads(kClusterFwdNv)) continue;
    const int64_t w = t / 32;
    if (pass == 0 && (nvc != kClusterFwdNv * t || w < 2 || (w & (w - 1)))) continue;
    const int stage_bytes = ring_slot_bytes(kClusterFwdNv, static_cast<int>(t));
    for (int st = 1; st <= kMaxRingStagesHost; ++st) {
      const int smem = st * stage_bytes;
      if (smem > kMaxSmemPerCta) break;
      int n = 0;
      if (kt.fwd_cluster_max_clusters(kind, c, static_cast<int>(t), smem, &n) != cudaSuccess ||
          n < 1)
        continue;
      int64_t inflight = static_cast<int64_t>(n) * c * (st > 1 ? st - 1 : 1) * stage_bytes / sms;
      if (inflight > kTarget) inflight = kTarget;
      if (inflight > best_inflight ||
          (inflight == best_inflight && n * c > best.max_clusters * best.cluster)) {
        best_inflight = inflight;
        best = ClusterChoice{c, static_cast<int>(t), static_cast<int>(hc), st, stage_bytes, n};
        found = true;
      }
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = std::make_pair(found, best);
  *out = best;
  return found;
}

// Long rows, backward: as cluster_fwd_geom, with kClusterBwdNv vectors per
// thread, at most bwd_max_threads(kClusterBwdNv) threads and at least 4
// stages of (dz, x[, dresidual]) slices.  LayerNorm: over every cluster size
// and stage count, the most bytes in flight per SM (up to the target), ties
// to more resident CTAs; RMSNorm: the smallest cluster that fits, with its
// stage count chosen the same way.  Measured on bf16 backward rows, smallest
// cluster against bytes in flight: LayerNorm 13088 x 10240 208 -> 164 us,
// 6528 x 20480 219 -> 170, 2720 x 49152 182 either way (C = 6: 512 threads on
// 150 SMs; C = 8 would be 384 threads on the 120 SMs that 8-CTA clusters
// reach, 225 us); RMSNorm with dresidual 7264 x 18432 211 -> 248 and 2720 x
// 49152 207 -> 240 us, against 230 -> 215 at 20480.  Cached.
bool cluster_bwd_geom(const KernelTable& kt, int in, bool ln, bool add, int64_t hidden, int vec,
                      int sms, ClusterChoice* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int64_t>, std::pair<bool, ClusterChoice>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, in, ln ? 1 : 0, add ? 1 : 0, hidden);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second.second;
      return it->second.first;
    }
  }
  constexpr int64_t kTarget = 224 * 1024;
  ClusterChoice best;
  bool found = false;
  int64_t best_inflight = -1;
  for (int c = 2; c <= 8 && (ln || !found); ++c) {
    if (hidden % (static_cast<int64_t>(c) * vec)) continue;
    const int64_t hc = hidden / c;
    const int64_t nvc = hc / vec;
    const int64_t t = ((nvc + kClusterBwdNv - 1) / kClusterBwdNv + 31) / 32 * 32;
    if (t > bwd_max_threads(kClusterBwdNv)) continue;
    const int stage_bytes = (add ? 3 : 2) * ring_slot_bytes(kClusterBwdNv, static_cast<int>(t));
    // at least four stages: the kernel holds the two rows of a pair while
    // the next pair's rows are in flight (measured on 4096 x 65536 bf16:
    // 405 us with four, 396 with up to six or eight)
    for (int st = 4; st <= kMaxRingStagesHost; ++st) {
      const int smem = st * stage_bytes;
      if (smem > kMaxSmemPerCta) break;
      int n = 0;
      if (kt.bwd_cluster_max_clusters(ln, add, c, static_cast<int>(t), smem, &n) != cudaSuccess ||
          n < 1)
        continue;
      int64_t inflight = static_cast<int64_t>(n) * c * (st - 1) * stage_bytes / sms;
      if (inflight > kTarget) inflight = kTarget;
      if (inflight > best_inflight ||
          (inflight == best_inflight && n * c > best.max_clusters * best.cluster)) {
        best_inflight = inflight;
        best = ClusterChoice{c, static_cast<int>(t), static_cast<int>(hc), st, stage_bytes, n};
        found = true;
      }
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = std::make_pair(found, best);
  *out = best;
  return found;
}

// The layout without the swizzled-scales flag.
gbn_quantize_layout base_layout(gbn_quantize_layout lay) {
  return static_cast<gbn_quantize_layout>(static_cast<int>(lay) & ~GBN_LAYOUT_SWIZZLED_SCALES);
}

gbn_status check_fwd_args(int64_t rows, int64_t hidden, gbn_dtype in, gbn_dtype w, gbn_dtype out,
                          gbn_norm_type norm, gbn_scaling_mode sc, gbn_quantize_layout layout) {
  if (norm != GBN_LAYERNORM && norm != GBN_RMSNORM) return GBN_ERR_ENUM;
  if (sc < GBN_SCALING_NONE || sc > GBN_SCALING_MXFP8_1D) return GBN_ERR_ENUM;
  const gbn_quantize_layout lay = base_layout(layout);
  if (lay < GBN_LAYOUT_ROWWISE || lay > GBN_LAYOUT_ROWWISE_COLWISE) return GBN_ERR_ENUM;
  if (lay != layout && sc != GBN_SCALING_MXFP8_1D) return GBN_ERR_ENUM;
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
  int parts;          // P: upper bound on the CTAs of the persistent grid
  size_t ws_bytes;    // P fp32 partial rows for dgamma (and dbeta)
};

// Ring choice of the backward row pass for geometry g (cached).
RingChoice bwd_ring_choice(const KernelTable& kt, gbn_dtype in, bool ln, bool add,
                           const RowGeom& g, int64_t hidden, int* stage_bytes) {
  *stage_bytes = (add ? 3 : 2) * static_cast<int>((hidden * esize(in) + 127) / 128 * 128);
  return choose_ring(20 + (ln ? 2 : 0) + (add ? 1 : 0), in, g, *stage_bytes, 4,
                     [&](int smem, int* o) { return kt.bwd_ring_occupancy(ln, add, g, smem, o); });
}

// P, the partial rows of the workspace: the persistent grid of the ring
// kernel (with or without the residual add, whichever is larger).  The
// generic kernel, used for misaligned pointers, runs at most P CTAs too.
gbn_status plan_bwd(int64_t rows, int64_t hidden, gbn_dtype in, gbn_norm_type norm,
                    int sm_margin, BwdPlan* plan) {
  int sms = 0;
  gbn_status st = device_sms(&sms);
  if (st != GBN_OK) return st;
  const int vec = 16 / esize(in);
  const bool ln = norm == GBN_LAYERNORM;
  RowGeom g = generic_geom();
  if (hidden % vec != 0 || !row_geom(hidden / vec, vec, 2, bwd_threads_cap, &g)) g = generic_geom();
  int occ = 0;
  const KernelTable& kt = table(in);
  // Rows that need 8 vectors per thread in the ring (its weights and
  // dgamma/dbeta partials then spill) run faster split over a cluster when
  // one fits (measured, bf16 LayerNorm 8192 x 16384: 270 vs 168 us; RMSNorm
  // with dresidual 8192 x 14000: 219 vs 172 us; fp32 8192 wide: even), and so
  // do LayerNorm rows at 3 vectors per thread, where the ring spills too
  // (bf16 13088 x 10240: 233 vs 162 us; 10912 x 12288: 201 vs 168 us, with
  // the cluster size chosen below; RMSNorm there is faster in the ring: 176
  // vs 193 us at 12288 with dresidual).
  if (g.vec != 1 && (g.nv == 8 || (ln && g.nv == 3))) {
    bool fits = true;
    for (int add = 0; add < 2; ++add) {
      ClusterChoice cc;
      if (!cluster_bwd_geom(kt, in, ln, add != 0, hidden, vec, sms, &cc)) fits = false;
    }
    if (fits) g = generic_geom();
  }
  if (g.vec != 1) {
    int sbytes = 0;
    for (int add = 0; add < 2; ++add) {
      const RingChoice rc = bwd_ring_choice(kt, in, ln, add != 0, g, hidden, &sbytes);
      if (rc.stages >= 1 && rc.occ > occ) occ = rc.occ;
    }
  }
  // Long rows: clusters (P = clusters; the generic fallback stays within P).
  int64_t cl_parts = 0;
  if (g.vec == 1 && hidden % vec == 0) {
    for (int add = 0; add < 2; ++add) {
      ClusterChoice cc;
      if (cluster_bwd_geom(kt, in, ln, add != 0, hidden, vec, sms, &cc)) {
        const int64_t n = static_cast<int64_t>(static_cast<double>(cc.max_clusters) *
                                               effective_sms(sms, sm_margin) / sms);
        if (n > cl_parts) cl_parts = n;
      }
    }
    if (cl_parts >= 1) occ = 1;
  }
  if (occ < 1) {
    if (kt.bwd_generic_occupancy(&occ) != cudaSuccess) return GBN_ERR_CUDA;
    if (occ < 1) occ = 1;
  }
  int64_t parts = cl_parts >= 1 ? cl_parts : static_cast<int64_t>(effective_sms(sms, sm_margin)) * occ;
  if (parts > rows) parts = rows;
  if (parts < 1) parts = 1;
  plan->geom = g;
  plan->parts = static_cast<int>(parts);
  plan->ws_bytes = static_cast<size_t>(parts) * static_cast<size_t>(hidden) * 4u * (ln ? 2u : 1u);
  return GBN_OK;
}

// Columnwise layouts of rows longer than one CTA's ring (the stripe kernel
// may still take them, up to 16 CTAs of 2048 two-byte columns): the shapes
// for which the forward may run the long-row kernel and then the columnwise
// tile kernel, which needs the row statistics in memory -- in mu / rsigma, or
// in the workspace when those are NULL.
bool long_colwise_shape(int64_t rows, int64_t hidden, int vec) {
  RowGeom g;
  return rows > 0 && rows % 32 == 0 && hidden % vec == 0 &&
         !row_geom(hidden / vec, vec, 4, fwd_ring_cap, &g);
}
// Workspace bytes for the row statistics: rsigma [rows] (and mu [rows]).
size_t stats_bytes(int64_t rows, bool ln) {
  return (static_cast<size_t>(rows) * 4u * (ln ? 2u : 1u) + 255u) / 256u * 256u;
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
  const gbn_quantize_layout lay = base_layout(quantize_layout);
  const bool colwise = scaling_mode != GBN_SCALING_NONE && lay != GBN_LAYOUT_ROWWISE;
  *bytes = colwise && long_colwise_shape(rows, hidden, 16 / esize(in_dtype))
               ? stats_bytes(rows, norm_type == GBN_LAYERNORM)
               : 0;
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
  const bool swizzle = base_layout(quantize_layout) != quantize_layout;
  quantize_layout = base_layout(quantize_layout);
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
  p.mx_swizzle = swizzle ? 1 : 0;

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
    const bool stripe_ok = vec_ok && rows % 32 == 0 && aligned(colwise_out, 32) &&
                           (qm != Q_MXFP8 || aligned(colwise_scale_inv, vec >= 8 ? 8 : 4)) &&
                           stripe_geom(kt, in_dtype, qm, ln, hidden, esize(in_dtype), sms, &sg);
    if (stripe_ok) {
      int64_t ncl = static_cast<int64_t>(static_cast<double>(sg.max_clusters) * esms / sms);
      if (ncl > rows / 32) ncl = rows / 32;
      if (ncl < 1) ncl = 1;
      const cudaError_t e = kt.stripe_launch(qm, ln, sg, p, static_cast<int>(ncl), stream);
      return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
    }
    // Rows too long for a stripe: the long-row kernel writes the row
    // statistics, any rowwise output and the amax, then the columnwise tile
    // kernel reads x again and writes the columnwise output from them.
    float* smu = ln ? mu : nullptr;
    float* srs = rsigma;
    if (((ln && !smu) || !srs) && workspace && aligned(workspace, 16) &&
        workspace_bytes >= stats_bytes(rows, ln)) {
      srs = static_cast<float*>(workspace);
      smu = ln ? srs + rows : nullptr;
    }
    ClusterChoice cc;
    const int kind = qm * 2 + (ln ? 1 : 0);
    if (vec_ok && long_colwise_shape(rows, hidden, vec) && srs && (!ln || smu) &&
        aligned(colwise_out, qm == Q_DELAYED ? 32 : 2) &&
        cluster_fwd_geom(kt, in_dtype, kind, qm, hidden, vec, sms, &cc)) {
      FwdParams pa = p;
      pa.mu = smu;
      pa.rsigma = srs;
      int64_t ncl = static_cast<int64_t>(static_cast<double>(cc.max_clusters) * esms / sms);
      if (ncl > rows) ncl = rows;
      if (ncl < 1) ncl = 1;
      cudaError_t e = kt.fwd_cluster_launch(kind, cc.cluster, cc.threads, cc.stages,
                                            cc.stages * cc.stage_bytes, cc.hc, pa,
                                            static_cast<int>(ncl), stream);
      if (e != cudaSuccess) return GBN_ERR_CUDA;
      int occ = 0;
      if (kt.colwise_occupancy(qm, ln, &occ) != cudaSuccess) return GBN_ERR_CUDA;
      const int64_t tiles = rows / 32 * ((hidden + kColTileCols - 1) / kColTileCols);
      int64_t grid = static_cast<int64_t>(esms) * (occ > 0 ? occ : 1);
      if (grid > tiles) grid = tiles;
      e = kt.colwise_launch(qm, ln, p, smu, srs, static_cast<int>(grid), stream);
      return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
    }
    vec_ok = false;  // generic kernel writes every layout
  }

  RowGeom gr;
  if (vec_ok && row_geom(hidden / vec, vec, 4, fwd_ring_cap, &gr)) {
    // Rows streamed through a shared-memory ring by bulk copies.
    const int stage_bytes = ring_slot_bytes(gr.nv, gr.threads);
    // LayerNorm rows that fill NV = 4 vectors of every thread of a CTA of 8 or
    // 16 warps take the one-pass mean/M2 variant (bf16 16384 x 16384: 94.1 ->
    // 88.0 us; at 2 and 4 warps, 2048 and 4096 wide, it measured 1-4 % slower
    // than the two-pass kernel, at 8 warps even).
    const int warps = gr.threads / 32;
    const bool one_pass = ln && gr.nv == 4 && hidden / vec == 4 * static_cast<int64_t>(gr.threads) &&
                          (warps == 8 || warps == 16);
    const int kind = qm * 2 + (ln ? 1 : 0) + (one_pass ? 6 : 0);
    const RingChoice rc = choose_ring(30 + kind, in_dtype, gr, stage_bytes, kMaxRingStagesHost,
                                      [&](int smem, int* o) {
                                        return kt.fwd_ring_occupancy(kind, gr, smem, o);
                                      });
    if (rc.stages >= 1) {
      int64_t grid = static_cast<int64_t>(esms) * rc.occ;
      if (grid > rows) grid = rows;
      if (grid < 1) grid = 1;
      const cudaError_t e = kt.fwd_ring_launch(kind, gr, rc.stages, rc.stages * stage_bytes, p,
                                               static_cast<int>(grid), stream);
      return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
    }
  }
  ClusterChoice cc;
  if (vec_ok && rows > 0 &&
      cluster_fwd_geom(kt, in_dtype, qm * 2 + (ln ? 1 : 0), qm, hidden, vec, sms, &cc)) {
    // Rows longer than one CTA's ring: each row split over a cluster.
    int64_t ncl = static_cast<int64_t>(static_cast<double>(cc.max_clusters) * esms / sms);
    if (ncl > rows) ncl = rows;
    if (ncl < 1) ncl = 1;
    const cudaError_t e = kt.fwd_cluster_launch(qm * 2 + (ln ? 1 : 0), cc.cluster, cc.threads,
                                                cc.stages, cc.stages * cc.stage_bytes, cc.hc, p,
                                                static_cast<int>(ncl), stream);
    return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
  }
  // Generic kernel: persistent over 32-row stripes.
  int occ = 0;
  if (kt.fwd_generic_occupancy(qm, &occ) != cudaSuccess) return GBN_ERR_CUDA;
  int64_t grid = static_cast<int64_t>(esms) * (occ > 0 ? occ : 1);
  if (grid > (rows + 31) / 32) grid = (rows + 31) / 32;
  if (grid < 1) grid = 1;
  const cudaError_t e = kt.fwd_generic_launch(qm, p, static_cast<int>(grid), stream);
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
  int sms = 0;
  st = device_sms(&sms);
  if (st != GBN_OK) return st;
  const int esms = effective_sms(sms, sm_margin);
  RingChoice rc;
  int stage_bytes = 0;
  if (g.vec != 1) rc = bwd_ring_choice(kt, in_dtype, ln, add, g, hidden, &stage_bytes);
  int occ = rc.occ;
  const bool ring = rc.stages >= 1;
  // Long rows: each row over a cluster, when the pointers allow vectors.
  ClusterChoice cc;
  const bool cluster = !ring && plan.geom.vec == 1 && hidden % vec == 0 && rows > 0 &&
                       aligned(dz, 16) && aligned(x, 16) && aligned(dx, 16) &&
                       (!dresidual || aligned(dresidual, 16)) && aligned(gamma, walign) &&
                       cluster_bwd_geom(kt, in_dtype, ln, add, hidden, vec, sms, &cc);
  if (!ring) {
    g = generic_geom();
    if (kt.bwd_generic_occupancy(&occ) != cudaSuccess) return GBN_ERR_CUDA;
  }
  int64_t grid = static_cast<int64_t>(esms) * (occ > 0 ? occ : 1);
  if (cluster) grid = static_cast<int64_t>(static_cast<double>(cc.max_clusters) * esms / sms);
  if (grid > plan.parts) grid = plan.parts;
  if (grid > rows && cluster) grid = rows;
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
  const cudaError_t le =
      ring      ? kt.bwd_ring_launch(ln, add, g, rc.stages, rc.stages * stage_bytes, p,
                                     static_cast<int>(grid), stream)
      : cluster ? kt.bwd_cluster_launch(ln, add, cc.cluster, cc.threads, cc.stages,
                                        cc.stages * cc.stage_bytes, cc.hc, p,
                                        static_cast<int>(grid), stream)
                : kt.bwd_generic_launch(p, static_cast<int>(grid), stream);
  if (le != cudaSuccess) return GBN_ERR_CUDA;

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

gbn_status gbn_selftest_copy_timeout(unsigned int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 2000000u) return GBN_ERR_SHAPE;
  const cudaError_t e =
      kernels_f32().probe_copy_timeout(static_cast<unsigned long long>(timeout_us) * 1000ull, stream);
  return e == cudaSuccess ? GBN_OK : GBN_ERR_CUDA;
}

gbn_status gbn_device_error(unsigned int* flags, int clear) {
  if (!flags) return GBN_ERR_NULL;
  unsigned int a = 0, b = 0, c = 0;
  if (kernels_f32().read_device_error(&a, clear != 0) != cudaSuccess ||
      kernels_bf16().read_device_error(&b, clear != 0) != cudaSuccess ||
      kernels_f16().read_device_error(&c, clear != 0) != cudaSuccess)
    return GBN_ERR_CUDA;
  *flags = a | b | c;
  return GBN_OK;
}

}  // extern "C"
