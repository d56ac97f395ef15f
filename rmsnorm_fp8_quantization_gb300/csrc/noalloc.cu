// Backward entry point for callers that cannot allocate device memory.
//
// gbn_norm_bwd needs a caller-provided workspace for its per-CTA dgamma /
// dbeta partials.  Some callers cannot provide one: code running where a
// cudaMalloc is not allowed or not wanted (inside a region being captured
// into a CUDA graph whose memory plan is fixed, a custom allocator that
// cannot be re-entered from this call site, or plugin hosts that forbid
// device allocation).  gbn_norm_bwd_noalloc serves them from a fixed
// scratch array that lives in this library's device image.
#include <mutex>

#include "gbn_internal.h"
#include "gbnorm.h"

namespace {

// Maximum scratch: the backward's partial rows must fit in it.  Every GPU on
// which the library's module is loaded holds this array until the process
// exits.
constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side handle, so the address is looked up
// once per device (this first call must not happen during stream capture).
gbn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
      return GBN_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return GBN_OK;
}

}  // namespace

extern "C" gbn_status gbn_norm_bwd_noalloc(const void* dz, const void* x, const float* mu,
                                           const float* rsigma, const void* gamma,
                                           const void* dresidual, void* dx, void* dgamma,
                                           void* dbeta, int64_t rows, int64_t hidden,
                                           gbn_dtype in_dtype, gbn_dtype w_dtype,
                                           gbn_norm_type norm_type, int zero_centered_gamma,
                                           int sm_margin, cudaStream_t stream) {
  size_t need = 0;
  gbn_status st = gbn_norm_bwd_workspace_size(rows, hidden, in_dtype, w_dtype, norm_type,
                                              zero_centered_gamma, sm_margin, &need);
  if (st != GBN_OK) return st;
  if (need > kScratchBytes) return GBN_ERR_WORKSPACE;
  void* ws = nullptr;
  st = scratch_address(&ws);
  if (st != GBN_OK) return st;
  return gbn_norm_bwd(dz, x, mu, rsigma, gamma, dresidual, dx, dgamma, dbeta, ws, kScratchBytes,
                      rows, hidden, in_dtype, w_dtype, norm_type, zero_centered_gamma, sm_margin,
                      stream);
}
