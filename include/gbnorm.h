/*
 * gbnorm — fused LayerNorm / RMSNorm forward and backward (and the scaled
 * masked softmax) for GB300 (sm_103a).
 *
 * C ABI of libgbnorm.so.  The norm operations follow two pages:
 *   "Implementation:NVIDIA TransformerEngine JAX XLA Normalization"
 *     (sections Description, Signature, I/O Contract): the forward handler's
 *     buffers (input, gamma, beta, scale, amax; output, colwise output, mu,
 *     rsigma, scale_inv, colwise scale_inv, updated amax, workspace), its
 *     attributes (norm type, scaling mode, quantize layout, zero-centered
 *     gamma, epsilon, SM margin), the workspace-size queries and the backward
 *     handler.
 *   "Implementation:NVIDIA TransformerEngine Ops Fused Backward Add RMSNorm"
 *     (sections Description, I/O Contract): the backward with the residual
 *     gradient added to the input gradient in the same kernel.
 * The softmax entry points (end of this file) follow "Migrate norms and
 * softmax kernels to NVRTC" (Description, JIT cost table), which names them.
 *
 * Arithmetic (x is one row of `hidden` elements; all device math in fp32):
 *   LayerNorm: mu = mean(x); var = mean((x - mu)^2); rsigma = 1/sqrt(var + eps)
 *              z = (x - mu) * rsigma * g' + beta
 *   RMSNorm:   rsigma = 1/sqrt(mean(x^2) + eps);  z = x * rsigma * g'
 *   g' = gamma, or 1 + gamma when zero_centered_gamma != 0.
 *   Backward:  xhat = (x - mu) * rsigma (LayerNorm) or x * rsigma (RMSNorm),
 *              dy = dz * g',
 *              LayerNorm dx = rsigma * (dy - mean(dy) - xhat * mean(dy * xhat))
 *              RMSNorm   dx = rsigma * (dy - xhat * mean(dy * xhat))
 *              dx += dresidual when dresidual != NULL,
 *              dgamma = sum over rows of dz * xhat, dbeta = sum over rows of dz.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major data
 *     owned by the caller.  The library allocates nothing, keeps no state
 *     between calls and never synchronizes: every operation (including the
 *     cudaMemsetAsync of updated_amax) is enqueued on `stream`, so the calls
 *     can be captured into a CUDA graph.
 *   - A status is returned; nothing is thrown and nothing aborts.  Arguments
 *     are validated before any work is enqueued; on an error nothing is
 *     enqueued.  A launch failure is reported as GBN_ERR_CUDA.
 *   - Buffers with a `rows` dimension may be NULL when rows == 0.
 *   - Pointers that are not 16-byte aligned (or a hidden size that is not a
 *     multiple of the 16-byte vector) are accepted and take a scalar path.
 *   - SM margin: the persistent grids use (SM count - sm_margin) SMs, at
 *     least one, times the kernel's occupancy.
 *   - 1 <= hidden <= 2^24 and rows >= 0 (else GBN_ERR_SHAPE).  Rows of up to
 *     18432 two-byte (9216 four-byte) elements run on one CTA each (the
 *     backward: up to 12288 / 6144, LayerNorm up to 8192 / 4096, and up to
 *     16384 / 8192 where no cluster split fits); longer rows are split over a
 *     thread-block cluster of up to 8 CTAs (forward up to 131072 / 65536
 *     elements, backward up to 65536 / 32768); longer still, or misaligned,
 *     they run on a slower generic kernel.
 *   - Norm outputs must not alias inputs.
 */
#ifndef GBNORM_H_
#define GBNORM_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Norm type: the page's NVTE_Norm_Type (LayerNorm or RMSNorm). */
typedef enum { GBN_LAYERNORM = 0, GBN_RMSNORM = 1 } gbn_norm_type;

/* Scaling mode of the output (the page's JAXX_Scaling_Mode: no scaling,
 * delayed per-tensor scaling, MXFP8 1D block scaling with 32 elements per
 * E8M0 scale). */
typedef enum {
  GBN_SCALING_NONE = 0,
  GBN_SCALING_DELAYED_TENSOR = 1,
  GBN_SCALING_MXFP8_1D = 2
} gbn_scaling_mode;

/* Which quantized outputs are written (the page's JAXX_Quantize_Layout:
 * rowwise, columnwise, or both).  Ignored when the scaling mode is NONE.
 *
 * GBN_LAYOUT_SWIZZLED_SCALES may be OR-ed into the layout with MXFP8 (no
 * counterpart on the pages; else GBN_ERR_ENUM).  The E8M0 scales then go to
 * padded buffers in the tiled order that block-scaled GEMMs read: a scale
 * matrix of R outer rows and B scales per row is padded to
 * R' = roundup(R, 128) x B' = roundup(B, 4) and stored as 512-byte tiles of
 * 128 x 4 scales, (R'/128) x (B'/4) tiles in row-major order; inside a tile,
 * scale (r, c) is byte 16 * (r % 32) + 4 * (r / 32) + c.  Rowwise scales:
 * R = rows, B = hidden/32 (row r, block b).  Columnwise scales: the operand
 * is used transposed, R = hidden, B = rows/32 (column h, rows 32s..32s+31 is
 * entry (h, s)).  Buffer sizes: R' * B' bytes.  Padding bytes are not
 * written. */
typedef enum {
  GBN_LAYOUT_ROWWISE = 0,
  GBN_LAYOUT_COLWISE = 1,
  GBN_LAYOUT_ROWWISE_COLWISE = 2,
  GBN_LAYOUT_SWIZZLED_SCALES = 0x100
} gbn_quantize_layout;

/* Element types.  Inputs and weights: F32, BF16, F16.  Unquantized output:
 * the input type.  Quantized output: E4M3 (OCP FP8, 1 byte); MXFP8 scales:
 * E8M0 (1 byte, bias 127). */
typedef enum { GBN_F32 = 0, GBN_BF16 = 1, GBN_F16 = 2, GBN_E4M3 = 3, GBN_E8M0 = 4 } gbn_dtype;

typedef enum {
  GBN_OK = 0,
  GBN_ERR_NULL = 1,      /* a pointer the chosen mode needs is NULL */
  GBN_ERR_DTYPE = 2,     /* unsupported dtype or dtype combination */
  GBN_ERR_SHAPE = 3,     /* rows/hidden out of range, or MXFP8 blocks do not tile */
  GBN_ERR_ALIGNMENT = 4, /* reserved: misaligned pointers take the scalar path */
  GBN_ERR_WORKSPACE = 5, /* workspace NULL or smaller than the queried size */
  GBN_ERR_ENUM = 6,      /* norm type, scaling mode or layout out of range */
  GBN_ERR_CUDA = 7       /* a CUDA runtime call or a launch failed */
} gbn_status;

/* Forward workspace size in bytes ("GetNormForwardWorkspaceSizes" on the
 * first page): room for the row statistics (rsigma, and mu for LayerNorm,
 * rounded up to 256 bytes) for columnwise FP8 layouts of rows % 32 == 0 rows
 * longer than one CTA's ring (over 18432 two-byte / 9216 four-byte
 * elements), 0 otherwise.  Host-only: no device is queried.  The call
 * validates its arguments; GBN_ERR_NULL if bytes is NULL. */
gbn_status gbn_norm_fwd_workspace_size(int64_t rows, int64_t hidden, gbn_dtype in_dtype,
                                       gbn_dtype w_dtype, gbn_dtype out_dtype,
                                       gbn_norm_type norm_type, gbn_scaling_mode scaling_mode,
                                       gbn_quantize_layout quantize_layout,
                                       int zero_centered_gamma, int sm_margin, int is_training,
                                       size_t* bytes);

/* Forward ("NormForwardFFI" on the first page).
 *
 *   x        [rows, hidden] in_dtype
 *   gamma    [hidden] w_dtype
 *   beta     [hidden] w_dtype, LayerNorm only (NULL for RMSNorm)
 *   scale    fp32 [1], delayed scaling only: the multiplier applied before the
 *            E4M3 cast (NULL otherwise)
 *   amax     fp32 [1], delayed scaling: the previous amax.  Accepted for
 *            interface parity and not read; updated_amax receives the fresh
 *            amax of this call.  May be NULL.
 *   out      rowwise output [rows, hidden]: in_dtype when the scaling mode is
 *            NONE, else E4M3 codes.  Required unless the layout is COLWISE.
 *   colwise_out  columnwise E4M3 output, required for COLWISE layouts:
 *            delayed scaling: the transpose, [hidden, rows];
 *            MXFP8: [rows, hidden] (not transposed), scaled per 32x1 block.
 *   mu       fp32 [rows], LayerNorm only; may be NULL (not written)
 *   rsigma   fp32 [rows]; may be NULL (not written)
 *   scale_inv        delayed: fp32 [1] = 1/scale (rowwise layouts);
 *                    MXFP8: E8M0 [rows, hidden/32] rowwise block scales
 *                    (tiled and padded with GBN_LAYOUT_SWIZZLED_SCALES)
 *   colwise_scale_inv  delayed: fp32 [1] = 1/scale (colwise layouts);
 *                    MXFP8: E8M0 [rows/32, hidden] columnwise block scales
 *                    (tiled and padded with GBN_LAYOUT_SWIZZLED_SCALES)
 *   updated_amax     fp32 [1], delayed scaling: max |z| over the whole output
 *                    (before scaling; NaN propagates).  Zeroed on `stream` by
 *                    this call, then reduced into.
 *   workspace        gbn_norm_fwd_workspace_size() bytes, 16-byte aligned, or
 *                    NULL.  Only columnwise FP8 layouts of rows longer than
 *                    one CTA's ring may use it: rows too long for the stripe
 *                    kernel run the long-row kernel and then a columnwise
 *                    tile kernel, which reads the row statistics from mu /
 *                    rsigma or, where those are NULL, from the workspace
 *                    (4 or, for LayerNorm, 8 bytes per row).  Without either
 *                    such a call takes the slower generic kernel; nothing
 *                    else reads the workspace.
 *   eps      added to the variance inside the square root.
 *
 * MXFP8 needs hidden % 32 == 0, and rows % 32 == 0 for columnwise layouts
 * (else GBN_ERR_SHAPE).  out_dtype must be in_dtype for NONE and GBN_E4M3
 * otherwise (else GBN_ERR_DTYPE). */
gbn_status gbn_norm_fwd(const void* x, const void* gamma, const void* beta, const float* scale,
                        const float* amax, void* out, void* colwise_out, float* mu,
                        float* rsigma, void* scale_inv, void* colwise_scale_inv,
                        float* updated_amax, void* workspace, size_t workspace_bytes,
                        int64_t rows, int64_t hidden, gbn_dtype in_dtype, gbn_dtype w_dtype,
                        gbn_dtype out_dtype, gbn_norm_type norm_type,
                        gbn_scaling_mode scaling_mode, gbn_quantize_layout quantize_layout,
                        int zero_centered_gamma, float eps, int sm_margin, cudaStream_t stream);

/* Backward workspace size in bytes ("GetNormBackwardWorkspaceSizes" on the
 * first page): fp32 partial dgamma (and dbeta for LayerNorm) rows, one per
 * CTA of the persistent grid.  Depends on the current device's SM count and
 * occupancy, so query it on the device that will run the call.
 * Returns GBN_ERR_CUDA if no device can be queried. */
gbn_status gbn_norm_bwd_workspace_size(int64_t rows, int64_t hidden, gbn_dtype in_dtype,
                                       gbn_dtype w_dtype, gbn_norm_type norm_type,
                                       int zero_centered_gamma, int sm_margin, size_t* bytes);

/* Backward (the first page's backward handler; with dresidual, the second
 * page's fused backward-add).
 *
 *   dz, x      [rows, hidden] in_dtype
 *   mu         fp32 [rows], LayerNorm only (NULL for RMSNorm)
 *   rsigma     fp32 [rows]
 *   gamma      [hidden] w_dtype
 *   dresidual  [rows, hidden] in_dtype, or NULL for no add
 *   dx         [rows, hidden] in_dtype
 *   dgamma     [hidden] w_dtype
 *   dbeta      [hidden] w_dtype, LayerNorm only (NULL for RMSNorm)
 *   workspace  at least gbn_norm_bwd_workspace_size() bytes, 16-byte aligned
 *              (GBN_ERR_WORKSPACE otherwise); its contents need no
 *              initialization and are overwritten.
 * Two kernels are enqueued: the row pass (dx and per-CTA partials) and a
 * finalize pass that sums the partials in a fixed order (deterministic for a
 * fixed device and sm_margin). */
gbn_status gbn_norm_bwd(const void* dz, const void* x, const float* mu, const float* rsigma,
                        const void* gamma, const void* dresidual, void* dx, void* dgamma,
                        void* dbeta, void* workspace, size_t workspace_bytes, int64_t rows,
                        int64_t hidden, gbn_dtype in_dtype, gbn_dtype w_dtype,
                        gbn_norm_type norm_type, int zero_centered_gamma, int sm_margin,
                        cudaStream_t stream);

/* Backward without a caller-provided workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory at the call site -- code running inside a region whose
 * device-memory plan is fixed (for example while a framework records a
 * replayable graph of its launches), behind a custom allocator that must not
 * be re-entered from here, or in plugin hosts that forbid device allocation.
 * gbn_norm_bwd needs a workspace for its per-CTA partials; this variant uses
 * a fixed 32 MiB scratch array that lives in the library's device image
 * (every GPU that loads the library holds it until the process exits) and
 * otherwise behaves exactly like gbn_norm_bwd (same arguments, minus the
 * workspace).
 *   - It allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - All calls share the one scratch array (it keeps the last call's
 *     contents; the backward overwrites every partial it reads), so calls
 *     that overlap on the GPU -- on different streams, or from several host
 *     threads -- race.  Serialize them.
 *   - Returns GBN_ERR_WORKSPACE when the problem's partials
 *     (gbn_norm_bwd_workspace_size) exceed 32 MiB. */
gbn_status gbn_norm_bwd_noalloc(const void* dz, const void* x, const float* mu,
                                const float* rsigma, const void* gamma, const void* dresidual,
                                void* dx, void* dgamma, void* dbeta, int64_t rows,
                                int64_t hidden, gbn_dtype in_dtype, gbn_dtype w_dtype,
                                gbn_norm_type norm_type, int zero_centered_gamma, int sm_margin,
                                cudaStream_t stream);

/* Device-side error bits, sticky across calls on the current device:
 *   bit 0 (GBN_DEVICE_ERR_COPY_TIMEOUT): a kernel waited longer than 2 s for
 *   one of its own bulk copies into shared memory, stopped early and left
 *   that call's outputs incomplete.
 * Kernels never trap or spin without bound; this flag is how such a failure
 * reaches the host.  The query synchronizes with the device.  With clear != 0
 * the bits are reset after reading. */
#define GBN_DEVICE_ERR_COPY_TIMEOUT 1u
gbn_status gbn_device_error(unsigned int* flags, int clear);

/* Self-test of that failure path (no counterpart on the pages): enqueues on
 * `stream` a one-thread kernel that waits for 16 bytes on an mbarrier that no
 * copy will ever fill, gives up after timeout_us microseconds (1 .. 2e6, else
 * GBN_ERR_SHAPE) and sets GBN_DEVICE_ERR_COPY_TIMEOUT, exactly as a kernel
 * whose bulk copy never landed would.  Nothing faults or traps; the context
 * stays usable. */
gbn_status gbn_selftest_copy_timeout(unsigned int timeout_us, cudaStream_t stream);

/* ---- Scaled (masked) softmax ("Migrate norms and softmax kernels to NVRTC",
 * Description and JIT cost table: scaled_masked_softmax,
 * scaled_upper_triang_masked_softmax, scaled_aligned_causal_masked_softmax,
 * forward and backward).  The page gives no formulas; the plain definitions
 * are used:
 *   y  = softmax over the last axis of scale * x, over the kept positions;
 *        masked positions get 0, and a row with no kept position is all 0;
 *   dx = scale * y * (dy - sum_j dy * y)   (y: the forward's output). */
typedef enum {
  GBN_SOFTMAX_NO_MASK = 0,
  GBN_SOFTMAX_PADDING = 1,        /* mask [mask_batches, 1, sq, sk] u8, nonzero = masked;
                                     batch b uses mask batch b % mask_batches */
  GBN_SOFTMAX_CAUSAL_UPPER = 2,   /* sq == sk; (i, j) kept iff j <= i */
  GBN_SOFTMAX_CAUSAL_ALIGNED = 3  /* bottom-right aligned; kept iff j <= i + (sk - sq) */
} gbn_softmax_mask;

/* Longest row (keys) of the softmax.  Rows whose byte length is not a
 * multiple of 16, or whose pointers are not 16-byte aligned, take a scalar
 * path limited to 2048 keys (longer: GBN_ERR_SHAPE). */
#define GBN_SOFTMAX_MAX_KEYS 16384

/* Forward.  x, y: [batches, heads, sq, sk] row-major in dtype (F32, BF16 or
 * F16), y may alias x; mask: see gbn_softmax_mask, NULL unless PADDING.
 * fp32 arithmetic.  Returns GBN_ERR_SHAPE for sk outside [1,
 * GBN_SOFTMAX_MAX_KEYS] or sq != sk with CAUSAL_UPPER; no rows: GBN_OK with
 * nothing enqueued. */
gbn_status gbn_softmax_fwd(const void* x, const uint8_t* mask, void* y, int64_t batches,
                           int64_t heads, int64_t sq, int64_t sk, int64_t mask_batches,
                           gbn_dtype dtype, gbn_softmax_mask mask_kind, float scale,
                           cudaStream_t stream);

/* Backward over `rows` rows of sk: dy, y, dx in dtype; dx may alias dy.
 * Masked positions have y = 0 and so dx = 0: no mask argument. */
gbn_status gbn_softmax_bwd(const void* dy, const void* y, void* dx, int64_t rows, int64_t sk,
                           gbn_dtype dtype, float scale, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char* gbn_status_string(gbn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H_ */
