"""ctypes binding of libgbnorm.so (the C ABI declared in include/gbnorm.h).

Argument marshalling only: every function has the C name and argument order,
takes torch tensors (device memory) or None for pointers and Python numbers
for the scalars, and returns the integer status.  All computation happens in
the library's CUDA kernels.  Importing fails loudly if the library has not
been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbnorm.so")

# Enums of include/gbnorm.h.
GBN_LAYERNORM, GBN_RMSNORM = 0, 1
GBN_SCALING_NONE, GBN_SCALING_DELAYED_TENSOR, GBN_SCALING_MXFP8_1D = 0, 1, 2
GBN_LAYOUT_ROWWISE, GBN_LAYOUT_COLWISE, GBN_LAYOUT_ROWWISE_COLWISE = 0, 1, 2
GBN_LAYOUT_SWIZZLED_SCALES = 0x100  # OR-ed into the layout (MXFP8)
GBN_F32, GBN_BF16, GBN_F16, GBN_E4M3, GBN_E8M0 = 0, 1, 2, 3, 4
(GBN_OK, GBN_ERR_NULL, GBN_ERR_DTYPE, GBN_ERR_SHAPE, GBN_ERR_ALIGNMENT, GBN_ERR_WORKSPACE,
 GBN_ERR_ENUM, GBN_ERR_CUDA) = range(8)

TORCH_DTYPE = {torch.float32: GBN_F32, torch.bfloat16: GBN_BF16, torch.float16: GBN_F16}

FUNCTIONS = ("gbn_norm_fwd_workspace_size", "gbn_norm_fwd", "gbn_norm_bwd_workspace_size",
             "gbn_norm_bwd", "gbn_norm_bwd_noalloc", "gbn_device_error", "gbn_status_string",
             "gbn_softmax_fwd", "gbn_softmax_bwd", "gbn_selftest_copy_timeout")
(GBN_SOFTMAX_NO_MASK, GBN_SOFTMAX_PADDING, GBN_SOFTMAX_CAUSAL_UPPER,
 GBN_SOFTMAX_CAUSAL_ALIGNED) = range(4)
GBN_SOFTMAX_MAX_KEYS = 16384
GBN_DEVICE_ERR_COPY_TIMEOUT = 1


class GbnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {gbn_status_string(status)} ({status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -m "
            "rmsnorm_fp8_quantization_gb300._build); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I, F, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                        ctypes.c_size_t)
    lib.gbn_norm_fwd_workspace_size.argtypes = [I64, I64, I, I, I, I, I, I, I, I, I,
                                                ctypes.POINTER(SZ)]
    lib.gbn_norm_fwd_workspace_size.restype = I
    lib.gbn_norm_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, I64, I64,
                                 I, I, I, I, I, I, I, F, I, P]
    lib.gbn_norm_fwd.restype = I
    lib.gbn_norm_bwd_workspace_size.argtypes = [I64, I64, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.gbn_norm_bwd_workspace_size.restype = I
    lib.gbn_norm_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I64, I64, I, I, I, I, I, P]
    lib.gbn_norm_bwd.restype = I
    lib.gbn_norm_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I, I, I, I, I, P]
    lib.gbn_norm_bwd_noalloc.restype = I
    lib.gbn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
    lib.gbn_device_error.restype = I
    lib.gbn_softmax_fwd.argtypes = [P, P, P, I64, I64, I64, I64, I64, I, I, F, P]
    lib.gbn_softmax_fwd.restype = I
    lib.gbn_softmax_bwd.argtypes = [P, P, P, I64, I64, I, F, P]
    lib.gbn_softmax_bwd.restype = I
    lib.gbn_selftest_copy_timeout.argtypes = [ctypes.c_uint, P]
    lib.gbn_selftest_copy_timeout.restype = I
    lib.gbn_status_string.argtypes = [I]
    lib.gbn_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def library():
    """The loaded ctypes.CDLL (for symbol checks)."""
    return _lib


# Pointer arguments are passed as plain integers (the argtypes declare them
# c_void_p, so ctypes converts them); None is NULL.
def _ptr(t):
    if t is None or isinstance(t, int):
        return t
    return t.data_ptr()


# The current stream's handle without constructing a torch.cuda.Stream
# object (a few microseconds per call otherwise); the public call is the
# fallback where the raw accessor is not available.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gbn_status_string(status: int) -> str:
    return _lib.gbn_status_string(int(status)).decode()


def gbn_device_error(clear=True):
    """Returns (status, flags): the sticky device-side error bits."""
    v = ctypes.c_uint(0)
    st = _lib.gbn_device_error(ctypes.byref(v), int(bool(clear)))
    return st, v.value


def gbn_norm_fwd_workspace_size(rows, hidden, in_dtype, w_dtype, out_dtype, norm_type,
                                scaling_mode, quantize_layout, zero_centered_gamma, sm_margin,
                                is_training):
    """Returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = _lib.gbn_norm_fwd_workspace_size(rows, hidden, in_dtype, w_dtype, out_dtype, norm_type,
                                          scaling_mode, quantize_layout,
                                          int(bool(zero_centered_gamma)), sm_margin,
                                          int(bool(is_training)), ctypes.byref(n))
    return st, n.value


def gbn_norm_fwd(x, gamma, beta, scale, amax, out, colwise_out, mu, rsigma, scale_inv,
                 colwise_scale_inv, updated_amax, workspace, workspace_bytes, rows, hidden,
                 in_dtype, w_dtype, out_dtype, norm_type, scaling_mode, quantize_layout,
                 zero_centered_gamma, eps, sm_margin, stream=None) -> int:
    return _lib.gbn_norm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(scale), _ptr(amax), _ptr(out),
                             _ptr(colwise_out), _ptr(mu), _ptr(rsigma), _ptr(scale_inv),
                             _ptr(colwise_scale_inv), _ptr(updated_amax), _ptr(workspace),
                             workspace_bytes, rows, hidden, in_dtype, w_dtype, out_dtype,
                             norm_type, scaling_mode, quantize_layout,
                             int(bool(zero_centered_gamma)), float(eps), sm_margin,
                             _stream(stream))


def gbn_norm_bwd_workspace_size(rows, hidden, in_dtype, w_dtype, norm_type, zero_centered_gamma,
                                sm_margin):
    """Returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = _lib.gbn_norm_bwd_workspace_size(rows, hidden, in_dtype, w_dtype, norm_type,
                                          int(bool(zero_centered_gamma)), sm_margin,
                                          ctypes.byref(n))
    return st, n.value


def gbn_norm_bwd(dz, x, mu, rsigma, gamma, dresidual, dx, dgamma, dbeta, workspace,
                 workspace_bytes, rows, hidden, in_dtype, w_dtype, norm_type,
                 zero_centered_gamma, sm_margin, stream=None) -> int:
    return _lib.gbn_norm_bwd(_ptr(dz), _ptr(x), _ptr(mu), _ptr(rsigma), _ptr(gamma),
                             _ptr(dresidual), _ptr(dx), _ptr(dgamma), _ptr(dbeta),
                             _ptr(workspace), workspace_bytes, rows, hidden, in_dtype, w_dtype,
                             norm_type, int(bool(zero_centered_gamma)), sm_margin,
                             _stream(stream))


def gbn_norm_bwd_noalloc(dz, x, mu, rsigma, gamma, dresidual, dx, dgamma, dbeta, rows, hidden,
                         in_dtype, w_dtype, norm_type, zero_centered_gamma, sm_margin,
                         stream=None) -> int:
    """The backward on the library's fixed scratch array (no workspace)."""
    return _lib.gbn_norm_bwd_noalloc(_ptr(dz), _ptr(x), _ptr(mu), _ptr(rsigma), _ptr(gamma),
                                     _ptr(dresidual), _ptr(dx), _ptr(dgamma), _ptr(dbeta), rows,
                                     hidden, in_dtype, w_dtype, norm_type,
                                     int(bool(zero_centered_gamma)), sm_margin, _stream(stream))


def gbn_softmax_fwd(x, mask, y, batches, heads, sq, sk, mask_batches, dtype, mask_kind, scale,
                    stream=None) -> int:
    return _lib.gbn_softmax_fwd(_ptr(x), _ptr(mask), _ptr(y), batches, heads, sq, sk,
                                mask_batches, dtype, mask_kind, float(scale), _stream(stream))


def gbn_softmax_bwd(dy, y, dx, rows, sk, dtype, scale, stream=None) -> int:
    return _lib.gbn_softmax_bwd(_ptr(dy), _ptr(y), _ptr(dx), rows, sk, dtype, float(scale),
                                _stream(stream))


def gbn_selftest_copy_timeout(timeout_us, stream=None) -> int:
    """Enqueues the bounded-wait self-test kernel (see include/gbnorm.h)."""
    return _lib.gbn_selftest_copy_timeout(int(timeout_us), _stream(stream))
