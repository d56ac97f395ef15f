"""CPU oracle for the fused norm forward/backward and its FP8 quantizers.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
``cpu_baseline`` / ``--impl reference`` leg use it.  The product path (the
CUDA library and its binding) never imports it and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++, double
precision); this module compiles it with g++ and marshals numpy / torch CPU
arrays through ctypes.  Citations per function are in ``oracle.cpp``:
"Implementation:NVIDIA TransformerEngine JAX XLA Normalization" (sections
Description, I/O Contract) and "Implementation:NVIDIA TransformerEngine Ops
Fused Backward Add RMSNorm" (Description, I/O Contract), plus the OCP FP8 and
OCP MX v1.0 format definitions.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F16 = 0, 1, 2
LAYERNORM, RMSNORM = 0, 1


def build(force: bool = False) -> str:
    """Compiles ``oracle.cpp`` into ``liboracle.so`` (g++, -O2, strict IEEE)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I, D, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                           ctypes.c_double, ctypes.c_float)
        lib.orc_e4m3_encode.argtypes = [D]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = D
        lib.orc_e8m0_code.argtypes = [F]
        lib.orc_e8m0_code.restype = ctypes.c_uint8
        lib.orc_bf16_bits.argtypes = [D]
        lib.orc_bf16_bits.restype = ctypes.c_uint16
        lib.orc_f16_bits.argtypes = [D]
        lib.orc_f16_bits.restype = ctypes.c_uint16
        lib.orc_widen.argtypes = [P, I, I64]
        lib.orc_widen.restype = D
        lib.orc_round.argtypes = [P, I64, I, P]
        lib.orc_round.restype = None
        lib.orc_norm_fwd.argtypes = [P, I, P, P, I, I64, I64, I, I, D, P, P, P]
        lib.orc_norm_fwd.restype = I
        lib.orc_quant_delayed.argtypes = [P, I64, F, P, P, P]
        lib.orc_quant_delayed.restype = None
        lib.orc_mxfp8_rowwise.argtypes = [P, I64, I64, P, P]
        lib.orc_mxfp8_rowwise.restype = None
        lib.orc_mxfp8_colwise.argtypes = [P, I64, I64, P, P]
        lib.orc_mxfp8_colwise.restype = None
        lib.orc_norm_bwd.argtypes = [P, P, I, P, P, P, I, P, I64, I64, I, I, P, P, P]
        lib.orc_norm_bwd.restype = I
        _lib = lib
        return lib


# ---- marshalling helpers ------------------------------------------------------

def _raw(a):
    """(contiguous numpy array holding the stored bits, oracle dtype code)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype == torch.float32:
                return t.numpy(), F32
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy(), BF16
            if t.dtype == torch.float16:
                return t.view(torch.int16).numpy(), F16
            raise TypeError(f"oracle: unsupported torch dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float16:
        return a, F16
    raise TypeError(f"oracle: unsupported numpy dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---- scalar format primitives -------------------------------------------------

def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def e4m3_decode(c: int) -> float:
    return float(_load().orc_e4m3_decode(int(c)))


def e8m0_code(a: float) -> int:
    return int(_load().orc_e8m0_code(float(a)))


def bf16_bits(v: float) -> int:
    return int(_load().orc_bf16_bits(float(v)))


def f16_bits(v: float) -> int:
    return int(_load().orc_f16_bits(float(v)))


def widen(a) -> np.ndarray:
    """Exact float64 values of a stored f32 / bf16 / f16 array."""
    raw, dt = _raw(a)
    lib = _load()
    flat = raw.reshape(-1)
    return np.array([lib.orc_widen(_ptr(flat), dt, i) for i in range(flat.size)],
                    dtype=np.float64).reshape(raw.shape)


def round_to(v: np.ndarray, dtype: str):
    """Rounds float64 values once (RNE) into 'f32', 'bf16' or 'f16'.

    Returns a torch CPU tensor of that dtype.
    """
    import torch
    v = np.ascontiguousarray(v, dtype=np.float64)
    if dtype == "f32":
        out = np.empty(v.shape, dtype=np.float32)
        _load().orc_round(_ptr(v), v.size, F32, _ptr(out))
        return torch.from_numpy(out)
    bits = np.empty(v.shape, dtype=np.int16)
    code = BF16 if dtype == "bf16" else F16
    _load().orc_round(_ptr(v), v.size, code, _ptr(bits))
    t = torch.from_numpy(bits)
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


# ---- forward / backward ---------------------------------------------------------

def norm_fwd(x, gamma, beta, norm: int, zero_centered_gamma: bool, eps: float):
    """z, mu, rsigma (float64) of LayerNorm (norm=0) or RMSNorm (norm=1)."""
    xr, in_dt = _raw(x)
    gr, w_dt = _raw(gamma)
    br = None
    if beta is not None:
        br, b_dt = _raw(beta)
        assert b_dt == w_dt, "gamma and beta share one dtype"
    rows, hidden = xr.shape
    z = np.empty((rows, hidden), dtype=np.float64)
    mu = np.empty(rows, dtype=np.float64)
    rs = np.empty(rows, dtype=np.float64)
    _load().orc_norm_fwd(_ptr(xr), in_dt, _ptr(gr), _ptr(br), w_dt, rows, hidden, norm,
                         int(bool(zero_centered_gamma)), float(eps), _ptr(z), _ptr(mu),
                         _ptr(rs))
    return z, mu, rs


def quant_delayed(z: np.ndarray, scale: float):
    """(E4M3 codes uint8, amax fp32, scale_inv fp32) of delayed per-tensor scaling."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    q = np.empty(z.shape, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    sinv = np.zeros(1, dtype=np.float32)
    _load().orc_quant_delayed(_ptr(z), z.size, float(np.float32(scale)), _ptr(q), _ptr(amax),
                              _ptr(sinv))
    return q, amax[0], sinv[0]


def mxfp8_rowwise(z: np.ndarray):
    """(codes [rows, hidden] uint8, E8M0 scales [rows, hidden/32] uint8)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    rows, hidden = z.shape
    assert hidden % 32 == 0
    q = np.empty((rows, hidden), dtype=np.uint8)
    s = np.empty((rows, hidden // 32), dtype=np.uint8)
    _load().orc_mxfp8_rowwise(_ptr(z), rows, hidden, _ptr(q), _ptr(s))
    return q, s


def mxfp8_colwise(z: np.ndarray):
    """(codes [rows, hidden] uint8, E8M0 scales [rows/32, hidden] uint8)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    rows, hidden = z.shape
    assert rows % 32 == 0
    q = np.empty((rows, hidden), dtype=np.uint8)
    s = np.empty((rows // 32, hidden), dtype=np.uint8)
    _load().orc_mxfp8_colwise(_ptr(z), rows, hidden, _ptr(q), _ptr(s))
    return q, s


def mxfp8_swizzle(s: np.ndarray):
    """The padded, tiled GEMM order of an E8M0 scale matrix s [R, B] (R outer
    rows, B scales per row), built tile by tile: R and B are padded to
    R' = roundup(R, 128), B' = roundup(B, 4); the tiles of 128 rows x 4
    scales follow each other in row-major order, 512 bytes each; a tile is 32
    lines of 16 bytes, line i holding the 4 scales of rows i, i + 32, i + 64,
    i + 96, in that order.  (The layout has no counterpart on the pages; it
    is the order block-scaled GEMMs read.)

    Returns (bytes [R' * B'] uint8, mask of the bytes that hold a scale)."""
    s = np.asarray(s, dtype=np.uint8)
    R, B = s.shape
    Rp, Bp = (R + 127) // 128 * 128, (B + 3) // 4 * 4
    out = np.zeros(Rp * Bp, dtype=np.uint8)
    held = np.zeros(Rp * Bp, dtype=bool)
    pos = 0
    for tr in range(Rp // 128):
        for tc in range(Bp // 4):
            for line in range(32):
                for quarter in range(4):
                    r = tr * 128 + quarter * 32 + line
                    for c4 in range(4):
                        c = tc * 4 + c4
                        if r < R and c < B:
                            out[pos] = s[r, c]
                            held[pos] = True
                        pos += 1
    return out, held


def norm_bwd(dz, x, mu, rsigma, gamma, dresidual, norm: int, zero_centered_gamma: bool):
    """dx [rows, hidden], dgamma [hidden], dbeta [hidden] (float64).

    ``mu`` / ``rsigma`` are the saved fp32 statistics (numpy float32 or torch).
    ``dbeta`` is None for RMSNorm.
    """
    dzr, in_dt = _raw(dz)
    xr, x_dt = _raw(x)
    assert x_dt == in_dt
    gr, w_dt = _raw(gamma)
    dr = None
    if dresidual is not None:
        dr, d_dt = _raw(dresidual)
        assert d_dt == in_dt
    rows, hidden = xr.shape
    rs = np.ascontiguousarray(np.asarray(rsigma, dtype=np.float32))
    mu_a = None if mu is None else np.ascontiguousarray(np.asarray(mu, dtype=np.float32))
    dx = np.empty((rows, hidden), dtype=np.float64)
    dg = np.empty(hidden, dtype=np.float64)
    db = np.empty(hidden, dtype=np.float64) if norm == LAYERNORM else None
    _load().orc_norm_bwd(_ptr(dzr), _ptr(xr), in_dt, _ptr(mu_a), _ptr(rs), _ptr(gr), w_dt,
                         _ptr(dr), rows, hidden, norm, int(bool(zero_centered_gamma)),
                         _ptr(dx), _ptr(dg), _ptr(db))
    return dx, dg, db
