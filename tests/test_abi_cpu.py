"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/gbnorm.h declares, and rejects bad arguments before touching
CUDA."""
import os
import re

import pytest
import torch

from conftest import ROOT


@pytest.fixture(scope="module")
def G():
    from rmsnorm_fp8_quantization_gb300 import _build
    _build.build()
    from rmsnorm_fp8_quantization_gb300 import gbnorm
    return gbnorm


def _header_functions():
    text = open(os.path.join(ROOT, "include", "gbnorm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gbn_\w+)\s*\(", text)))


def test_header_functions_are_exported(G):
    names = _header_functions()
    assert set(names) == set(G.FUNCTIONS), names
    lib = G.library()
    for n in names:
        assert hasattr(lib, n), n


def test_header_enums_match_binding(G):
    text = open(os.path.join(ROOT, "include", "gbnorm.h")).read()
    for name, val in re.findall(r"\b(GBN_[A-Z0-9_]+)\s*=\s*(0x[0-9a-fA-F]+|\d+)", text):
        assert getattr(G, name) == int(val, 0), name


def test_status_strings(G):
    for s in range(8):
        assert G.gbn_status_string(s).startswith("GBN_")


def _fwd(G, **kw):
    args = dict(x=None, gamma=None, beta=None, scale=None, amax=None, out=None, colwise_out=None,
                mu=None, rsigma=None, scale_inv=None, colwise_scale_inv=None, updated_amax=None,
                workspace=None, workspace_bytes=0, rows=64, hidden=1024, in_dtype=G.GBN_BF16,
                w_dtype=G.GBN_F32, out_dtype=G.GBN_BF16, norm_type=G.GBN_LAYERNORM,
                scaling_mode=G.GBN_SCALING_NONE, quantize_layout=G.GBN_LAYOUT_ROWWISE,
                zero_centered_gamma=0, eps=1e-5, sm_margin=0, stream=0)
    args.update(kw)
    return G.gbn_norm_fwd(**args)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def test_fwd_validation_without_gpu(G):
    assert _fwd(G) == G.GBN_ERR_NULL
    assert _fwd(G, x=FAKE, gamma=FAKE, out=FAKE) == G.GBN_ERR_NULL          # LayerNorm needs beta
    assert _fwd(G, norm_type=7) == G.GBN_ERR_ENUM
    assert _fwd(G, scaling_mode=3) == G.GBN_ERR_ENUM
    assert _fwd(G, quantize_layout=-1) == G.GBN_ERR_ENUM
    assert _fwd(G, out_dtype=G.GBN_F32) == G.GBN_ERR_DTYPE                  # unquantized: out = in
    assert _fwd(G, scaling_mode=G.GBN_SCALING_DELAYED_TENSOR) == G.GBN_ERR_DTYPE  # needs E4M3
    assert _fwd(G, in_dtype=G.GBN_E4M3) == G.GBN_ERR_DTYPE
    assert _fwd(G, hidden=0) == G.GBN_ERR_SHAPE
    assert _fwd(G, rows=-1) == G.GBN_ERR_SHAPE
    assert _fwd(G, hidden=(1 << 24) + 1) == G.GBN_ERR_SHAPE                 # past the largest row
    assert _fwd(G, hidden=1 << 24) == G.GBN_ERR_NULL                         # the largest passes shape
    mx = dict(scaling_mode=G.GBN_SCALING_MXFP8_1D, out_dtype=G.GBN_E4M3)
    assert _fwd(G, hidden=48, **mx) == G.GBN_ERR_SHAPE                       # blocks of 32
    assert _fwd(G, rows=40, quantize_layout=G.GBN_LAYOUT_COLWISE, **mx) == G.GBN_ERR_SHAPE
    dl = dict(scaling_mode=G.GBN_SCALING_DELAYED_TENSOR, out_dtype=G.GBN_E4M3,
              norm_type=G.GBN_RMSNORM, x=FAKE, gamma=FAKE, out=FAKE)
    assert _fwd(G, **dl) == G.GBN_ERR_NULL                                   # scale, updated_amax
    assert _fwd(G, quantize_layout=G.GBN_LAYOUT_COLWISE, scale=FAKE, updated_amax=FAKE,
                **dl) == G.GBN_ERR_NULL                                      # colwise_out


def test_fwd_workspace_size(G):
    """Zero except for the columnwise FP8 layouts of rows longer than one CTA's
    ring (room for rsigma, and mu for LayerNorm, rounded up to 256 bytes);
    computed on the host, no device needed."""
    q = lambda rows, hidden, in_dt, norm, sc, lay: G.gbn_norm_fwd_workspace_size(
        rows, hidden, in_dt, G.GBN_BF16, G.GBN_BF16 if sc == G.GBN_SCALING_NONE else G.GBN_E4M3,
        norm, sc, lay, 0, 0, 0)
    assert q(16384, 4096, G.GBN_BF16, G.GBN_LAYERNORM, G.GBN_SCALING_NONE,
             G.GBN_LAYOUT_ROWWISE) == (G.GBN_OK, 0)
    # rows that fit one CTA's ring, or rowwise only: none
    assert q(1024, 16384, G.GBN_BF16, G.GBN_RMSNORM, G.GBN_SCALING_DELAYED_TENSOR,
             G.GBN_LAYOUT_ROWWISE_COLWISE) == (G.GBN_OK, 0)
    assert q(1024, 65536, G.GBN_BF16, G.GBN_RMSNORM, G.GBN_SCALING_DELAYED_TENSOR,
             G.GBN_LAYOUT_ROWWISE) == (G.GBN_OK, 0)
    # long rows, columnwise: 4 bytes per row (RMSNorm), 8 (LayerNorm)
    assert q(1024, 65536, G.GBN_BF16, G.GBN_RMSNORM, G.GBN_SCALING_DELAYED_TENSOR,
             G.GBN_LAYOUT_COLWISE) == (G.GBN_OK, 4096)
    assert q(96, 18464, G.GBN_BF16, G.GBN_LAYERNORM, G.GBN_SCALING_MXFP8_1D,
             G.GBN_LAYOUT_ROWWISE_COLWISE) == (G.GBN_OK, 768)
    assert q(64, 18432, G.GBN_BF16, G.GBN_LAYERNORM, G.GBN_SCALING_MXFP8_1D,
             G.GBN_LAYOUT_COLWISE) == (G.GBN_OK, 0)  # the widest ring row
    assert q(64, 9248, G.GBN_F32, G.GBN_LAYERNORM, G.GBN_SCALING_MXFP8_1D,
             G.GBN_LAYOUT_COLWISE | G.GBN_LAYOUT_SWIZZLED_SCALES) == (G.GBN_OK, 512)
    # ragged rows take the generic kernel: none
    assert q(1000, 65536, G.GBN_BF16, G.GBN_RMSNORM, G.GBN_SCALING_DELAYED_TENSOR,
             G.GBN_LAYOUT_COLWISE) == (G.GBN_OK, 0)
    st, _ = G.gbn_norm_fwd_workspace_size(16384, 4008, G.GBN_BF16, G.GBN_BF16, G.GBN_E4M3,
                                          G.GBN_RMSNORM, G.GBN_SCALING_MXFP8_1D,
                                          G.GBN_LAYOUT_ROWWISE, 0, 0, 1)
    assert st == G.GBN_ERR_SHAPE


def _bwd(G, **kw):
    args = dict(dz=None, x=None, mu=None, rsigma=None, gamma=None, dresidual=None, dx=None,
                dgamma=None, dbeta=None, workspace=None, workspace_bytes=0, rows=64, hidden=1024,
                in_dtype=G.GBN_BF16, w_dtype=G.GBN_BF16, norm_type=G.GBN_RMSNORM,
                zero_centered_gamma=0, sm_margin=0, stream=0)
    args.update(kw)
    return G.gbn_norm_bwd(**args)


def test_bwd_validation_without_gpu(G):
    ok = dict(dz=FAKE, x=FAKE, rsigma=FAKE, gamma=FAKE, dx=FAKE, dgamma=FAKE)
    assert _bwd(G) == G.GBN_ERR_NULL
    assert _bwd(G, norm_type=2, **ok) == G.GBN_ERR_ENUM
    assert _bwd(G, w_dtype=G.GBN_E8M0, **ok) == G.GBN_ERR_DTYPE
    assert _bwd(G, hidden=0, **ok) == G.GBN_ERR_SHAPE
    assert _bwd(G, hidden=(1 << 24) + 1, **ok) == G.GBN_ERR_SHAPE
    assert _bwd(G, rows=-1, **ok) == G.GBN_ERR_SHAPE
    assert _bwd(G, norm_type=G.GBN_LAYERNORM, **ok) == G.GBN_ERR_NULL       # mu, dbeta
    assert _bwd(G, **ok) == G.GBN_ERR_WORKSPACE                             # no workspace
    assert _bwd(G, workspace=FAKE + 4, **ok) == G.GBN_ERR_WORKSPACE         # misaligned


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_bwd_workspace_query_without_device_reports_cuda_error(G):
    st, _ = G.gbn_norm_bwd_workspace_size(64, 1024, G.GBN_BF16, G.GBN_BF16, G.GBN_RMSNORM, 0, 0)
    assert st == G.GBN_ERR_CUDA


def test_header_compiles_as_c99_and_cpp17(tmp_path):
    import shutil
    import subprocess
    cuda_inc = "/usr/local/cuda/include"
    if not shutil.which("gcc") or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    src = tmp_path / "use.c"
    src.write_text('#include "gbnorm.h"\n'
                   "int main(void) {\n"
                   "  gbn_quantize_layout l = (gbn_quantize_layout)(GBN_LAYOUT_ROWWISE |\n"
                   "                                                GBN_LAYOUT_SWIZZLED_SCALES);\n"
                   "  (void)l; (void)&gbn_norm_fwd; (void)&gbn_softmax_fwd;\n"
                   "  return 0;\n}\n")
    inc = ["-I", os.path.join(ROOT, "include"), "-I", cuda_inc]
    for cmd in (["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", *inc, str(src)],
                ["g++", "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", *inc,
                 str(src)]):
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
