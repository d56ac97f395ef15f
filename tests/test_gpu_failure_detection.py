"""Failure detection without a GPU fault: a kernel's bounded wait for a copy
that never lands gives up, records GBN_DEVICE_ERR_COPY_TIMEOUT in the sticky
device flag, and returns; the host reads the flag, clears it, and the
context keeps working (no trap, no assert, no hang)."""
import pytest
import torch

from rmsnorm_fp8_quantization_gb300 import gbnorm as G
from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_sets_the_flag_and_the_context_survives(gpu):
    st, _ = G.gbn_device_error(clear=True)
    assert st == G.GBN_OK
    assert G.gbn_selftest_copy_timeout(20000) == G.GBN_OK      # 20 ms
    torch.cuda.synchronize()
    st, flags = G.gbn_device_error(clear=True)
    assert st == G.GBN_OK and flags & G.GBN_DEVICE_ERR_COPY_TIMEOUT
    st, flags = G.gbn_device_error(clear=False)
    assert flags == 0, "clear did not reset the flag"

    # the context is still usable: a normal call runs and raises no flag
    w = WORKLOADS["ln_bf16_16384x4096"].with_shape(64)
    inp = make_inputs(w)
    out = gpu.norm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda(),
                       norm="layernorm", eps=w.eps)
    torch.cuda.synchronize()
    assert torch.isfinite(out["out"].float()).all()
    st, flags = G.gbn_device_error(clear=False)
    assert st == G.GBN_OK and flags == 0


def test_selftest_rejects_out_of_range_limits(gpu):
    assert G.gbn_selftest_copy_timeout(0) == G.GBN_ERR_SHAPE
    assert G.gbn_selftest_copy_timeout(2000001) == G.GBN_ERR_SHAPE
