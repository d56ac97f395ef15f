import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Rows of whitespace-separated fields from tests/golden/<name>, comments dropped."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def parse_float(s):
    s = s.strip()
    if s.lower().startswith(("0x", "-0x")):
        return float.fromhex(s)
    return float(s)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def gpu():
    """The built library's allocating wrappers, on a CUDA device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fp8_quantization_gb300 import _build
    _build.build()
    from rmsnorm_fp8_quantization_gb300 import ops
    return ops
