import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes")


def load_golden(name):
    """Parses a ``key = value`` fixture under tests/golden/ ('#' starts a comment)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            if re.fullmatch(r"[\[\]\d,.\-+eE\s]+", v) and re.search(r"\d", v):
                v = eval(v, {"__builtins__": {}})  # numbers and nested lists only
            out[k] = v
    return out


@pytest.fixture(scope="session")
def golden():
    return load_golden


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test that loaded the library: no kernel left a timeout
    (or, in the bounds-checked build, an out-of-bounds index) in the device
    status word, and the library is the build SHMM_CHECKED asks for."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from partial_sum_reduction_gb300 import shmm as m
    if m._lib is None:
        return
    import torch
    torch.cuda.synchronize()
    m.shmm_sync_status()
    assert m.shmm_bounds_checked() == (os.environ.get("SHMM_CHECKED") == "1")
