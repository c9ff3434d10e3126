import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large workload (full-size shapes)")


def read_golden(name):
    """Parse a whitespace table under tests/golden/: key -> (values, tol)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            out[parts[0]] = ([float(x) for x in parts[1:-1]], float(parts[-1]))
    return out


@pytest.fixture
def golden():
    return read_golden


@pytest.fixture(scope="session")
def built_library():
    """Build libattn_fa2.so if it is missing or stale (nvcc cross-compiles for
    sm_103a without a GPU) and return its path."""
    from tiled_attention_fa2_gb300 import _build

    return _build.build()


def pytest_sessionfinish(session, exitstatus):
    """Write the measured parity errors (ATTN_PARITY_REPORT=path.json)."""
    path = os.environ.get("ATTN_PARITY_REPORT")
    if not path:
        return
    try:
        from parity import REPORT
    except ImportError:
        return
    import json

    with open(path, "w") as f:
        json.dump(REPORT, f, indent=1)
