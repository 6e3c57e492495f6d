import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def read_golden(name):
    """Parse a tests/golden fixture: 'key: ints...' lines, '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [int(t) for t in v.split()]
    return out


@pytest.fixture(scope="session")
def rs():
    """The CUDA library, built for sm_103a and loaded (GPU tests only)."""
    from lsd_radix_sort_gb300 import build
    build.build()
    import lsd_radix_sort_gb300 as mod
    mod.load_library()
    return mod
