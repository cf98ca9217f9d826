import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Lines of a golden fixture without comments or blank lines, split."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def fc_lib():
    """The CUDA library, built in-tree if it is missing."""
    from gradient_aggregation_gb300 import build as fcbuild
    fcbuild.build_library()
    from gradient_aggregation_gb300 import fc
    return fc.lib()
