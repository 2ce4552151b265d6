import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libqmlp.so")
    config.addinivalue_line("markers", "slow: large oracle work (still CPU)")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def cuda_available():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test requested but torch.cuda.is_available() is False (a CPU skip is not a GPU pass)")
    return True
