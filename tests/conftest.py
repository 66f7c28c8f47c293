"""Shared test set-up: markers, paths, the oracle build and GPU helpers."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)  # results do not depend on the thread count
    return oracle


@pytest.fixture(scope="session")
def cuda():
    """The CUDA library binding; GPU tests need a device and fail loudly when
    the compiled library is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import csa2_sparse_attention_03_b300 as csa2
    csa2.load()  # raises if libcsa2.so is absent
    return csa2
