import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden(name: str) -> dict:
    """key = value lines of a golden fixture (comments start with #)."""
    out = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = line.split("=", 1)
                out[k.strip()] = v.strip()
    return out


def golden_rows(name: str) -> list:
    rows = []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line and "=" not in line:
                rows.append(line)
    return rows


@pytest.fixture(scope="session")
def tqlib():
    """The built C-ABI library (built here if missing; nvcc cross-compiles without a GPU)."""
    from rotated_kv_cache_gb300 import build

    build.build()
    import rotated_kv_cache_gb300 as tqm

    return tqm


@pytest.fixture(scope="session")
def cuda(tqlib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return tqlib
