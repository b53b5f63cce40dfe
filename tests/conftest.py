import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs on the GB300 box")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def libgemm():
    """The built library's binding (builds libgemm.so first if it is stale)."""
    from accelerator_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


class _OracleCache:
    """Memoised oracle results keyed by the seeded-input recipe."""

    def __init__(self):
        self._full = {}

    def full(self, key, A, B, fmt="f32"):
        import oracle
        k = (key, fmt)
        if k not in self._full:
            self._full[k] = oracle.gemm(A, B, fmt=fmt)
        return self._full[k]


@pytest.fixture(scope="session")
def oracle_cache():
    return _OracleCache()
