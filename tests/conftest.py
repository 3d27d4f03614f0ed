import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle as orc
    orc.build()
    return orc


@pytest.fixture(scope="session")
def ott():
    """The CUDA library's Python binding, on a GPU machine."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_kv_cache_ott_gb300 as pkg
    pkg.load()  # raises if the extension is missing: no fallback
    return pkg
