import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")

import pytest  # noqa: E402


@pytest.fixture(scope="session")
def fbm_gpu():
    """The library, built in-tree for sm_103a, on a CUDA device."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fmha_block_map_gb300 import build

    build.build()
    import fmha_block_map_gb300 as fbm

    fbm.lib()
    return fbm
