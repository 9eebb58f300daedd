import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size case (minutes)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def V():
    """The CUDA library's binding, built first if its sources are newer (the
    build is incremental); GPU tests skip where there is no CUDA device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_attention_video_smooth_gb300 import build
    build.build()
    from bit_attention_video_smooth_gb300 import vca
    return vca
