import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU statistical test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    return oracle


@pytest.fixture(scope="session")
def tsv():
    """The GPU library's Python binding (builds the shared library if missing)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verification_attention_gb300 as t

    return t
