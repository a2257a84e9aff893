import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (tens of seconds)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The product library, built for sm_103a, on a machine with a GPU."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_indexer_pmqa_gb300 import pmqa

    pmqa.load()
    return pmqa
