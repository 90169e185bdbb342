import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")


def bits(x) -> np.ndarray:
    """Round float values to bf16 (RNE) and return the uint16 bit patterns."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_value(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture
def rng():
    return np.random.default_rng(12345)
