import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_PARITY_LINES = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "perf: performance measurement, not a correctness check")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a visible CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def parity_report():
    """Lines (one per full-output parity case) printed in the run's summary."""
    return _PARITY_LINES


def pytest_terminal_summary(terminalreporter):
    if _PARITY_LINES:
        terminalreporter.write_sep("-", "full-output parity against the oracle")
        for line in _PARITY_LINES:
            terminalreporter.write_line(line)
