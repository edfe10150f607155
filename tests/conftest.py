import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqkv.so")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of host time")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.Oracle()


@pytest.fixture(scope="session")
def qkv():
    """The product binding on a GPU; fails loudly when the CUDA library is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected on a machine without CUDA")
    import qkv_rope_kv_gb300 as q
    q.load()
    return q


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One line with the largest parity errors of every GPU comparison made in this run."""
    gh = sys.modules.get("gpu_helpers")
    line = gh.parity_summary() if gh is not None else ""
    if line:
        terminalreporter.write_line(line)
