import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libverkv")
    config.addinivalue_line("markers", "slow: long CPU statistics test")


def pytest_terminal_summary(terminalreporter):
    """One line with the GPU-vs-oracle parity counters of the run (heads compared, tie-swapped F
    sets and decisions, the largest errors and the largest g gap of a swapped token)."""
    mod = sys.modules.get("tests.parity")
    if mod is None or not mod.SUITE["heads"]:
        return
    terminalreporter.write_line("parity summary: " + " ".join(
        f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}" for k, v in mod.SUITE.items()))
