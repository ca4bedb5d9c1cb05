import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the disagreement budgets of the parity tests (decisions,
    disagreements, low-margin decisions), pass or fail."""
    import sys as _sys
    vh = _sys.modules.get("tests.verify_harness")
    if vh is None:
        return
    for line in vh.budget_lines():
        terminalreporter.write_line("disagreement budget: " + line)
