import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_16_gb300 import binding
    return binding


def pytest_terminal_summary(terminalreporter):
    """Per parity test: requests compared with the oracle, how many were
    fully checked, how many had an open accept chain (left out), how many
    final tokens were checked against a set of admissible tokens, and how
    many requests held a decision margin below 1e-6."""
    try:
        from parity_helpers import COUNTS
    except ImportError:
        return
    if not COUNTS:
        return
    tr = terminalreporter
    tr.write_sep("-", "oracle parity counts (margin 1e-6)")
    tot = [0, 0, 0, 0, 0]
    for test, *vals in COUNTS:
        tot = [a + b for a, b in zip(tot, vals)]
        tr.write_line(f"{test}: requests {vals[0]}, checked {vals[1]}, open {vals[2]}, "
                      f"final sets {vals[3]}, near ties {vals[4]}")
    tr.write_line(f"TOTAL: requests {tot[0]}, checked {tot[1]}, open {tot[2]}, "
                  f"final sets {tot[3]}, near ties {tot[4]}")
