import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library's Python binding; fails loudly when it cannot be loaded."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    import causal_gqa_attention_row_gb300 as g
    g.load()  # raises if the shared library is missing
    return g


def pytest_terminal_summary(terminalreporter):
    """The largest error each parity comparison saw, beside its tolerance."""
    from margins import OBSERVED
    if not OBSERVED:
        return
    tr = terminalreporter
    tr.section("parity margins (max abs error observed / tolerance)")
    for test, what, err, tol in OBSERVED:
        tr.write_line(f"{err:10.3e} / {tol:7.1e}  ({err / tol:6.1%})  {test}{' ' + what if what else ''}")
    worst = max(OBSERVED, key=lambda r: r[2] / r[3])
    tr.write_line(f"closest to its bound: {worst[0]} {worst[1]} at {worst[2] / worst[3]:.1%} of the tolerance")
