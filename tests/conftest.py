import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """How the GPU parity checks used their tolerance (nothing when no GPU
    test ran)."""
    try:
        from gpu_setup import TOL_STATS
    except Exception:
        return
    if TOL_STATS["calls"]:
        terminalreporter.write_line(
            f"parity tolerance: {TOL_STATS['calls']} checks, {TOL_STATS['checked']} elements, "
            f"{TOL_STATS['needed_half_ulp']} inside the bound only through its half-ulp term, "
            f"worst |gpu - oracle| = {TOL_STATS['worst_frac_of_bound']:.3f} x the bound")
