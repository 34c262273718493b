import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library (fails loudly if it is missing on a GPU machine)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu-marked test run without a CUDA device")
    from tiled_memory_efficient_gb300 import _lib
    return _lib.load()


def pytest_terminal_summary(terminalreporter):
    """Per-comparison parity record of the GPU tests: largest error against
    the fp64 oracle, the tolerance, and how many elements needed the widened
    bound (half an ulp of the stored dtype above the tolerance)."""
    try:
        from tests import helpers
    except Exception:
        return
    if not helpers.RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity records ({len(helpers.RECORDS)} comparisons)")
    for what, name, n, emax, tol, nw, eflat, rmax in helpers.RECORDS:
        tr.write_line(f"{what[:70]:70s} {name:3s} n={n:<10d} max={emax:.2e} tol={tol:g} "
                      f"flat_max={eflat:.2e} widened={nw} max|ref|={rmax:.2f}")
    # the summary last, so that the end of the log carries it
    widened = [r for r in helpers.RECORDS if r[5] > 0]
    tr.write_line(f"comparisons with elements under the widened bound: {len(widened)}")
    worst_flat = {}
    for what, name, n, emax, tol, nw, eflat, rmax in helpers.RECORDS:
        key = (name, tol)
        if eflat / tol >= worst_flat.get(key, (-1.0, ""))[0]:
            worst_flat[key] = (eflat / tol, what)
    for (name, tol), (ratio, what) in sorted(worst_flat.items()):
        tr.write_line(f"worst {name} (tol {tol:g}) under the flat bound: {ratio:.2f} x tol in {what}")
