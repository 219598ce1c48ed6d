import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The information-only flip counts of the GPU parity tests: the oracle's
    selection on its own block sums against the GPU's selection."""
    mod = sys.modules.get("gpu_common")
    flips = getattr(mod, "FLIPS", None) if mod else None
    if not flips:
        return
    tr = terminalreporter
    tr.section("selection flips: oracle on its own block sums vs GPU (information only)")
    for what, mflips, n, sflips in flips:
        sel = "" if sflips is None else f", selected blocks differing: {sflips}"
        tr.write_line(f"{what}: mask entries differing {mflips} of {n}{sel}")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when the device or library is missing;
    # nothing here silently downgrades them to CPU.
    pass
