import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # The library and the oracle are built from source in-tree (nvcc cross-compiles
    # without a GPU); a stale or missing build is rebuilt once per session.
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    oracle.build()


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The flat max-abs / mean-abs of every parity comparison that ran."""
    try:
        import harness
    except ImportError:
        return
    if not harness.RECORDS:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle (flat max-abs bar 1e-2, mean-abs 1e-3)")
    worst = max(r[1] for r in harness.RECORDS)
    for what, mx, mean, size, rounding in harness.RECORDS:
        tag = "  [bf16 output-rounding allowance]" if rounding else ""
        tr.write_line(f"{mx:.3e}  {mean:.3e}  {size:>10d}  {what}{tag}")
    tr.write_line(f"{len(harness.RECORDS)} comparisons; largest flat max-abs {worst:.3e}")
