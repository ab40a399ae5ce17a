import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case, minutes of host time")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The margin check's report: per case, the rows whose selection was
    checked, the query rows the generator redrew to reach the 1e-3 margin,
    and the smallest k-th / (k+1)-th oracle score margin left."""
    harness = sys.modules.get("harness")
    if harness is None or not getattr(harness, "MARGIN_REPORT", None):
        return
    tr = terminalreporter
    tr.section("selection margins (oracle k-th minus (k+1)-th score)")
    tr.write_line("%-40s %10s %10s %8s %12s" % ("case", "rows", "ranked", "redrawn", "min margin"))
    for e in harness.MARGIN_REPORT:
        mm = "-" if e["min_margin"] is None else "%.3e" % e["min_margin"]
        tr.write_line("%-40s %10d %10d %8d %12s" % (e["case"], e["rows"], e["ranked_rows"], e["redrawn"], mm))
    path = os.environ.get("SSA_MARGIN_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(harness.MARGIN_REPORT, f, indent=1)
