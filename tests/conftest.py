import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


def pytest_terminal_summary(terminalreporter):
    """The literal-tolerance report of the GPU parity tests (elements outside
    |gpu - oracle| <= 1e-2 + 1e-2 |oracle| against the plain definition, per tensor) and the
    near-tie counts of the routing checks."""
    mod = sys.modules.get("gpu_common")
    rep = getattr(mod, "REPORT", None)
    if not rep or not (rep["plain"] or rep["near_ties"]):
        return
    import json
    tr = terminalreporter
    tr.section("parity with the plain definition (literal tolerance)")
    if rep["near_ties"]:
        tr.write_line("near-tie tokens (adjacent top-(k+1) selection gap < 1e-6):")
        for r in rep["near_ties"]:
            tr.write_line(f"  {r['case']:32s} {r['near_ties']:6d} of {r['tokens']}")
    tr.write_line("case / tensor: elements outside, worst excess; bf16 storage alone: outside, worst")
    for r in rep["plain"]:
        tr.write_line(f"  {r['case']:28s} {r['tensor']:8s} {r['exceed']:8d}/{r['size']:<10d} "
                      f"{r['worst_excess']:+.2e}   storage {r['storage_exceed']:8d} "
                      f"{r['storage_worst_excess']:+.2e}")
    path = os.environ.get("MOE_PARITY_REPORT")
    if path:
        with open(path, "w") as fh:
            json.dump(rep, fh, indent=1)
