import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The parity record: per test, the worst normwise error (the pass bar)
    and the worst elementwise diagnostic |g - r| / max(|r|, 1e-3 max|r|) over
    the tensors it compared.  NT_PARITY_REPORT=<path> also writes every
    comparison as JSON."""
    try:
        from _helpers import PARITY_RECORD
    except ImportError:
        return
    if not PARITY_RECORD:
        return
    worst = {}
    for r in PARITY_RECORD:
        w = worst.setdefault(r["test"], {"normwise": 0.0, "elementwise": 0.0, "n": 0})
        w["normwise"] = max(w["normwise"], r["normwise"])
        w["elementwise"] = max(w["elementwise"], r["elementwise"])
        w["n"] += 1
    terminalreporter.write_sep("-", "parity: worst normwise / elementwise error per test")
    for name, w in sorted(worst.items()):
        terminalreporter.write_line(f"{w['normwise']:.3e}  {w['elementwise']:.3e}  ({w['n']})  {name}")
    path = os.environ.get("NT_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump({"per_test": worst, "comparisons": PARITY_RECORD}, f, indent=1)
