import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running parity case")


def pytest_terminal_summary(terminalreporter):
    """Per-check counts of forward O elements above the flat bound (the
    exceptions that the derived bound of tests/parity.py then covers)."""
    parity = sys.modules.get("parity")
    rows = getattr(parity, "O_EXCEPTIONS", None)
    if not rows:
        return
    total = sum(n for _, n, _ in rows)
    above = sum(b for _, _, b in rows)
    terminalreporter.section("forward O: elements above max(1e-2, 1 bf16 ulp)")
    terminalreporter.write_line(f"{len(rows)} checks, {total} elements checked, {above} above the flat bound")
    for what, n, b in rows:
        if b:
            terminalreporter.write_line(f"  {b} of {n}: {what}")
