"""Shared test configuration: markers and import paths.

``-m gpu`` tests need a GB300 and the CUDA library; everything else runs on a
CPU-only host (oracle pins, host-side logic, the library's exported symbols).
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: longer CPU-only checks")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Every GPU-vs-oracle comparison of the session, and how many drawn
    tokens differed only inside the boundary band (printed under -q too)."""
    try:
        from oracle import compare
    except Exception:
        return
    t = compare.TALLY
    if t["sequences"] == 0:
        return
    terminalreporter.write_line(compare.tally_line())
    for label, cases in t["cases"]:
        terminalreporter.write_line(f"  boundary cases{f' ({label})' if label else ''}: {cases}")
