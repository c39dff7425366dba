"""Shared pytest configuration: the ``gpu`` marker and repo-root imports."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    """Exemption counts of the write-parity cases that ran (the near-boundary rule for packed codes)."""
    try:
        from tests.harness import EXEMPTION_LOG
    except Exception:
        return
    if not EXEMPTION_LOG:
        return
    terminalreporter.write_line("write parity exemptions (case: exempt / codes compared, by kind):")
    for case, n, e, kinds in EXEMPTION_LOG:
        terminalreporter.write_line(f"  {case}: {e} / {n} ({e / max(n, 1):.2e}) {kinds}")
