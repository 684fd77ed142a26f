import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libhisa.so")


def pytest_terminal_summary(terminalreporter):
    """The worst error ratios of every parity check run (oracle/parity.py STATS)."""
    try:
        from oracle import parity
    except Exception:
        return
    if parity.STATS:
        terminalreporter.write_sep("-", "parity figures (worst per test)")
        terminalreporter.write_line(parity.format_stats())
