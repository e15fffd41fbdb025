import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Near-tie rows of the fused-head tests: counted and reported, not failed."""
    from near_ties import NEAR_TIE, RECORDS
    if not RECORDS:
        return
    terminalreporter.section(f"near ties (oracle top-2 gap < {NEAR_TIE:g})")
    for name, n, rows, checked, total in RECORDS:
        terminalreporter.write_line(f"{name}: {n} of {rows} rows; planted length checked on {checked} of "
                                    f"{total} requests")
