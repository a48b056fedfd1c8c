import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")


def pytest_terminal_summary(terminalreporter):
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "REPORT", None):
        return
    terminalreporter.write_sep("-", "boundary exclusions of the full-size workloads")
    for name, (stats, extra) in sorted(parity.REPORT.items()):
        terminalreporter.write_line(f"{name}: {stats} {extra}".rstrip())
