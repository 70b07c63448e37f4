"""Shared pytest configuration: the `gpu` marker and repo-root imports."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The parity tests' exempt decisions (oracle margin below 1e-4), per test."""
    try:
        from tests.gpu_harness import EXEMPT
    except Exception:
        return
    if not EXEMPT:
        return
    tr = terminalreporter
    tr.section("exempt decisions (oracle margin < 1e-4)")
    tot_e = tot_n = 0
    for test, kind, e, n in EXEMPT:
        tr.write_line(f"{e:6d} / {n:8d}  {kind:16s} {test}")
        tot_e += e
        tot_n += n
    tr.write_line(f"{tot_e:6d} / {tot_n:8d}  in all")
