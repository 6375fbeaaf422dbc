import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libbkv.so")


def pytest_terminal_summary(terminalreporter):
    """The attention parity tests' worst errors (tests/_parity.py), one line per test."""
    mod = sys.modules.get("_parity")
    if mod is None or not getattr(mod, "WORST", None):
        return
    tr = terminalreporter
    tr.section("attention parity: worst error per test (relative = over the row's max |want|)")
    for key in sorted(mod.WORST):
        dtype, rows, err_abs, err_rel = mod.WORST[key]
        tr.write_line(f"{dtype:5s} rows {rows:7d}  abs {err_abs:.3e}  rel {err_rel:.3e}  {key}")
