import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the errors of every GPU parity comparison of the session: per
    tensor the Frobenius relative error, the worst row's relative error and
    the largest absolute error (gpu_helpers.errors)."""
    helpers = sys.modules.get("gpu_helpers")
    report = getattr(helpers, "REPORT", None)
    if not report:
        return
    tr = terminalreporter
    tr.section("parity errors against the oracle (frob, worst row, max abs)")
    worst = {}
    for test, key, frob, row, maxabs in report:
        tr.write_line(f"{test}  {key:10s} {frob:.3e} {row:.3e} {maxabs:.3e}")
        w = worst.get(key)
        worst[key] = (max(frob, w[0]), max(row, w[1]), max(maxabs, w[2])) if w else (frob, row, maxabs)
    tr.write_line("worst per tensor over the session:")
    for key, (frob, row, maxabs) in sorted(worst.items()):
        tr.write_line(f"  {key:10s} {frob:.3e} {row:.3e} {maxabs:.3e}")
