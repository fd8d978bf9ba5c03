import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library on a B300)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Raw and allowed output errors of the GPU parity checks (tests/gpu_util.py check_close):
    the worst check of each test file, and every full-size check."""
    mod = sys.modules.get("gpu_util")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", "output error vs the oracle, in rms(ref): raw / after half a bf16 ulp (tolerance)")
    worst = {}
    for test, what, raw, err, tol in recs:
        f = test.split("::")[0].split("/")[-1]
        if f not in worst or err / tol > worst[f][3] / worst[f][4]:
            worst[f] = (test, what, raw, err, tol)
    for f, (test, what, raw, err, tol) in sorted(worst.items()):
        tr.write_line("worst of %d in %s: %.2e / %.2e (%g)  %s %s" % (
            sum(1 for r in recs if r[0].split("::")[0].split("/")[-1] == f), f, raw, err, tol,
            test.split("::", 1)[-1], what))
    for test, what, raw, err, tol in recs:
        if "full_size" in test:
            tr.write_line("%.2e / %.2e (%g)  %s %s" % (raw, err, tol, test.split("::", 1)[-1], what))
