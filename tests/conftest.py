import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes")


def pytest_terminal_summary(terminalreporter):
    """The worst LSE error each GPU parity test saw, against the tolerance it used."""
    mod = sys.modules.get("tests.mla_cases")
    log = getattr(mod, "LSE_LOG", None)
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "worst |lse_gpu - lse_oracle| per test (tolerance, ratio)")
    for key, (err, ratio, tol) in sorted(log.items()):
        tr.write_line(f"{err:10.3e}  tol {tol:9.3e}  ratio {ratio:6.3f}  {key}")
