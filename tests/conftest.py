import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity at the benchmark's workload sizes")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)

    return load


def pytest_sessionfinish(session, exitstatus):
    """Write the float-parity margins of the GPU tests (if any ran) to the
    directory named by PARITY_REPORT_DIR (no report without it)."""
    mod = sys.modules.get("tests.gpu_util")
    rep = getattr(mod, "REPORT", None) if mod else None
    out = os.environ.get("PARITY_REPORT_DIR")
    if not rep or not out:
        return
    os.makedirs(out, exist_ok=True)
    name = os.environ.get("PARITY_REPORT", "parity_report.txt")
    with open(os.path.join(out, name), "a") as f:
        for what, err, rms, ratio in rep:
            f.write(f"{what}\tmax_err={err:.4e}\trms={rms:.4e}\tratio={ratio:.4e}\n")
