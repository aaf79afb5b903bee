import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case (full-size configs)")


@pytest.fixture(scope="session", autouse=True)
def _built_host_libs():
    """Host-side libraries (datagen, oracle) are compiled once per session if missing."""
    import datagen
    import oracle
    if not os.path.exists(os.path.join(ROOT, "datagen", "libdg_host.so")):
        datagen.build()
    if not os.path.exists(os.path.join(ROOT, "oracle", "libmsa_oracle.so")):
        oracle.build()
    yield


_PARITY_LOG = []


@pytest.fixture
def parity_log(request):
    """Records a parity report (set counts: rows, mismatches, near-tie rows, strict-invalid rows; attention:
    max abs / rel error and cosine).  The reports are printed, and written as JSON at the end of the session
    to the path in MSA_PARITY_REPORT when that variable is set."""
    def log(case, **reports):
        _PARITY_LOG.append(dict(test=request.node.nodeid, case=case, **reports))
        print(case, reports)
    return log


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("MSA_PARITY_REPORT")
    if path and _PARITY_LOG:
        with open(path, "w") as f:
            json.dump(_PARITY_LOG, f, indent=1)
