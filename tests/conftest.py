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
