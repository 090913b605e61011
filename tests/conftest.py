import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the kernels through the C-ABI")
    config.addinivalue_line("markers", "slow: full-size case (minutes of CPU time for the oracle)")


@pytest.fixture(scope="session", autouse=True)
def _host_libs():
    """Build the host-only helper libraries (generator, oracle) once per session."""
    import oracle
    import synth
    synth.build()
    oracle.build()
    yield
