import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session", autouse=True)
def _built_host_libs():
    """Compile the CPU oracle and the host input generator once per session."""
    import oracle
    import synth
    oracle.build()
    synth.build(gpu=False)
    yield
