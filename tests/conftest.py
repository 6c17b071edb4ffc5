import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload; minutes")


def _need_build():
    from synth import HOST_SO
    import oracle
    return not (os.path.exists(HOST_SO) and os.path.exists(oracle.SO))


@pytest.fixture(scope="session", autouse=True)
def _built():
    """Build the host libraries once per session if they are missing."""
    if _need_build():
        import synth.build
        import oracle.build
        synth.build.build()
        oracle.build.build()
    yield
