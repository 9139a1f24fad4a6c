import os
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_sessionstart(session):
    # The package refuses to import without its compiled library; build it
    # (and the oracle) first when this checkout has not been built yet.
    lib = os.path.join(ROOT, "dropout_lowbias32_hash32_gb300", "_lib", "librng_lowbias32.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__.build()


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
