import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def ref():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    from tests import _parity
    if _parity.LOG:
        exc = sum(e for _, e, _ in _parity.LOG)
        dec = sum(d for _, _, d in _parity.LOG)
        terminalreporter.write_line(f"near-tie decisions excused: {exc} of {dec} compared in {len(_parity.LOG)} checks")
        for what, e, d in _parity.LOG:
            if e:
                terminalreporter.write_line(f"  {what}: {e} of {d}")
