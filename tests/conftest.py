import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _no_out_of_range_access():
    """Under the bounds-checked library (CTP_LIBRARY_VARIANT=check) every test
    must end with no walk access outside its buffer."""
    yield
    if os.environ.get("CTP_LIBRARY_VARIANT") != "check":
        return
    import back_projection_ctp_b300._binding as b
    if b._lib is None:
        return
    count, index, extent, site = b.ctp_check_violations()
    assert count == 0, f"{count} out-of-range accesses (first: index {index} of {extent}, site {site})"
