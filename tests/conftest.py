import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _no_failed_index_check(request):
    """Under the bounds-checked build (TV_CHECKED=1), every GPU test must end
    with no failed index check recorded by the library."""
    yield
    if os.environ.get("TV_CHECKED", "0") in ("", "0") or request.node.get_closest_marker("gpu") is None:
        return
    import speculative_decoding_tree_tv_gb300 as tv
    site = tv.check_take()
    if request.node.name.startswith("test_selftest"):
        return
    assert site == 0, f"failed index check at unit {site >> 16}, line {site & 0xffff}"
