import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


@pytest.fixture(autouse=True)
def no_failed_bound_checks(request):
    """Under a bounds-checking debug build of the library (ROPE3D_LIB), every
    GPU test must end with no failed index check."""
    yield
    if request.node.get_closest_marker("gpu") is None or not os.environ.get("ROPE3D_LIB"):
        return
    import rope_rope3d_apply_gb300 as r

    built, errors = r.rope3d_debug_bounds(reset=True)
    if built:
        assert errors == 0, f"{errors} failed bound checks"
