"""Shared pytest configuration: markers, import paths and session fixtures."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_addoption(parser):
    parser.addoption("--dc-bounds", action="store_true",
                     help="build the bounds-checked library (libdc_bounds.so) and run every test "
                          "against it; each GPU test then also fails if a kernel skipped an "
                          "access outside its job's range (DC_ERR_BOUNDS)")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")
    if config.getoption("--dc-bounds"):
        from reduce_copy_rank_gb300 import _build

        _build.build(bounds=True)
        os.environ["DC_LIBRARY"] = "bounds"


@pytest.fixture(autouse=True)
def _no_bounds_fault(request):
    """With --dc-bounds: after every GPU test, no kernel may have skipped an
    access outside its job's range."""
    yield
    if os.environ.get("DC_LIBRARY") == "bounds" and request.node.get_closest_marker("gpu"):
        import reduce_copy_rank_gb300 as dc

        assert dc.lib().dc_bounds_checked() == 1
        st = dc.dc_check_device()
        assert st != 7, dc.last_error()  # DC_ERR_BOUNDS


@pytest.fixture(scope="session")
def orc():
    """The C oracle (built on first use)."""
    import oracle

    return oracle.default()
