"""The checked build (CCL_BOUNDS_CHECK) compiles and links on the CPU, and
each library reports which build it is (ccl_bounds_checked) -- so that a
source change that breaks only the checked build fails here, not on the GPU.
No kernel runs."""
import ctypes

import pytest

import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import build as ccl_build

pytestmark = pytest.mark.cpu


def test_checked_and_default_builds_report_themselves():
    checked = ccl_build.build_checked()
    default = ccl_build.build()
    assert ctypes.CDLL(checked).ccl_bounds_checked() == 1
    assert ctypes.CDLL(default).ccl_bounds_checked() == 0
    # every symbol the header declares is exported by the checked library too
    lib = ctypes.CDLL(checked)
    for name in ccl.EXPORTS:
        assert hasattr(lib, name), name
