import ctypes
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--range-checked", action="store_true", default=False,
                     help="run every test on the range-checked library (-DDCN_DEBUG_BOUNDS) "
                          "instead of the normal one: any access outside its tensor makes the "
                          "call return DCN_ERR_INTERNAL")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def native(request):
    """The CUDA library's binding, with the library built in-tree (the
    range-checked one under --range-checked)."""
    from deformable_convolution_03_b300 import build, binding
    build.build()
    if request.config.getoption("--range-checked"):
        binding.LIB_PATH = build.build(debug_bounds=True)
        binding._lib = None
        L = binding.lib()
        L.dcn_internal_debug_bounds.restype = ctypes.c_int
        assert L.dcn_internal_debug_bounds() == 1
    return binding


class Options:
    """The library's kernel-selection switches (a test hook the library exports
    without declaring it in its public header)."""

    def __init__(self, lib):
        self.lib = lib

    def set(self, name: str, value: int) -> None:
        rc = self.lib.dcn_internal_set_option(name.encode(), int(value))
        assert rc == 0, f"unknown switch {name}"

    def update(self, switches: dict) -> None:
        for k, v in switches.items():
            self.set(k, v)


@pytest.fixture
def opts(native):
    """Switches set by a test, all put back to their defaults afterwards."""
    L = native.lib()
    L.dcn_internal_set_option.argtypes = [ctypes.c_char_p, ctypes.c_int]
    L.dcn_internal_set_option.restype = ctypes.c_int
    L.dcn_internal_reset_options.argtypes = []
    L.dcn_internal_reset_options.restype = None
    L.dcn_internal_reset_options()
    yield Options(L)
    L.dcn_internal_reset_options()
