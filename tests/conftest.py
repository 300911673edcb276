import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")


PIN_DIR = os.path.join(ROOT, "tests", "pins")
PIN_LIB = os.path.join(PIN_DIR, "_build", "libcurand_philox_pin.so")


def build_curand_pin():
    """Host-compiled curand Philox4x32-10 (the pin for both Philox implementations)."""
    src = os.path.join(PIN_DIR, "curand_philox_pin.cu")
    if os.path.exists(PIN_LIB) and os.path.getmtime(PIN_LIB) >= os.path.getmtime(src):
        return PIN_LIB
    os.makedirs(os.path.dirname(PIN_LIB), exist_ok=True)
    tmp = PIN_LIB + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, src],
                   check=True, capture_output=True)
    os.replace(tmp, PIN_LIB)
    return PIN_LIB


@pytest.fixture(scope="session")
def curand_pin():
    import ctypes
    import shutil

    if shutil.which("nvcc") is None:
        pytest.skip("nvcc not available to build the curand pin")
    lib = ctypes.CDLL(build_curand_pin())
    lib.pin_curand_philox4x32_10.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    lib.pin_curand_philox4x32_10.restype = None
    return lib
