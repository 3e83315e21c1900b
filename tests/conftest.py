import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def pin_lib():
    """The independent E4M3 nearest-value checker (tests/pins), built with gcc."""
    import ctypes
    src = os.path.join(ROOT, "tests", "pins", "e4m3_nearest.c")
    out = os.path.join(tempfile.mkdtemp(prefix="fp8pin"), "libpin.so")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           src, "-o", out, "-lm"])
    L = ctypes.CDLL(out)
    L.check_chunk.restype = ctypes.c_int64
    L.check_chunk.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                              ctypes.POINTER(ctypes.c_int64)]
    L.table_value.restype = ctypes.c_double
    L.table_value.argtypes = [ctypes.c_int]
    return L
