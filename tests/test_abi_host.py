"""C ABI checks that need no GPU: the library builds, loads, exports every symbol that the
header declares, and rejects bad arguments before it touches the CUDA runtime."""
import ctypes
import os
import re

import pytest

import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import build

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4_gemv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return nv.library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("nvfp4_gemv", "nvfp4_gemv_gate_up", "nvfp4_gemv_gate_up_swiglu", "nvfp4_moe_gemv"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a():
    cmd = build.nvcc_command()
    assert "-gencode=arch=compute_103a,code=sm_103a" in cmd
    assert os.path.exists(build.LIB_PATH)


def test_version_and_status_strings(lib):
    assert lib.nvfp4_version() >= 100
    for code in range(8):
        assert len(nv.status_string(code)) > 0
    assert nv.status_string(99) == "unknown status"


P = ctypes.c_void_p
FAKE = P(4096)  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 32, None), 1),     # null weights
    ((FAKE, FAKE, 1.0, None, FAKE, 0, 1, 16, 32, None), 1),     # null x
    ((FAKE, FAKE, 1.0, FAKE, None, 0, 1, 16, 32, None), 1),     # null y
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, 9, 16, 32, None), 2),     # M > 8
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, -1, 16, 32, None), 2),    # negative M
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, 1, -5, 32, None), 2),     # negative N
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 24, None), 2),     # K % 16 != 0
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 2, 1, 16, 32, None), 4),     # bad output type
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, 0, 16, 32, None), 0),     # M == 0: nothing to do
    ((FAKE, FAKE, 1.0, FAKE, FAKE, 0, 3, 0, 32, None), 0),      # N == 0: nothing to do
])
def test_dense_validation(lib, args, expect):
    assert lib.nvfp4_gemv(*args) == expect


def test_gate_up_validation(lib):
    f = lib.nvfp4_gemv_gate_up
    assert f(FAKE, FAKE, 1.0, None, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 32, None) == 1
    assert f(FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 33, None) == 2
    assert f(FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, FAKE, 1, 0, 16, 32, None) == 0


def test_gate_up_swiglu_validation(lib):
    f = lib.nvfp4_gemv_gate_up_swiglu
    inf = float("inf")
    ok = [FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, inf, FAKE, 0, 1, 16, 32, None]
    bad = list(ok); bad[3] = None                     # null up weights
    assert f(*bad) == 1
    bad = list(ok); bad[8] = None                     # null y
    assert f(*bad) == 1
    for lim in (0.0, -1.0, float("nan")):             # the clamp limit must be > 0
        bad = list(ok); bad[7] = lim
        assert f(*bad) == 2
    bad = list(ok); bad[12] = 40                      # K % 16 != 0
    assert f(*bad) == 2
    bad = list(ok); bad[10] = 9                       # M > 8
    assert f(*bad) == 2
    bad = list(ok); bad[9] = 3                        # bad output type
    assert f(*bad) == 4
    empty = list(ok); empty[10] = 0                   # M == 0: nothing to do
    assert f(*empty) == 0


def test_moe_validation(lib):
    f = lib.nvfp4_moe_gemv
    ok = [FAKE, FAKE, FAKE, 8, FAKE, 2, 4, FAKE, 0, FAKE, 0, 64, 32, None, None]
    bad = list(ok); bad[4] = None                     # null ids
    assert f(*bad) == 1
    bad = list(ok); bad[3] = 0                        # E == 0
    assert f(*bad) == 2
    bad = list(ok); bad[12] = 40                      # K % 16 != 0
    assert f(*bad) == 2
    bad = list(ok); bad[10] = 7                       # bad output type
    assert f(*bad) == 4
    empty = list(ok); empty[5] = 0                    # T == 0: nothing to do
    assert f(*empty) == 0
