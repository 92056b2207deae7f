"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
entry point that include/moe.h declares, and its host-side argument checks
answer before any device call."""
import ctypes
import os
import re
import shutil

import pytest

from quantized_moe_expert_router_gb300 import build, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

pytestmark = pytest.mark.skipif(shutil.which(build.NVCC) is None, reason="nvcc not found")


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status|const\s+char\s*\*)\s*(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.MOE_LIB)


def test_header_declares_the_binding_names():
    assert declared_entry_points() == sorted(moe.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_entry_points() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    seen = set()
    for s in range(9):
        msg = lib.moe_status_string(s)
        assert msg and msg not in seen, (s, msg)
        seen.add(msg)
    assert lib.moe_status_string(1000)  # unknown codes still get a string


def _create(lib, **kw):
    cfg = moe.moe_config(**{**dict(num_experts=896, top_k=16, hidden=3584, intermediate=3072,
                                   max_tokens=8, flags=0), **kw})
    out = ctypes.c_void_p()
    lib.moe_layer_create.argtypes = [ctypes.POINTER(moe.moe_config), ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_layer_create.restype = ctypes.c_int
    return lib.moe_layer_create(ctypes.byref(cfg), 0, ctypes.byref(out)), out


@pytest.mark.parametrize("kw,status", [
    (dict(top_k=0), 2), (dict(top_k=33), 2), (dict(num_experts=4, top_k=8), 2),
    (dict(hidden=100), 2), (dict(hidden=8192), 2), (dict(intermediate=32), 2),
    (dict(max_tokens=0), 1), (dict(flags=1), 1),
])
def test_create_rejects_bad_configs_on_the_host(lib, kw, status):
    got, out = _create(lib, **kw)
    assert got == status and not out.value


def test_null_arguments_are_rejected(lib):
    lib.moe_packed_bytes.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_packed_bytes.restype = ctypes.c_int
    assert lib.moe_packed_bytes(None, None) == 1
    lib.moe_layer_destroy.argtypes = [ctypes.c_void_p]
    lib.moe_layer_destroy.restype = ctypes.c_int
    assert lib.moe_layer_destroy(None) in (0, 1)
