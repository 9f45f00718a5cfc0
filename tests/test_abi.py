"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/moe.h declares (no GPU needed; nothing is computed)."""
import ctypes
import os
import re

import quantized_moe_expert_layer_gb300 as moe


def _declared():
    src = open(moe.HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:int|void|const char\*)\s+(moe_\w+)\s*\(", src, flags=re.M))


def test_header_declares_the_binding_exports():
    assert _declared() == set(moe.EXPORTS)


def test_library_builds_and_exports_all_symbols():
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    path = moe.build()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(lib, name), name
    moe.lib()


def test_errors_without_a_layer_are_reported():
    lib = moe.lib()
    out = ctypes.c_void_p(123)
    rc = lib.moe_layer_create(7, 256, 128, 8, 2, 0, ctypes.byref(out))
    assert rc == moe.EINVAL and out.value is None
    assert b"format" in lib.moe_last_error()
    rc = lib.moe_layer_create(1, 250, 128, 8, 2, 0, ctypes.byref(out))
    assert rc == moe.EINVAL and b"multiples" in lib.moe_last_error()
    rc = lib.moe_layer_create(1, 256, 128, 8, 9, 0, ctypes.byref(out))
    assert rc == moe.EINVAL
    rc = lib.moe_layer_create(1, 65536 + 64, 128, 8, 2, 0, ctypes.byref(out))
    assert rc == moe.EINVAL and b"at most" in lib.moe_last_error()
    assert lib.moe_forward(None, None, 1, None, None) == moe.EINVAL
    assert lib.moe_place_experts(None, None) == moe.EINVAL
    assert lib.moe_layer_placement(None, None, None, None) == moe.EINVAL
    assert lib.moe_layer_reserve(None, 4) == moe.EINVAL
