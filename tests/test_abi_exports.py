"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlora_nf4.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qlora_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def libpath():
    from bit_quantized_fine_nf4_b300 import build_lib
    return build_lib.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("qlora_nf4_quantize", "qlora_nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd"):
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (qlora_[a-z0-9_]+)", out))
    assert set(_declared()) <= exported


def test_binding_lists_every_declared_symbol():
    from bit_quantized_fine_nf4_b300 import EXPORTS
    assert sorted(EXPORTS) == _declared()


def test_strerror_and_no_device_paths(libpath):
    """Host-only calls work without a GPU; device calls fail cleanly instead of crashing."""
    lib = ctypes.CDLL(libpath)
    lib.qlora_strerror.restype = ctypes.c_char_p
    assert lib.qlora_strerror(0) == b"ok"
    assert lib.qlora_strerror(4) == b"bounded device wait expired"
    b = ctypes.c_size_t(0)
    assert lib.qlora_nf4_quantize_workspace_bytes(ctypes.c_int64(256), ctypes.c_int64(256), ctypes.byref(b)) == 0
    assert b.value >= 256 * 256 // 64 * 4
    assert lib.qlora_nf4_quantize_workspace_bytes(ctypes.c_int64(256), ctypes.c_int64(100), ctypes.byref(b)) == 1
    import torch
    if not torch.cuda.is_available():
        lib.qlora_device_sm_count.restype = ctypes.c_int
        assert lib.qlora_device_sm_count() == 0

