"""The C ABI library builds, loads and exports every function include/*.h
declares; host-only argument checks answer without touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

import adapter_linear_gb300 as al
from adapter_linear_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if cuda_build.needs_build():
        cuda_build.build()
    return al.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*[\s\*]+([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_binding_exports():
    names = declared_functions()
    assert names == set(al.EXPORTS), names ^ set(al.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.lora_abi_version() == 1


def test_checked_build_exports_every_declared_symbol(lib):
    """The range-checked build (LORA_CHECK) has the same ABI."""
    path = os.path.join(os.path.dirname(al.__file__), "liblora_linear_check.so")
    if not os.path.exists(path):
        from adapter_linear_gb300 import build as cuda_build
        cuda_build.build(check=True)
    checked = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(checked, name), name
    checked.lora_status_string.restype = ctypes.c_char_p
    assert checked.lora_status_string(13) == b"a checked kernel met an index out of range"


def test_status_strings(lib):
    for code in range(0, 14):
        s = al.lora_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert al.lora_status_string(99) == "unknown status"


def test_null_handles_are_rejected_on_the_host(lib):
    assert lib.lora_pool_destroy(None) == al.LORA_ERR_ARG
    assert lib.lora_pool_reserve(None, 4) == al.LORA_ERR_ARG
    assert lib.lora_unload_adapter(None, 0) == al.LORA_ERR_ARG
    assert lib.lora_load_adapter(None, 0, None, None, 8, 16.0) == al.LORA_ERR_ARG
    assert lib.lora_linear(None, None, None, None, 4, None, None) == al.LORA_ERR_ARG
    assert lib.lora_base_linear(None, None, None, 4, None, None) == al.LORA_ERR_ARG
    assert lib.lora_linear_host(None, None, None, None, 4, None, None) == al.LORA_ERR_ARG
    assert lib.lora_pool_check_errors(None) == al.LORA_ERR_ARG
    assert lib.lora_pool_set_prefill_kernel(None, al.LORA_PREFILL_PAIR) == al.LORA_ERR_ARG
    assert lib.lora_test_delayed_copy(None, None, 4, 10, None) == al.LORA_ERR_ARG
    assert lib.lora_pool_set_path(None, 0) == al.LORA_ERR_ARG
    assert lib.lora_pool_stats(None, None) == al.LORA_ERR_ARG
    out = ctypes.c_void_p()
    assert lib.lora_pool_create(0, 16, 256, 256, ctypes.byref(out)) == al.LORA_ERR_ARG
    assert lib.lora_pool_create(4, 0, 256, 256, ctypes.byref(out)) == al.LORA_ERR_RANK
    assert lib.lora_pool_create(4, 257, 256, 256, ctypes.byref(out)) == al.LORA_ERR_RANK
    assert lib.lora_pool_create(4, 16, 250, 256, ctypes.byref(out)) == al.LORA_ERR_SHAPE
    assert lib.lora_pool_create(4, 16, 256, 0, ctypes.byref(out)) == al.LORA_ERR_SHAPE
    assert lib.lora_pool_create(4, 16, 256, 256, None) == al.LORA_ERR_ARG


def test_product_path_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(al.LibraryMissing):
        # a fresh loader pointed at a missing file: no fallback is attempted
        al._lib, saved = None, al._lib
        try:
            al.load_library(str(tmp_path / "missing.so"))
        finally:
            al._lib = saved


def test_no_oracle_on_the_product_path():
    pkg = os.path.join(ROOT, "adapter_linear_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path, encoding="utf-8").read()
            assert "import oracle" not in text and "oracle." not in text, path
            assert "lora_oracle" not in text, path
