"""The C ABI: the library loads and exports every function include/ikbo.h
declares (no GPU needed, no compute calls)."""
import ctypes
import os
import re

import pytest

from broadcast_gemm_attention_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ikbo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ikbo_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ikbo_plan_create", "ikbo_plan", "ikbo_lce_forward", "ikbo_attn_forward",
                     "ikbo_plan_get_status", "ikbo_plan_destroy", "ikbo_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert set(binding.SIGNATURES) == set(declared_functions())
    for name in declared_functions():
        assert hasattr(binding, name), name


def test_status_strings_and_version_need_no_gpu(lib):
    binding.load(build.LIB)
    assert binding.ikbo_version() == 106
    assert binding.ikbo_status_string(0) == "ok"
    assert "range" in binding.ikbo_status_string(4)
    assert binding.ikbo_status_string(99) == "unknown status"


def test_null_arguments_are_rejected_before_any_cuda_call(lib):
    binding.load(build.LIB)
    L = binding.load()
    assert L.ikbo_plan_create(None, 1, 1, 1) == binding.IKBO_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.ikbo_plan_create(ctypes.byref(h), 0, 1, 1) == binding.IKBO_ERR_INVALID_ARG
    assert h.value is None
    assert L.ikbo_plan(None, None, 1, 1, 1, 8, None) == binding.IKBO_ERR_INVALID_ARG
    assert L.ikbo_lce_forward(None, None, None, None, None, None, None, 1, 1, 8, 8, None) == \
        binding.IKBO_ERR_INVALID_ARG
    assert L.ikbo_attn_forward(None, None, None, None, None, None, 1, 128, 1.0, None) == \
        binding.IKBO_ERR_INVALID_ARG
    L.ikbo_plan_destroy(None)


def test_product_fails_loudly_without_the_library(tmp_path):
    import importlib
    b2 = importlib.reload(binding)
    try:
        b2._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            b2.load(str(tmp_path / "missing.so"))
    finally:
        importlib.reload(binding)
