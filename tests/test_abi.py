"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad input before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import build as native_build
from packed_varlen_attention_aware_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hdpattn.h")


@pytest.fixture(scope="module")
def lib():
    native_build.build()
    return pkg.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(hdp_[a-z_]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("hdp_plan_create", "hdp_attention_fwd", "hdp_lse_merge", "hdp_flops_per_shard"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert set(syms) == set(binding.EXPORTED)
    for name in syms:
        assert hasattr(lib, name), name


def test_python_binding_has_every_symbol():
    for name in declared_symbols():
        assert callable(getattr(pkg, name, None)), name


def test_status_strings(lib):
    assert pkg.hdp_status_string(pkg.HDP_OK) == "HDP_OK"
    assert pkg.hdp_status_string(pkg.HDP_ERR_DEVICE_TIMEOUT) == "HDP_ERR_DEVICE_TIMEOUT"
    assert pkg.hdp_status_string(99) == "HDP_ERR_UNKNOWN"


def test_host_argument_checks(lib):
    V = ctypes.c_void_p
    out = V()
    assert lib.hdp_plan_create(None, 4, 256, None, ctypes.byref(out)) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert "d_lengths" in pkg.hdp_last_error_message()
    assert lib.hdp_plan_create(V(16), 0, 256, None, ctypes.byref(out)) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_plan_create(V(16), 4, 0, None, ctypes.byref(out)) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_plan_create_ex(V(16), 4, 256, 8, None, ctypes.byref(out)) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_plan_create(V(16), 4, 256, None, None) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_plan_view(None, None) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_plan_destroy(None) == pkg.HDP_OK
    args = [None, V(16), V(16), V(16), 32, 8, 128, ctypes.c_float(0.1), 0, None, 0, V(16), V(16), None]
    assert lib.hdp_attention_fwd(*args) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_lse_merge(None, V(16), V(16), 4, 64, V(16), V(16), None) == pkg.HDP_ERR_INVALID_ARGUMENT
    for bad in ((0, 10, 64), (2, -1, 64), (2, 10, 3), (2, 10, 260)):
        assert lib.hdp_lse_merge_rows(*bad, V(16), V(16), V(16), V(16), None) == pkg.HDP_ERR_INVALID_ARGUMENT
    assert lib.hdp_lse_merge_rows(2, 0, 64, None, None, None, None, None) == pkg.HDP_OK
    assert lib.hdp_flops_per_shard(None, 128, 32, V(16), None) == pkg.HDP_ERR_INVALID_ARGUMENT
    n = ctypes.c_size_t()
    assert lib.hdp_attention_workspace_bytes(None, 32, 128, 0, ctypes.byref(n)) == pkg.HDP_ERR_INVALID_ARGUMENT


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        binding._lib_saved = binding._lib
        try:
            binding._lib = None
            binding.load(str(tmp_path / "nope.so"))
        finally:
            binding._lib = binding._lib_saved
