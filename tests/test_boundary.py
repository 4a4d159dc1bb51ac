"""The C-ABI boundary without a GPU: the library builds for sm_103a, loads,
and exports every entry point include/hs.h declares; the binding exposes the
same names; structure layouts match the header."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hs.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = _declared()
    for must in ("hs_pool_create", "hs_resolve", "hs_gather", "hs_sparse_mla_decode",
                 "hs_offload_prefix", "hs_commit_offload", "hs_check_errors"):
        assert must in names


def test_library_exports_every_declared_symbol():
    import sparse_attention_kv_hs_gb300 as hs
    lib = hs.load()
    for name in _declared():
        assert hasattr(lib, name), f"libhs.so does not export {name}"
        assert name in hs.EXPORTED or name == "hs_status_string"
    assert set(hs.EXPORTED) <= set(_declared())


def test_status_strings_and_version_need_no_gpu():
    import sparse_attention_kv_hs_gb300 as hs
    assert hs.status_string(hs.HS_OK) == "HS_OK"
    assert "capacity" in hs.status_string(hs.HS_ERR_CAPACITY).lower()
    assert "sm_103a" in hs.hs_version()


def test_struct_layouts_match_the_header():
    import sparse_attention_kv_hs_gb300 as hs
    # 8 x int32 + 2 x int64
    assert ctypes.sizeof(hs.hs_pool_desc) == 48
    assert hs.hs_pool_desc.host_tokens.offset == 32
    # 12 pointers + 3 x int64
    assert ctypes.sizeof(hs.hs_pool_views) == 12 * 8 + 3 * 8


def test_library_is_built_for_sm103a_only():
    """The build's target is recorded in the library's version string (the
    build script passes a single -gencode for compute_103a / sm_103a)."""
    import sparse_attention_kv_hs_gb300 as hs
    from sparse_attention_kv_hs_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "sm_103a" in hs.hs_version()


def test_null_arguments_are_rejected_without_a_gpu():
    import sparse_attention_kv_hs_gb300 as hs
    lib = hs.load()
    assert lib.hs_pool_create(None, None) == hs.HS_ERR_INVALID
    assert lib.hs_resolve(None, 0, 1, None, None, None, None, None, None) == hs.HS_ERR_INVALID
    assert lib.hs_gather(None, 0, None, 0, None, None) == hs.HS_ERR_INVALID
    assert lib.hs_sparse_mla_decode(None, 0, None, None, 128, 512, 1.0, None, None, None) == \
        hs.HS_ERR_INVALID
    assert lib.hs_check_errors(None, None) == hs.HS_ERR_INVALID
    assert lib.hs_step_advance(None, None) == hs.HS_ERR_INVALID


def test_error_codes_match_the_header():
    """The binding's status and device-error constants are the header's values."""
    import sparse_attention_kv_hs_gb300 as hs
    text = open(HEADER).read()
    defines = {m.group(1): int(m.group(2)) for m in
               re.finditer(r"#define\s+HS_DEV_ERR_([A-Z]+)\s+(\d+)", text)}
    assert defines, "no HS_DEV_ERR_ defines found"
    for name, value in defines.items():
        assert getattr(hs, "DEV_ERR_" + name) == value, name
    enum = {m.group(1): int(m.group(2)) for m in
            re.finditer(r"\bHS_(OK|ERR_[A-Z]+)\s*=\s*(-?\d+)", text)}
    for name, value in enum.items():
        assert getattr(hs, "HS_" + name) == value, name


def test_unpinnable_host_pool_is_out_of_memory_before_any_allocation():
    """A host pool larger than the machine's physical memory returns HS_ERR_OOM
    from the size check, before any CUDA call (so also without a GPU), and
    leaves the output handle NULL."""
    import sparse_attention_kv_hs_gb300 as hs
    lib = hs.load()
    desc = hs.hs_pool_desc(4, 2, 256, 512, 256, 576, 64, 0, 1 << 40, 4)  # 2 x 2^40 x 1152 B
    out = ctypes.c_void_p(12345)
    assert lib.hs_pool_create(ctypes.byref(desc), ctypes.byref(out)) == hs.HS_ERR_OOM
    assert out.value is None


def test_wait_offload_argument_errors_need_no_gpu():
    import sparse_attention_kv_hs_gb300 as hs
    lib = hs.load()
    assert lib.hs_wait_offload(None, 1000) == hs.HS_ERR_INVALID
    assert lib.hs_wait_offload(ctypes.c_void_p(8), -1) == hs.HS_ERR_INVALID
    assert lib.hs_pool_touch_host(None, None) == hs.HS_ERR_INVALID
