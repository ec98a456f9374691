"""The C-ABI library builds, loads and exports every symbol include/pagedkv.h
declares; host-side validation rejects bad arguments without launching.
No compute call runs here (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_115_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = declared_functions()
    for need in ("pkv_slot_mapping", "pkv_kv_write", "pkv_attention_decode",
                 "pkv_attention_workspace_bytes", "pkv_kv_block_copy", "pkv_get_device_error"):
        assert need in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_binding_wraps_every_symbol():
    from paged_kv_cache_115_gb300 import ops
    assert sorted(ops.EXPORTED) == declared_functions()


def test_status_strings_and_version(lib):
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE_TOO_SMALL"
    assert lib.pkv_status_string(99) == b"PKV_UNKNOWN_STATUS"
    assert lib.pkv_version() >> 16 == 1


def test_host_validation_without_launch(lib):
    vp = ctypes.c_void_p
    lib.pkv_last_error_message.restype = ctypes.c_char_p
    f = lib.pkv_kv_write
    f.argtypes = [vp, vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp]
    # zero tokens: nothing to do
    assert f(None, None, None, 0, None, None, 8, 16, 8, 128, 1, None) == 0
    # null pointers with work to do
    assert f(None, None, None, 4, None, None, 8, 16, 8, 128, 1, None) == 1
    assert b"null" in lib.pkv_last_error_message()
    # bad dtype
    assert f(None, None, None, 4, None, None, 8, 16, 8, 128, 7, None) == 1
    g = lib.pkv_kv_block_copy
    g.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, vp]
    assert g(None, None, None, -1, 8, 16, 8, 128, 1, None) == 1
    sw = lib.pkv_kv_block_swap
    sw.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64, vp,
                   ctypes.c_int64, vp]
    assert sw(None, None, 8, None, None, 4, 32768, None, 0, None) == 0      # nothing to move
    assert sw(None, None, 8, None, None, 4, 32768, None, -1, None) == 1     # negative count
    assert sw(None, None, 8, None, None, 4, 0, None, 1, None) == 1          # empty blocks
    assert sw(None, vp(64), 8, None, None, 4, 32768, None, 1, None) == 1    # V on one side only
    assert b"both" in lib.pkv_last_error_message()
    assert sw(None, None, 8, None, None, 4, 32768, None, 1, None) == 1      # null pools
    assert sw(vp(64), None, 2**62, vp(64), None, 4, 32768, vp(64), 1, None) == 1  # overflow
    h = lib.pkv_slot_mapping
    h.argtypes = [vp, ctypes.c_int32, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, vp, vp]
    assert h(None, 4, None, 0, 16, 10, None, None) == 0
    assert h(None, 0, None, 3, 16, 10, None, None) == 1


def test_attention_plan_validation(lib):
    from paged_kv_cache_115_gb300 import ops
    sz = ctypes.c_size_t(0)
    cfg = ops.AttentionConfig()
    f = lib.pkv_attention_workspace_bytes
    f.argtypes = [ctypes.c_int32] * 7 + [ctypes.POINTER(ops.AttentionConfig),
                                         ctypes.POINTER(ctypes.c_size_t)]
    # H_q not a multiple of H_kv
    assert f(4, 6, 4, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 1
    # CUDA-core plan needs no device: fp32, 4 seqs, 4 heads, D 64, K 4, max len 16
    cfg.kernel = 2
    assert f(4, 4, 2, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 0
    assert sz.value >= 4 * 4 * 64 * 4
    # unsupported head_dim
    assert f(4, 4, 2, 48, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 2
    # reserved fields must be zero
    cfg.reserved[0] = 1
    assert f(4, 4, 2, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 1
    cfg.reserved[0] = 0
    # share_prefix is 0 or 1; the CUDA-core plan ignores it (same workspace)
    cfg.share_prefix = 2
    assert f(4, 4, 2, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 1
    base = ctypes.c_size_t(0)
    cfg.share_prefix = 0
    assert f(4, 4, 2, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(base)) == 0
    cfg.share_prefix = 1
    assert f(4, 4, 2, 64, 4, 16, 0, ctypes.byref(cfg), ctypes.byref(sz)) == 0
    assert sz.value == base.value
