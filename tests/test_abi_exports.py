"""The C-ABI library loads and exports every entry point include/*.h declares (no GPU needed)."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from mla_absorbed_decode_absorb_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_path_calls():
    names = declared_functions()
    for n in ["mla_append_kv", "mla_absorb_q", "mla_decode_attn", "mla_out_absorb"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_entry_points(lib):
    lib.mla_status_string.restype = ctypes.c_char_p
    assert lib.mla_status_string(0) == b"MLA_OK"
    assert b"BOUNDS" in lib.mla_status_string(6)
    assert lib.mla_abi_version() >= 1
    lib.mla_rope_table_bytes.restype = ctypes.c_size_t
    assert lib.mla_rope_table_bytes(100) == 100 * 64 * 4
    # explicit split size: pure host arithmetic, no device query
    n = ctypes.c_int(0)
    assert lib.mla_decode_num_splits(8, 1, 32769, 64, ctypes.byref(n)) == 0
    assert n.value == 9  # 513 pages in 64-page chunks
    sz = ctypes.c_size_t(0)
    assert lib.mla_decode_workspace_size(8, 1, 32769, 64, ctypes.byref(sz)) == 0
    assert sz.value >= 8 * 9 * 128 * (512 + 1) * 4
    assert lib.mla_decode_workspace_size(8, 1, 4096, 64, ctypes.byref(sz)) == 0
    assert sz.value == 0  # a single split needs no workspace


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    lib.mla_append_kv.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                                          ctypes.c_int, ctypes.c_void_p]
    assert lib.mla_append_kv(None, None, None, None, 1, None, 1, None, 1, 1, 1, None) == 1
    assert lib.mla_append_kv(None, None, None, None, 1, None, 1, None, 1, -1, 1, None) == 1
    # n_q outside [1, 8]
    n = ctypes.c_int(0)
    assert lib.mla_decode_num_splits(1, 9, 100, 4, ctypes.byref(n)) == 1
    assert lib.mla_decode_num_splits(1, 2, 1, 4, ctypes.byref(n)) == 1  # max_kv_len < n_q
