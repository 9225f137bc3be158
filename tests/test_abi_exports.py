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
    assert sz.value >= 8 * 9 * 128 * (512 * 2 + 4)  # bf16 partial rows + float32 log-sum-exps
    assert lib.mla_decode_workspace_size(8, 1, 4096, 64, ctypes.byref(sz)) == 0
    assert sz.value == 0  # a single split needs no workspace


def test_short_context_plan(lib):
    """With an automatic split, at most two (sequence, query) units over at most 1024
    cached tokens take the short-context kernel with a single split; an explicit split,
    more units or a longer context keep the tensor-core split kernel.  The cases
    below need no device query."""
    flag, n = ctypes.c_int(-1), ctypes.c_int(0)
    for B, n_q, kv, sp, short in [(1, 1, 257, 0, 1), (2, 1, 1024, 0, 1), (1, 2, 1024, 0, 1), (1, 1, 1, 0, 1),
                                  (1, 1, 257, 1, 0), (1, 1, 257, 1000, 0), (1, 1, 1025, 64, 0), (3, 1, 100, 4, 0)]:
        assert lib.mla_decode_uses_short_path(B, n_q, kv, sp, ctypes.byref(flag)) == 0
        assert flag.value == short, (B, n_q, kv, sp)
        if short:
            assert lib.mla_decode_num_splits(B, n_q, kv, sp, ctypes.byref(n)) == 0 and n.value == 1
    assert lib.mla_decode_uses_short_path(1, 1, 100, 0, None) == 1


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


def test_new_entry_points_validate_before_any_launch(lib):
    """Argument checks of the fused prologue, the pair projection, the host-link copy and the
    timeout self-test, all of which return before touching the device."""
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.mla_append_absorb_q.argtypes = [P, P, P, P, P, P, I, P, P, I, P, I64, P, I, I, P]
    # n_q = 0 and n_q = 9 are outside [1, MLA_MAX_NQ]; null pointers with B > 0
    assert lib.mla_append_absorb_q(*([None] * 6), 1, None, None, 1, None, 1, None, 1, 0, None) == 1
    assert lib.mla_append_absorb_q(*([None] * 6), 1, None, None, 1, None, 1, None, 1, 9, None) == 1
    assert lib.mla_append_absorb_q(*([None] * 6), 1, None, None, 1, None, 1, None, 1, 1, None) == 1
    assert lib.mla_append_absorb_q(*([None] * 6), 1, None, None, 1, None, 1, None, 0, 1, None) == 0  # B = 0
    lib.mla_linear_pair_workspace_size.argtypes = [I, I, I, I, ctypes.POINTER(SZ)]
    sz = SZ(0)
    assert lib.mla_linear_pair_workspace_size(32, 100, 512, 64, ctypes.byref(sz)) == 1  # K % 64
    assert lib.mla_linear_pair_workspace_size(0, 128, 512, 64, ctypes.byref(sz)) == 1   # T < 1
    assert lib.mla_linear_pair_workspace_size(32, 128, 512, 0, ctypes.byref(sz)) == 1   # N1 < 1
    lib.mla_linear_pair.argtypes = [P, I, I, P, I, P, P, I, P, P, SZ, P]
    assert lib.mla_linear_pair(None, 32, 128, None, 512, None, None, 64, None, None, 0, None) == 1
    lib.mla_copy_async.argtypes = [P, P, SZ, P]
    assert lib.mla_copy_async(None, None, 0, None) == 0   # nothing to copy
    assert lib.mla_copy_async(None, None, 16, None) == 1
    lib.mla_selftest_wait_timeout.argtypes = [I64, P]
    assert lib.mla_selftest_wait_timeout(0, None) == 1
    assert lib.mla_selftest_wait_timeout(3_000_000_000, None) == 1


def test_merge_refuses_a_short_or_misaligned_workspace(lib):
    """The merge entry point validates the workspace on the host before it launches
    anything: a workspace smaller than the plan or not 16-byte aligned returns
    MLA_ERR_WORKSPACE (the pointers below are never dereferenced)."""
    B, n_q, kv, sp = 2, 1, 1000, 4  # 16 pages in 4 splits
    n = ctypes.c_int(0)
    assert lib.mla_decode_num_splits(B, n_q, kv, sp, ctypes.byref(n)) == 0 and n.value == 4
    sz = ctypes.c_size_t(0)
    assert lib.mla_decode_workspace_size(B, n_q, kv, sp, ctypes.byref(sz)) == 0 and sz.value > 0
    f = lib.mla_decode_combine
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_size_t] + [ctypes.c_void_p] * 3
    o_latent = ctypes.c_void_p(0x20000)
    assert f(B, n_q, kv, sp, ctypes.c_void_p(0x10008), sz.value, o_latent, None, None) == 3  # misaligned
    assert f(B, n_q, kv, sp, ctypes.c_void_p(0x10000), sz.value - 256, o_latent, None, None) == 3  # short
    assert f(B, n_q, kv, sp, None, sz.value, o_latent, None, None) == 3  # missing
