"""Thin Python binding over ``libmla_decode.so`` (the C ABI of include/mla_decode.h).

Argument marshalling only: every function checks dtypes, devices and
contiguity, passes raw device pointers and the current CUDA stream to the
C entry point of the same name, and raises :class:`MLAError` on a non-OK
status.  Outputs not supplied by the caller are allocated with torch (the
library itself never allocates).  There is no fallback: if the library has
not been built, importing this module raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .workloads import D_LATENT, D_NOPE, D_ROPE, D_ROW, N_HEADS

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m mla_absorbed_decode_absorb_gb300.build` "
        "(or __graft_entry__.build()); there is no non-CUDA fallback")

lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

_SIGS = {
    "mla_abi_version": ([], _i),
    "mla_status_string": ([_i], ctypes.c_char_p),
    "mla_rope_table_bytes": ([_i], _sz),
    "mla_rope_table_init": ([_p, _i, _p], _i),
    "mla_append_kv": ([_p, _p, _p, _p, _i, _p, _i, _p, _i64, _i, _i, _p], _i),
    "mla_absorb_q": ([_p, _p, _p, _p, _p, _i, _p, _i, _i, _p], _i),
    "mla_append_absorb_q": ([_p, _p, _p, _p, _p, _p, _i, _p, _p, _i, _p, _i64, _p, _i, _i, _p], _i),
    "mla_copy_async": ([_p, _p, _sz, _p], _i),
    "mla_selftest_wait_timeout": ([_i64, _p], _i),
    "mla_append_absorb_q_fp8": ([_p, _p, _p, _p, _p, _p, _i, _p, _p, _i, _p, _p, _p, _i64, _p, _i, _i, _p], _i),
    "mla_decode_workspace_size": ([_i, _i, _i, _i, ctypes.POINTER(_sz)], _i),
    "mla_decode_num_splits": ([_i, _i, _i, _i, ctypes.POINTER(_i)], _i),
    "mla_decode_uses_short_path": ([_i, _i, _i, _i, ctypes.POINTER(_i)], _i),
    "mla_decode_attn": ([_p, _p, _i64, _p, _i, _p, _i, _i, _i, _i, _p, _sz, _p, _p, _p], _i),
    "mla_decode_attn_partial": ([_p, _p, _i64, _p, _i, _p, _i, _i, _i, _i, _p, _sz, _p, _p, _p], _i),
    "mla_decode_combine": ([_i, _i, _i, _i, _p, _sz, _p, _p, _p], _i),
    "mla_out_absorb": ([_p, _p, _p, _i, _i, _p], _i),
    "mla_combine_out_absorb": ([_i, _i, _i, _i, _p, _sz, _p, _p, _p, _p, _p], _i),
    "mla_get_device_status": ([_p], _i),
    "mla_set_launch_overlap": ([_i], _i),
    "mla_decompress_kv": ([_p, _i64, _p, _i, _p, _i, _i, _p, _p, _p, _p, _p], _i),
    "mla_prefill_attn": ([_p, _p, _p, _p, _i, _p, _p, _i, _p, _i64, _p, _i, _p, _i, _i, _p, _p, _p], _i),
    "mla_get_launch_overlap": ([], _i),
    "mla_linear_workspace_size": ([_i, _i, _i, ctypes.POINTER(_sz)], _i),
    "mla_linear": ([_p, _p, _p, _i, _i, _i, _p, _sz, _p], _i),
    "mla_linear_pair_workspace_size": ([_i, _i, _i, _i, ctypes.POINTER(_sz)], _i),
    "mla_linear_pair": ([_p, _i, _i, _p, _i, _p, _p, _i, _p, _p, _sz, _p], _i),
    "mla_linear_strided": ([_p, _p, _p, _i, _i, _i, _i64, _i, _i, _p, _sz, _p], _i),
    "mla_rope_q": ([_p, _p, _p, _i, _p, _i, _i, _p], _i),
    "mla_f32_to_bf16": ([_p, _p, _i64, _p], _i),
    "mla_append_kv_fp8": ([_p, _p, _p, _p, _i, _p, _i, _p, _p, _p, _i64, _i, _i, _p], _i),
    "mla_decode_attn_fp8_partial": ([_p, _p, _p, _p, _i64, _p, _i, _p, _i, _i, _i, _i, _p, _sz, _p, _p, _p], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, \
    MLA_ERR_BOUNDS, MLA_ERR_RANGE = range(8)
MLA_MAX_NQ = 8  # new tokens per sequence the absorbed kernels take (MLA_MAX_NQ of the C header)


class MLAError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {mla_status_string(status)}")
        self.status = status


def mla_status_string(status: int) -> str:
    return lib.mla_status_string(int(status)).decode()


def _check(where: str, status: int) -> None:
    if status != MLA_OK:
        raise MLAError(where, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_or_pinned(t: torch.Tensor, name: str, dtype, shape=None) -> int:
    """An output the kernels may store to across the host link: a CUDA tensor, or a
    pinned (page-locked) host tensor."""
    if isinstance(t, torch.Tensor) and t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name} is pageable host memory: pin it (tensor.pin_memory())")
        if t.dtype != dtype or not t.is_contiguous() or (shape is not None and tuple(t.shape) != tuple(shape)):
            raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape}")
        return t.data_ptr()
    return _dev(t, name, dtype, shape)


def _dev(t: torch.Tensor, name: str, dtype, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def mla_abi_version() -> int:
    return lib.mla_abi_version()


def rope_table(max_positions: int, device=None, stream=None) -> torch.Tensor:
    """[max_positions, 64] float32: cos then sin of the 32 RoPE frequencies (mla_rope_table_init)."""
    t = torch.empty(max_positions, D_ROPE, dtype=torch.float32, device=device or "cuda")
    _check("mla_rope_table_init", lib.mla_rope_table_init(t.data_ptr(), int(max_positions), _stream(stream)))
    return t


def mla_append_kv(c_kv_new, k_pe_new, seq_lens_before, page_table, rope, cache, stream=None):
    B, n_new = c_kv_new.shape[:2]
    args = (
        _dev(c_kv_new, "c_kv_new", torch.bfloat16, (B, n_new, D_LATENT)),
        _dev(k_pe_new, "k_pe_new", torch.bfloat16, (B, n_new, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(page_table, "page_table", torch.int32),
        int(page_table.shape[1]),
        _dev(rope, "rope_table", torch.float32),
        int(rope.shape[0]),
        _dev(cache, "cache", torch.bfloat16),
        int(cache.shape[0]),
        int(B), int(n_new), _stream(stream))
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages]")
    if tuple(cache.shape[1:]) != (64, D_ROW):
        raise ValueError("cache must be [num_pages, 64, 576]")
    _check("mla_append_kv", lib.mla_append_kv(*args))
    return cache


MLA_LINEAR_MAX_T = 256


def mla_linear_workspace_size(T, K, N) -> int:
    n = _sz(0)
    _check("mla_linear_workspace_size", lib.mla_linear_workspace_size(int(T), int(K), int(N), ctypes.byref(n)))
    return int(n.value)


def alloc_linear_workspace(T, K, N, device):
    n = mla_linear_workspace_size(T, K, N)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def mla_linear_pair_workspace_size(T: int, K: int, N0: int, N1: int) -> int:
    out = _sz(0)
    _check("mla_linear_pair_workspace_size",
           lib.mla_linear_pair_workspace_size(int(T), int(K), int(N0), int(N1), ctypes.byref(out)))
    return int(out.value)


def mla_linear_pair(x, w0, w1, y0=None, y1=None, workspace=None, stream=None):
    """``y0 = x w0^T`` and ``y1 = x w1^T`` in one launch."""
    T, K = x.shape
    N0, N1 = w0.shape[0], w1.shape[0]
    if y0 is None:
        y0 = torch.empty(T, N0, dtype=torch.bfloat16, device=x.device)
    if y1 is None:
        y1 = torch.empty(T, N1, dtype=torch.bfloat16, device=x.device)
    need = mla_linear_pair_workspace_size(T, K, N0, N1)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check("mla_linear_pair", lib.mla_linear_pair(
        _dev(x, "x", torch.bfloat16, (T, K)), int(T), int(K),
        _dev(w0, "w0", torch.bfloat16, (N0, K)), int(N0), _dev(y0, "y0", torch.bfloat16, (T, N0)),
        _dev(w1, "w1", torch.bfloat16, (N1, K)), int(N1), _dev(y1, "y1", torch.bfloat16, (T, N1)),
        0 if not need else _dev(workspace, "workspace", torch.uint8), 0 if not need else workspace.numel(),
        _stream(stream)))
    return y0, y1


def mla_linear(x, w, y=None, workspace=None, stream=None):
    """``y [T, N] = x [T, K] w [N, K]^T`` in bf16 (fp32 accumulation)."""
    T, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    need = mla_linear_workspace_size(T, K, N)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check("mla_linear", lib.mla_linear(
        _dev(x, "x", torch.bfloat16, (T, K)), _dev(w, "w", torch.bfloat16, (N, K)),
        _dev(y, "y", torch.bfloat16, (T, N)), int(T), int(K), int(N),
        0 if not need else _dev(workspace, "workspace", torch.uint8), 0 if not need else workspace.numel(),
        _stream(stream)))
    return y


def mla_linear_strided(x, w, y, y_ld, seg, seg_ld, workspace=None, stream=None):
    """``mla_linear`` writing element (t, n) to ``y.flatten()[t*y_ld + (n//seg)*seg_ld + n%seg]``."""
    T, K = x.shape
    N = w.shape[0]
    need = mla_linear_workspace_size(T, K, N)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if y.dtype != torch.bfloat16 or not y.is_cuda:
        raise TypeError("y must be a CUDA bf16 tensor")
    extent = y.untyped_storage().nbytes() // y.element_size() - y.storage_offset()
    if (T - 1) * y_ld + (N // seg - 1) * seg_ld + seg > extent:
        raise ValueError("y's storage is too small for the strided output")
    _check("mla_linear_strided", lib.mla_linear_strided(
        _dev(x, "x", torch.bfloat16, (T, K)), _dev(w, "w", torch.bfloat16, (N, K)), y.data_ptr(),
        int(T), int(K), int(N), int(y_ld), int(seg), int(seg_ld),
        0 if not need else _dev(workspace, "workspace", torch.uint8), 0 if not need else workspace.numel(),
        _stream(stream)))
    return y


def mla_rope_q(q_rope, seq_lens_before, rope, q_abs, stream=None):
    B, n_q = q_rope.shape[:2]
    _check("mla_rope_q", lib.mla_rope_q(
        _dev(q_rope, "q_rope", torch.bfloat16, (B, n_q, N_HEADS, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)), int(B), int(n_q), _stream(stream)))
    return q_abs


def mla_f32_to_bf16(src, dst, stream=None):
    if src.numel() != dst.numel():
        raise ValueError("src and dst sizes differ")
    _check("mla_f32_to_bf16", lib.mla_f32_to_bf16(
        _dev(src, "src", torch.float32), _dev(dst, "dst", torch.bfloat16), int(src.numel()), _stream(stream)))
    return dst


def fp8_cache_empty(num_pages, device, fill_code=0x7F):
    """An FP8 latent cache: (E4M3 codes [P, 64, 512] uint8, scales [P, 64] f32, keys [P, 64, 64] f16).

    Unwritten slots hold ``fill_code`` (0x7F is E4M3 NaN), NaN scales and NaN keys.
    """
    c8 = torch.full((num_pages, 64, D_LATENT), fill_code, dtype=torch.uint8, device=device)
    scale = torch.full((num_pages, 64), float("nan"), dtype=torch.float32, device=device)
    kr = torch.full((num_pages, 64, D_ROPE), float("nan"), dtype=torch.float16, device=device)
    return c8, scale, kr


def mla_append_kv_fp8(c_kv_new, k_pe_new, seq_lens_before, page_table, rope, cache_fp8, stream=None):
    c8, scale, kr = cache_fp8
    B, n_new = c_kv_new.shape[:2]
    P = int(c8.shape[0])
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages]")
    _check("mla_append_kv_fp8", lib.mla_append_kv_fp8(
        _dev(c_kv_new, "c_kv_new", torch.bfloat16, (B, n_new, D_LATENT)),
        _dev(k_pe_new, "k_pe_new", torch.bfloat16, (B, n_new, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(c8, "cache_c8", torch.uint8, (P, 64, D_LATENT)),
        _dev(scale, "cache_scale", torch.float32, (P, 64)),
        _dev(kr, "cache_kr", torch.float16, (P, 64, D_ROPE)),
        P, int(B), int(n_new), _stream(stream)))
    return cache_fp8


def mla_decode_attn_fp8_partial(q_abs, cache_fp8, page_table, kv_lens, n_q, max_kv_len, split_pages, workspace,
                                o_latent, lse=None, stream=None):
    c8, scale, kr = cache_fp8
    B = kv_lens.shape[0]
    P = int(c8.shape[0])
    _check("mla_decode_attn_fp8_partial", lib.mla_decode_attn_fp8_partial(
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)),
        _dev(c8, "cache_c8", torch.uint8, (P, 64, D_LATENT)),
        _dev(scale, "cache_scale", torch.float32, (P, 64)),
        _dev(kr, "cache_kr", torch.float16, (P, 64, D_ROPE)),
        P, _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(kv_lens, "kv_lens", torch.int32, (B,)),
        int(B), int(n_q), int(max_kv_len), int(split_pages),
        0 if workspace is None else _dev(workspace, "workspace", torch.uint8),
        0 if workspace is None else workspace.numel(),
        _dev(o_latent, "o_latent", torch.float32, (B, n_q, N_HEADS, D_LATENT)),
        0 if lse is None else _dev(lse, "lse", torch.float32, (B, n_q, N_HEADS)),
        _stream(stream)))


def mla_absorb_q(q_nope, q_rope, seq_lens_before, w_uk, rope, q_abs=None, stream=None):
    B, n_q = q_nope.shape[:2]
    if q_abs is None:
        q_abs = torch.empty(B, n_q, N_HEADS, D_ROW, dtype=torch.bfloat16, device=q_nope.device)
    _check("mla_absorb_q", lib.mla_absorb_q(
        _dev(q_nope, "q_nope", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        _dev(q_rope, "q_rope", torch.bfloat16, (B, n_q, N_HEADS, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(w_uk, "w_uk", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)),
        int(B), int(n_q), _stream(stream)))
    return q_abs


def mla_append_absorb_q(c_kv_new, k_pe_new, q_nope, q_rope, seq_lens_before, page_table, w_uk, rope, cache,
                        q_abs, stream=None):
    """mla_append_kv and mla_absorb_q in one launch (n_new = n_q)."""
    B, n_q = q_nope.shape[:2]
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages]")
    if tuple(cache.shape[1:]) != (64, D_ROW):
        raise ValueError("cache must be [num_pages, 64, 576]")
    _check("mla_append_absorb_q", lib.mla_append_absorb_q(
        _dev(c_kv_new, "c_kv_new", torch.bfloat16, (B, n_q, D_LATENT)),
        _dev(k_pe_new, "k_pe_new", torch.bfloat16, (B, n_q, D_ROPE)),
        _dev(q_nope, "q_nope", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        _dev(q_rope, "q_rope", torch.bfloat16, (B, n_q, N_HEADS, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(w_uk, "w_uk", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(cache, "cache", torch.bfloat16), int(cache.shape[0]),
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)),
        int(B), int(n_q), _stream(stream)))
    return cache, q_abs


def mla_append_absorb_q_fp8(c_kv_new, k_pe_new, q_nope, q_rope, seq_lens_before, page_table, w_uk, rope,
                            cache_fp8, q_abs, stream=None):
    """mla_append_kv_fp8 and mla_absorb_q in one launch (n_new = n_q)."""
    B, n_q = q_nope.shape[:2]
    c8, scale, kr = cache_fp8
    P = int(c8.shape[0])
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages]")
    _check("mla_append_absorb_q_fp8", lib.mla_append_absorb_q_fp8(
        _dev(c_kv_new, "c_kv_new", torch.bfloat16, (B, n_q, D_LATENT)),
        _dev(k_pe_new, "k_pe_new", torch.bfloat16, (B, n_q, D_ROPE)),
        _dev(q_nope, "q_nope", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        _dev(q_rope, "q_rope", torch.bfloat16, (B, n_q, N_HEADS, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(w_uk, "w_uk", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(c8, "cache_c8", torch.uint8, (P, 64, D_LATENT)),
        _dev(scale, "cache_scale", torch.float32, (P, 64)),
        _dev(kr, "cache_kr", torch.float16, (P, 64, D_ROPE)),
        P,
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)),
        int(B), int(n_q), _stream(stream)))
    return cache_fp8, q_abs


def mla_copy(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """dst <- src (same number of bytes, both contiguous) with mla_copy_async: device
    tensors of the current device or pinned (page-locked) host tensors."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type == "cpu" and not t.is_pinned():
            raise ValueError(f"{name} is pageable host memory: pin it (tensor.pin_memory())")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise ValueError("dst and src differ in size")
    _check("mla_copy_async", lib.mla_copy_async(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)))
    return dst


def mla_decode_workspace_size(B: int, n_q: int, max_kv_len: int, split_pages: int = 0) -> int:
    out = _sz(0)
    _check("mla_decode_workspace_size",
           lib.mla_decode_workspace_size(int(B), int(n_q), int(max_kv_len), int(split_pages), ctypes.byref(out)))
    return int(out.value)


def mla_decode_num_splits(B: int, n_q: int, max_kv_len: int, split_pages: int = 0) -> int:
    out = _i(0)
    _check("mla_decode_num_splits",
           lib.mla_decode_num_splits(int(B), int(n_q), int(max_kv_len), int(split_pages), ctypes.byref(out)))
    return int(out.value)


def mla_decode_uses_short_path(B: int, n_q: int, max_kv_len: int, split_pages: int = 0) -> bool:
    out = _i(0)
    _check("mla_decode_uses_short_path",
           lib.mla_decode_uses_short_path(int(B), int(n_q), int(max_kv_len), int(split_pages), ctypes.byref(out)))
    return bool(out.value)


def alloc_workspace(B, n_q, max_kv_len, split_pages=0, device=None):
    n = mla_decode_workspace_size(B, n_q, max_kv_len, split_pages)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def _decode_args(q_abs, cache, page_table, kv_lens, n_q, max_kv_len, split_pages, workspace, o_latent,
                 lse, stream):
    B = kv_lens.shape[0]
    return (
        _dev(q_abs, "q_abs", torch.bfloat16, (B, n_q, N_HEADS, D_ROW)),
        _dev(cache, "cache", torch.bfloat16), int(cache.shape[0]),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(kv_lens, "kv_lens", torch.int32, (B,)),
        int(B), int(n_q), int(max_kv_len), int(split_pages),
        0 if workspace is None else _dev(workspace, "workspace", torch.uint8),
        0 if workspace is None else workspace.numel(),
        _dev(o_latent, "o_latent", torch.float32, (B, n_q, N_HEADS, D_LATENT)),
        0 if lse is None else _dev(lse, "lse", torch.float32, (B, n_q, N_HEADS)),
        _stream(stream))


def mla_decode_attn(q_abs, cache, page_table, kv_lens, n_q, max_kv_len, split_pages=0, workspace=None,
                    o_latent=None, lse=None, stream=None, want_lse=True):
    """Split attention plus combine; returns (o_latent [B,n_q,128,512] f32, lse [B,n_q,128] f32 or None)."""
    B = kv_lens.shape[0]
    if o_latent is None:
        o_latent = torch.empty(B, n_q, N_HEADS, D_LATENT, dtype=torch.float32, device=q_abs.device)
    if lse is None and want_lse:
        lse = torch.empty(B, n_q, N_HEADS, dtype=torch.float32, device=q_abs.device)
    if workspace is None:
        workspace = alloc_workspace(B, n_q, max_kv_len, split_pages, q_abs.device)
    _check("mla_decode_attn", lib.mla_decode_attn(*_decode_args(
        q_abs, cache, page_table, kv_lens, n_q, max_kv_len, split_pages, workspace, o_latent, lse, stream)))
    return o_latent, lse


def mla_decode_attn_partial(q_abs, cache, page_table, kv_lens, n_q, max_kv_len, split_pages, workspace,
                            o_latent, lse=None, stream=None):
    _check("mla_decode_attn_partial", lib.mla_decode_attn_partial(*_decode_args(
        q_abs, cache, page_table, kv_lens, n_q, max_kv_len, split_pages, workspace, o_latent, lse, stream)))


def mla_decode_combine(B, n_q, max_kv_len, split_pages, workspace, o_latent, lse=None, stream=None):
    _check("mla_decode_combine", lib.mla_decode_combine(
        int(B), int(n_q), int(max_kv_len), int(split_pages),
        0 if workspace is None else _dev(workspace, "workspace", torch.uint8),
        0 if workspace is None else workspace.numel(),
        _dev(o_latent, "o_latent", torch.float32, (B, n_q, N_HEADS, D_LATENT)),
        0 if lse is None else _dev(lse, "lse", torch.float32, (B, n_q, N_HEADS)),
        _stream(stream)))


def mla_out_absorb(o_latent, w_uv, out=None, stream=None):
    B, n_q = o_latent.shape[:2]
    if out is None:
        out = torch.empty(B, n_q, N_HEADS, D_NOPE, dtype=torch.bfloat16, device=o_latent.device)
    _check("mla_out_absorb", lib.mla_out_absorb(
        _dev(o_latent, "o_latent", torch.float32, (B, n_q, N_HEADS, D_LATENT)),
        _dev(w_uv, "w_uv", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev_or_pinned(out, "out", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        int(B), int(n_q), _stream(stream)))
    return out


def mla_combine_out_absorb(B, n_q, max_kv_len, split_pages, workspace, o_latent, w_uv, out=None, lse=None,
                           stream=None):
    """Split merge + value up-projection in one launch (the merged O' is not written)."""
    if out is None:
        out = torch.empty(B, n_q, N_HEADS, D_NOPE, dtype=torch.bfloat16, device=w_uv.device)
    _check("mla_combine_out_absorb", lib.mla_combine_out_absorb(
        int(B), int(n_q), int(max_kv_len), int(split_pages),
        0 if workspace is None else _dev(workspace, "workspace", torch.uint8),
        0 if workspace is None else workspace.numel(),
        0 if o_latent is None else _dev(o_latent, "o_latent", torch.float32, (B, n_q, N_HEADS, D_LATENT)),
        _dev(w_uv, "w_uv", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev_or_pinned(out, "out", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        0 if lse is None else _dev(lse, "lse", torch.float32, (B, n_q, N_HEADS)),
        _stream(stream)))
    return out


def mla_decompress_kv(cache, page_table, kv_lens, max_kv_len, w_uk, w_uv, k_nope=None, v=None, stream=None):
    """Non-absorbed path: per-head keys and values [B, 128, max_kv_len, 128] decompressed from the cache."""
    B = int(kv_lens.shape[0])
    shape = (B, N_HEADS, int(max_kv_len), D_NOPE)
    if k_nope is None:
        k_nope = torch.empty(shape, dtype=torch.bfloat16, device=cache.device)
    if v is None:
        v = torch.empty(shape, dtype=torch.bfloat16, device=cache.device)
    _check("mla_decompress_kv", lib.mla_decompress_kv(
        _dev(cache, "cache", torch.bfloat16), int(cache.shape[0]),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(kv_lens, "kv_lens", torch.int32, (B,)), B, int(max_kv_len),
        _dev(w_uk, "w_uk", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev(w_uv, "w_uv", torch.bfloat16, (N_HEADS, D_NOPE, D_LATENT)),
        _dev(k_nope, "k_nope", torch.bfloat16, shape), _dev(v, "v", torch.bfloat16, shape), _stream(stream)))
    return k_nope, v


def mla_prefill_attn(q_nope, q_rope, seq_lens_before, rope, k_nope, v, cache, page_table, kv_lens,
                     out=None, lse=None, stream=None):
    """Non-absorbed path: causal MHA of the new tokens over the decompressed keys and values."""
    B, n_q = q_nope.shape[:2]
    max_kv_len = int(k_nope.shape[2])
    if out is None:
        out = torch.empty(B, n_q, N_HEADS, D_NOPE, dtype=torch.bfloat16, device=q_nope.device)
    _check("mla_prefill_attn", lib.mla_prefill_attn(
        _dev(q_nope, "q_nope", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        _dev(q_rope, "q_rope", torch.bfloat16, (B, n_q, N_HEADS, D_ROPE)),
        _dev(seq_lens_before, "seq_lens_before", torch.int32, (B,)),
        _dev(rope, "rope_table", torch.float32), int(rope.shape[0]),
        _dev(k_nope, "k_nope", torch.bfloat16, (B, N_HEADS, max_kv_len, D_NOPE)),
        _dev(v, "v", torch.bfloat16, (B, N_HEADS, max_kv_len, D_NOPE)), max_kv_len,
        _dev(cache, "cache", torch.bfloat16), int(cache.shape[0]),
        _dev(page_table, "page_table", torch.int32), int(page_table.shape[1]),
        _dev(kv_lens, "kv_lens", torch.int32, (B,)), int(B), int(n_q),
        _dev(out, "out", torch.bfloat16, (B, n_q, N_HEADS, D_NOPE)),
        0 if lse is None else _dev(lse, "lse", torch.float32, (B, n_q, N_HEADS)),
        _stream(stream)))
    return out


def mla_set_launch_overlap(level: int):
    """0: plain stream order; 1: programmatic dependent launch (prologues overlap
    the previous kernel); 2: as 1 and the weights are read before the previous
    kernel finishes (only while nothing in flight writes them)."""
    _check("mla_set_launch_overlap", lib.mla_set_launch_overlap(int(level)))


def mla_get_launch_overlap() -> int:
    return int(lib.mla_get_launch_overlap())


def mla_get_device_status(stream=None) -> int:
    return int(lib.mla_get_device_status(_stream(stream)))
