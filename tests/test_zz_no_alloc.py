"""mla_decode_attn_noalloc: the decode attention entry point for callers that may
not allocate device memory (its split partials live in a fixed array inside the
library).  Called through the C ABI, its output must match mla_decode_attn's on
the same inputs, on two calls in a row (the second reuses the array the first
call left behind), and a plan too large for the array must be refused.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from mla_absorbed_decode_absorb_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LAT_REL_L2 = 5e-3     # same bound as the latent-output parity tests
LSE_MAX_ABS = 2e-2


def _noalloc(lib):
    f = lib.mla_decode_attn_noalloc
    p, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [p, p, i64, p, i, p, i, i, i, i, p, p, p]
    f.restype = i
    return f


def _call(f, s, split_pages, o, lse):
    return f(s.q_abs.data_ptr(), s.cache.data_ptr(), s.cache.shape[0], s.page_table.data_ptr(),
             s.page_table.shape[1], s.kv_lens.data_ptr(), s.B, s.n_q, s.max_kv_len, split_pages,
             o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def test_noalloc_matches_decode_attn_twice():
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession

    f = _noalloc(ops.lib)
    inp = W.generate(W.custom("noalloc", [1500, 900, 2000], n_q=2), seed=7)
    split_pages = 4
    s = DecodeSession(inp, split_pages=split_pages)
    s.step()  # cache holds the new tokens, q_abs is filled
    assert s.num_splits > 1  # the partials really go through the library's array
    ref_o, ref_lse = ops.mla_decode_attn(s.q_abs, s.cache, s.page_table, s.kv_lens, s.n_q, s.max_kv_len,
                                         split_pages)
    torch.cuda.synchronize()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _call(f, s, split_pages, o, lse) == ops.MLA_OK
        torch.cuda.synchronize()
        assert ops.mla_get_device_status() == ops.MLA_OK
        assert rel_l2(o.cpu().numpy(), ref_o.cpu().numpy()) <= LAT_REL_L2
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= LSE_MAX_ABS


def test_noalloc_refuses_a_plan_larger_than_its_array():
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession

    f = _noalloc(ops.lib)
    inp = W.generate(W.custom("noalloc_big", [4000] * 8, n_q=1), seed=8)
    s = DecodeSession(inp, split_pages=1)   # 8 sequences x 63 splits > 63 units
    s.step()
    o = torch.zeros_like(s.o_latent)
    lse = torch.zeros_like(s.lse)
    assert _call(f, s, 1, o, lse) == ops.MLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert float(o.abs().sum()) == 0.0  # nothing was launched
