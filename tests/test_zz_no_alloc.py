"""mla_decode_attn_noalloc: the decode attention entry point for callers that may
not allocate device memory (its split partials live in a fixed array inside the
library).  Called through the C ABI, its output must equal mla_decode_attn's on
the same inputs bit for bit (both run the same kernels on the same split plan,
so any difference means a wrong place in the array), on two calls in a row (the
second reuses the array the first call left behind), also for a single-split
plan that writes the output directly; a plan too large for the array must be
refused.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from mla_absorbed_decode_absorb_gb300 import workloads as W

pytestmark = pytest.mark.gpu


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


def bits32(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy()


@pytest.mark.parametrize("lens,n_q,split_pages", [([1500, 900, 2000], 2, 4), ([300, 40], 1, 1000), ([300], 1, 0)])
def test_noalloc_equals_decode_attn_twice(lens, n_q, split_pages):
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession

    f = _noalloc(ops.lib)
    inp = W.generate(W.custom("noalloc", lens, n_q=n_q), seed=7)
    s = DecodeSession(inp, split_pages=split_pages)
    s.step()  # cache holds the new tokens, q_abs is filled
    ref_o, ref_lse = ops.mla_decode_attn(s.q_abs, s.cache, s.page_table, s.kv_lens, s.n_q, s.max_kv_len,
                                         split_pages)
    torch.cuda.synchronize()
    # the first case sends its partials through the library's array, the second
    # (splits longer than the sequences) has one split and writes O' directly, the
    # third (one short sequence, automatic split) runs the short-context kernel
    assert (s.num_splits > 1) == (split_pages == 4)
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _call(f, s, split_pages, o, lse) == ops.MLA_OK
        torch.cuda.synchronize()
        assert ops.mla_get_device_status() == ops.MLA_OK
        assert np.array_equal(bits32(o), bits32(ref_o))
        assert np.array_equal(bits32(lse), bits32(ref_lse))


def test_noalloc_refuses_a_plan_larger_than_its_array():
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession

    f = _noalloc(ops.lib)
    inp = W.generate(W.custom("noalloc_big", [4000] * 8, n_q=1), seed=8)
    s = DecodeSession(inp, split_pages=1)   # 8 sequences x 63 splits > 127 units
    s.step()
    o = torch.zeros_like(s.o_latent)
    lse = torch.zeros_like(s.lse)
    assert _call(f, s, 1, o, lse) == ops.MLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert float(o.abs().sum()) == 0.0  # nothing was launched
