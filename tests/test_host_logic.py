"""Host-side logic: the seeded workload generator and the byte/FLOP accounting."""

import math

import torch

from mla_absorbed_decode_absorb_gb300 import accounting as A
from mla_absorbed_decode_absorb_gb300 import workloads as W


def test_generator_is_deterministic():
    wl = W.custom("t", [3, 70], n_q=2)
    a, b = W.generate(wl, seed=5), W.generate(wl, seed=5)
    for x, y in [(a.c_kv, b.c_kv), (a.q_nope, b.q_nope), (a.page_table, b.page_table), (a.w_uk, b.w_uk)]:
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
    c = W.generate(wl, seed=6)
    assert not torch.equal(a.c_kv.view(torch.int16), c.c_kv.view(torch.int16))


def test_page_tables_are_shuffled_and_disjoint():
    wl = W.custom("t", [0, 63, 64, 200, 1000], n_q=1)
    inp = W.generate(wl, seed=0)
    used = []
    for b, kv in enumerate(inp.kv_lens.tolist()):
        need = math.ceil(kv / 64)
        row = inp.page_table[b].tolist()
        assert all(p >= 0 for p in row[:need]) and all(p == -1 for p in row[need:])
        used += row[:need]
    assert len(used) == len(set(used))
    assert max(used) < inp.num_pages == len(used) + math.ceil(0.1 * len(used))
    assert used != sorted(used)


def test_shapes_and_distributions():
    inp = W.generate(W.custom("t", [500], n_q=4), seed=0)
    assert inp.kv_lens.tolist() == [504] and inp.prior_lens.tolist() == [500]
    assert inp.c_kv.shape == (504, 512) and inp.k_pe.shape == (504, 64)
    assert inp.q_nope.shape == (1, 4, 128, 128) and inp.q_rope.shape == (1, 4, 128, 64)
    assert abs(float(inp.w_uk.float().std()) - 0.02) < 0.001
    assert abs(float(inp.c_kv.float().std()) - 1.0) < 0.02
    c_new, k_new = inp.new_tokens()
    assert torch.equal(c_new[0, 0].view(torch.int16), inp.c_kv[500].view(torch.int16))


def test_ragged_lengths_in_range():
    wl = W.scaled(W.WORKLOADS["ragged_b128_l1024_8192"], batch=16)
    g = torch.Generator().manual_seed(0)
    L = torch.randint(1024, 8193, (16,), generator=g)
    assert L.min() >= 1024 and L.max() <= 8192


def test_bench_workload_accounting():
    """Config 2 (B=32, L=4096): 32*4097*1152 B and 36.52 GFLOP of attention."""
    kv = [4097] * 32
    assert A.step_cache_bytes(kv) == 32 * 4097 * 1152
    assert abs(A.step_cache_bytes(kv) / 1e6 - 151.03) < 0.01
    assert abs(A.step_attention_flops(kv, 1) / 1e9 - 36.52) < 0.01
    # MTP: 4 causal queries share each cache read
    f = A.step_attention_flops([8196], 4)
    assert f == sum(8192 + j + 1 for j in range(4)) * A.flops_per_token_pair()
    t, bound = A.roofline_seconds(kv, 1, 6798.2, 1931.1)
    assert bound == "hbm" and abs(t * 1e6 - 22.22) < 0.01
