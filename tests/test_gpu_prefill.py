"""The non-absorbed (prefill / chunked-prefill) path through the C ABI, against the oracle.

mla_decompress_kv must give the oracle's per-head keys and values (bf16 outputs of
an fp32 accumulation: within 2^-8 relative plus a small absolute floor), and
zeros in the rows up to the next 128-token boundary; mla_prefill_attn must give
the oracle's output O within max-abs 1e-2 and relative L2 5e-3 (as the absorbed
path), and its log-sum-exp within 5e-3 (the largest error seen is 1.5e-3, on the
2048-token prompt).  The same session switches to this path
for steps of 64 or more new tokens.
"""

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from mla_absorbed_decode_absorb_gb300 import workloads as W

from test_gpu_parity import bits, oracle_sequence, rel_l2

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_L2, LSE_MAX_ABS = 1e-2, 5e-3, 5e-3


def session(inp, **kw):
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession
    s = DecodeSession(inp, **kw)
    s.step()
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    return s


def check_prefill(s, inp, heads):
    o_gpu = s.out.float().cpu().numpy()
    lse_gpu = s.lse.cpu().numpy()
    o_all, r_all, dl = [], [], 0.0
    for b in range(inp.batch):
        o_ref, _, lse_ref = oracle_sequence(inp, b, heads)
        o = o_gpu[b][:, heads]
        assert np.isfinite(o).all()
        dl = max(dl, float(np.abs(lse_gpu[b][:, heads] - lse_ref).max()))
        o_all.append(o), r_all.append(o_ref)
    o, r = np.concatenate(o_all), np.concatenate(r_all)
    print(f"prefill {inp.batch} x {inp.n_q}: rel-L2 O {rel_l2(o, r):.3e} max |dO| {np.abs(o - r).max():.3e} "
          f"max |dlse| {dl:.3e}")
    assert dl <= LSE_MAX_ABS, dl
    assert np.abs(o - r).max() <= O_MAX_ABS, np.abs(o - r).max()
    assert rel_l2(o, r) <= O_REL_L2, rel_l2(o, r)
    return rel_l2(o, r)


def test_decompress_kv_parity():
    inp = W.generate(W.custom("decompress", [0, 63, 200, 700], n_q=64), seed=21)
    s = session(inp)
    assert s.path == "non_absorbed"
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    k_gpu = s.k_nope.float().cpu().numpy()
    v_gpu = s.v.float().cpu().numpy()
    heads = list(range(128))  # every (head, K or V) unit of the decompression's work list
    for b in range(inp.batch):
        c_bits, _ = (bits(x) for x in inp.sequence(b))
        c = O.bf16_bits_to_f64(c_bits)
        kv = c.shape[0]
        k_ref, v_ref = O.decompress_kv(c, w_uk[heads], w_uv[heads])
        for got, ref in ((k_gpu, k_ref), (v_gpu, v_ref)):
            g = got[b][heads][:, :kv].transpose(1, 0, 2)
            tol = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
            assert (np.abs(g - ref) <= tol).all(), np.abs(g - ref).max()
            pad_end = min(s.max_kv_len, (kv + 127) // 128 * 128)
            assert (got[b][:, kv:pad_end] == 0).all()


def test_decompress_kv_ragged_writes_only_its_tiles():
    """Ragged lengths (half a tile, one past a page, tile edges, one long
    sequence): the oracle's keys and values for sampled heads, zeros up to the
    next 128-token boundary, and nothing written past it (the outputs start
    filled with a sentinel)."""
    from mla_absorbed_decode_absorb_gb300 import ops
    inp = W.generate(W.custom("decompress_ragged", [0, 1, 127, 128, 300, 0, 900], n_q=64), seed=24)
    s = session(inp)
    sentinel = 7.0
    k = torch.full(tuple(s.k_nope.shape), sentinel, dtype=torch.bfloat16, device=s.k_nope.device)
    v = torch.full_like(k, sentinel)
    ops.mla_decompress_kv(s.cache, s.page_table, s.kv_lens, s.max_kv_len, s.w_uk, s.w_uv, k_nope=k, v=v)
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    heads = [0, 1, 63, 64, 126, 127]
    k_gpu = k.float().cpu().numpy()
    v_gpu = v.float().cpu().numpy()
    for b in range(inp.batch):
        c = O.bf16_bits_to_f64(bits(inp.sequence(b)[0]))
        kv = c.shape[0]
        k_ref, v_ref = O.decompress_kv(c, w_uk[heads], w_uv[heads])
        pad_end = min(s.max_kv_len, (kv + 127) // 128 * 128)
        for got, ref in ((k_gpu, k_ref), (v_gpu, v_ref)):
            g = got[b][heads][:, :kv].transpose(1, 0, 2)
            tol = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
            assert (np.abs(g - ref) <= tol).all(), (b, np.abs(g - ref).max())
            assert (got[b][:, kv:pad_end] == 0).all(), b
            assert (got[b][:, pad_end:] == sentinel).all(), b


def test_decompress_kv_bad_inputs_leave_other_sequences_intact():
    """A page id past the pool, then a length past max_kv_len, in one sequence:
    MLA_ERR_BOUNDS (read and cleared), and every other sequence's keys and values
    are still the oracle's, although the CTA pairs that share weight loads mix
    tiles of different sequences."""
    from mla_absorbed_decode_absorb_gb300 import ops
    inp = W.generate(W.custom("decompress_bad", [200, 0, 130, 300], n_q=64), seed=25)
    s = session(inp)
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    heads = [0, 77, 127]

    def check(k, v, skip):
        k_gpu, v_gpu = k.float().cpu().numpy(), v.float().cpu().numpy()
        for b in range(inp.batch):
            if b == skip:
                continue
            c = O.bf16_bits_to_f64(bits(inp.sequence(b)[0]))
            kv = c.shape[0]
            k_ref, v_ref = O.decompress_kv(c, w_uk[heads], w_uv[heads])
            for got, ref in ((k_gpu, k_ref), (v_gpu, v_ref)):
                g = got[b][heads][:, :kv].transpose(1, 0, 2)
                tol = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
                assert (np.abs(g - ref) <= tol).all(), (b, np.abs(g - ref).max())

    pt = s.page_table.clone()
    pt[1, 0] = inp.num_pages + 5   # sequence 1's only page, past the pool
    k, v = ops.mla_decompress_kv(s.cache, pt, s.kv_lens, s.max_kv_len, s.w_uk, s.w_uv)
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_ERR_BOUNDS
    assert ops.mla_get_device_status() == ops.MLA_OK
    check(k, v, skip=1)

    kv_lens = s.kv_lens.clone()
    kv_lens[2] = s.max_kv_len + 1   # longer than the buffers
    k, v = ops.mla_decompress_kv(s.cache, s.page_table, kv_lens, s.max_kv_len, s.w_uk, s.w_uv)
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_ERR_BOUNDS
    assert ops.mla_get_device_status() == ops.MLA_OK
    check(k, v, skip=2)


@pytest.mark.parametrize("lengths,n_q", [([0, 1, 63, 500], 64), ([130, 0], 100), ([64, 1000], 129), ([300], 256)])
def test_prefill_parity(lengths, n_q):
    inp = W.generate(W.custom("prefill", lengths, n_q=n_q), seed=22)
    s = session(inp)
    assert s.path == "non_absorbed" and s.launches_per_step() == 3
    check_prefill(s, inp, heads=[0, 77, 127])


@pytest.mark.parametrize("n_q", [1, 4])
def test_both_paths_agree_on_short_steps(n_q):
    """A short step through the non-absorbed path: the oracle's answer, and
    close to the absorbed path's (different roundings, same definition)."""
    inp = W.generate(W.custom("both", [0, 70, 640], n_q=n_q), seed=23)
    a = session(inp, path="absorbed")
    n = session(inp, path="non_absorbed")
    assert a.path == "absorbed" and n.path == "non_absorbed"
    check_prefill(n, inp, heads=[0, 31, 127])
    assert rel_l2(n.out.float().cpu().numpy(), a.out.float().cpu().numpy()) <= 2 * O_REL_L2


@pytest.mark.parametrize("name", sorted(n for n in W.PREFILL_WORKLOADS if n in ("chunk_b4_l4096_c512", "prompt_b8_c2048")))
def test_prefill_full_size_sampled(name):
    """The benched non-absorbed workloads at full size, in the bench's launch
    configuration: a chunk of 512 new tokens after 4096 (B = 4; four query tiles
    over 4,608 keys) and a 2048-token prompt (B = 8; sixteen query tiles per head).
    The oracle checks every new token of the first and the last sequence on three
    heads (the decompressed keys and values, O and lse), which spans every query
    tile and every key tile of those sequences."""
    inp = W.generate(W.PREFILL_WORKLOADS[name], seed=0)
    s = session(inp)
    assert s.path == "non_absorbed"
    heads = [0, 77, 127]
    o_gpu = s.out.float().cpu().numpy()
    lse_gpu = s.lse.cpu().numpy()
    o_all, r_all, dl = [], [], 0.0
    for b in sorted({0, inp.batch - 1}):
        o_ref, _, lse_ref = oracle_sequence(inp, b, heads)
        o = o_gpu[b][:, heads]
        assert np.isfinite(o).all()
        dl = max(dl, float(np.abs(lse_gpu[b][:, heads] - lse_ref).max()))
        o_all.append(o), r_all.append(o_ref)
    o, r = np.concatenate(o_all), np.concatenate(r_all)
    print(f"{name}: rel-L2 O {rel_l2(o, r):.3e} max |dO| {np.abs(o - r).max():.3e} max |dlse| {dl:.3e}")
    assert dl <= LSE_MAX_ABS, dl
    assert np.abs(o - r).max() <= O_MAX_ABS, np.abs(o - r).max()
    assert rel_l2(o, r) <= O_REL_L2, rel_l2(o, r)
