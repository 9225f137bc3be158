"""Parity of the FP8-latent-cache path (through the C ABI) with the CPU oracle.

The cache image (E4M3 codes, float32 scales, float16 keys) must match the
oracle's own append bit for bit; the outputs must match the oracle's plain
definition evaluated on the dequantised cache values within the tolerances of
the bf16 path (O: max-abs 1e-2, relative L2 5e-3; O' relative L2 5e-3; lse
max-abs 2e-2), at small sizes with ragged tails and at the benchmark size on
sampled sequences and heads.
"""

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from mla_absorbed_decode_absorb_gb300 import workloads as W
from test_gpu_parity import LAT_REL_L2, LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, bits, rel_l2, run_session

pytestmark = pytest.mark.gpu


def oracle_fp8_images(inp: W.Inputs):
    """The oracle's append of every sequence's history, then of this step's tokens."""
    P = inp.num_pages
    img = (np.full((P, 64, 512), 0x7F, np.uint8), np.full((P, 64), np.nan, np.float32),
           np.full((P, 64, 64), 0x7E00, np.uint16))
    pt = inp.page_table.numpy()
    for b in range(inp.batch):
        hc, hk = inp.history(b)
        if hc.shape[0]:
            img = O.append_kv_fp8(*img, bits(hc)[None], bits(hk)[None], [0], pt[b:b + 1])
    c_new, k_new = inp.new_tokens()
    return O.append_kv_fp8(*img, bits(c_new), bits(k_new), inp.prior_lens.numpy(), pt)


def oracle_sequence_fp8(inp: W.Inputs, img, b: int, heads=None):
    kv = int(inp.kv_lens[b])
    c, kr = O.gather_sequence_fp8(*img, inp.page_table.numpy()[b], kv)
    q_nope = O.bf16_bits_to_f64(bits(inp.q_nope[b]))
    q_rope = O.bf16_bits_to_f64(bits(inp.q_rope[b]))
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    return O.decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, int(inp.prior_lens[b]), heads)


def gpu_images(s):
    c8, scale, kr = s.cache_fp8
    return (c8.cpu().numpy(), scale.cpu().numpy(), kr.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def check_outputs_fp8(s, inp, img, seqs, heads=None):
    if s.fused_finish and s.num_splits > 1:
        s.combine()
        torch.cuda.synchronize()
    o_gpu = s.out.float().cpu().numpy()
    lat_gpu = s.o_latent.cpu().numpy()
    lse_gpu = s.lse.cpu().numpy()
    hsel = slice(None) if heads is None else list(heads)
    o_all, o_ref_all, lat_all, lat_ref_all = [], [], [], []
    for b in seqs:
        o_ref, lat_ref, lse_ref = oracle_sequence_fp8(inp, img, b, heads)
        o, lat, lse = o_gpu[b][:, hsel], lat_gpu[b][:, hsel], lse_gpu[b][:, hsel]
        assert np.isfinite(o).all() and np.isfinite(lat).all()
        assert np.abs(lse - lse_ref).max() <= LSE_MAX_ABS, (b, np.abs(lse - lse_ref).max())
        o_all.append(o), o_ref_all.append(o_ref), lat_all.append(lat), lat_ref_all.append(lat_ref)
    o, o_ref = np.concatenate(o_all), np.concatenate(o_ref_all)
    lat, lat_ref = np.concatenate(lat_all), np.concatenate(lat_ref_all)
    assert np.abs(o - o_ref).max() <= O_MAX_ABS, np.abs(o - o_ref).max()
    assert rel_l2(o, o_ref) <= O_REL_L2, rel_l2(o, o_ref)
    assert rel_l2(lat, lat_ref) <= LAT_REL_L2, rel_l2(lat, lat_ref)


SMALL = {
    "edges_q1": W.custom("edges_q1_fp8", [0, 62, 63, 64, 127, 300], n_q=1, cache_format="fp8"),
    "mtp_q4": W.custom("mtp_q4_fp8", [0, 1, 61, 124, 200], n_q=4, cache_format="fp8"),
    "long_tail": W.custom("long_tail_fp8", [1500, 1029], n_q=1, cache_format="fp8"),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_fp8_append_bit_exact(name):
    inp = W.generate(SMALL[name], seed=3)
    s = run_session(inp)
    got, ref = gpu_images(s), oracle_fp8_images(inp)
    assert np.array_equal(got[0], ref[0])
    assert np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))
    assert np.array_equal(got[2], ref[2])


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("split_pages", [0, 1, 3])
def test_fp8_decode_parity_small(name, split_pages):
    inp = W.generate(SMALL[name], seed=4)
    s = run_session(inp, split_pages=split_pages)
    check_outputs_fp8(s, inp, oracle_fp8_images(inp), range(inp.batch))


def test_fp8_fused_append_absorb_matches_separate_calls():
    """mla_append_absorb_q_fp8 writes the cache image and q_abs of mla_append_kv_fp8
    followed by mla_absorb_q, bit for bit."""
    inp = W.generate(SMALL["mtp_q4"], seed=12)
    a = run_session(inp, fused_prologue=True)
    b = run_session(inp, fused_prologue=False)
    assert a.stage_names()[0] == "append_absorb" and b.stage_names()[:2] == ["append", "absorb"]
    for x, y in zip(gpu_images(a), gpu_images(b)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert np.array_equal(bits(a.q_abs), bits(b.q_abs))
    assert np.array_equal(bits(a.out), bits(b.out))


def test_fp8_decode_full_size_sampled():
    """The FP8 benchmark workload at full size, in the bench's launch configuration:
    sampled sequences (first, middle, last) on sampled heads."""
    wl = W.FP8_WORKLOADS["batched_b32_l4096_fp8"]
    inp = W.generate(wl, seed=0)
    s = run_session(inp)
    seqs = [0, inp.batch // 2, inp.batch - 1]
    check_outputs_fp8(s, inp, oracle_fp8_images(inp), seqs, heads=[0, 41, 127])
