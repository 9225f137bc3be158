"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element.

Tolerances: the append's cache image must match bit for bit; the final output O
must match the fp64 oracle within max-abs 1e-2 and relative L2 5e-3 (bf16
operands, fp32 accumulation).  O' and the log-sum-exp are checked too.
"""

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from mla_absorbed_decode_absorb_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_L2 = 1e-2, 5e-3       # final output O
LAT_REL_L2 = 5e-3                      # latent output O'
# log-sum-exp, natural-log units.  Its error comes from the bf16 query (2^-9
# relative per element) and the fp16 partial-score exchange.  With one or two
# visible tokens the lse is essentially one score and carries that error whole
# (up to 2.3e-3 seen in the small cases); over thousands of tokens the softmax
# weights average it down (at most 6.0e-4 over every head and query of the five
# full-size workloads).  The bound keeps a margin of about 2x over the largest.
LSE_MAX_ABS = 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def oracle_cache_image(inp: W.Inputs) -> np.ndarray:
    """The oracle's own append of every sequence's history, then of this step's tokens."""
    img = np.full((inp.num_pages, 64, 576), W.CACHE_SENTINEL_BITS, dtype=np.uint16)
    pt = inp.page_table.numpy()
    for b in range(inp.batch):
        hc, hk = inp.history(b)
        if hc.shape[0]:
            img = O.append_kv(img, bits(hc)[None], bits(hk)[None], [0], pt[b:b + 1])
    c_new, k_new = inp.new_tokens()
    return O.append_kv(img, bits(c_new), bits(k_new), inp.prior_lens.numpy(), pt)


def oracle_sequence(inp: W.Inputs, b: int, heads=None):
    """Oracle outputs for sequence b from the cache rows the oracle's append writes."""
    c_bits, k_bits = (bits(x) for x in inp.sequence(b))
    kv = c_bits.shape[0]
    c = O.bf16_bits_to_f64(c_bits)
    kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(kv)))
    q_nope = O.bf16_bits_to_f64(bits(inp.q_nope[b]))
    q_rope = O.bf16_bits_to_f64(bits(inp.q_rope[b]))
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    return O.decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, int(inp.prior_lens[b]), heads)


def run_session(inp, split_pages=None, **kw):
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession
    s = DecodeSession(inp, split_pages=split_pages, **kw)
    s.step()
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    return s


def check_outputs(s, inp, seqs, heads=None):
    if s.fused_finish and s.num_splits > 1:
        s.combine()  # the fused finish does not write the merged O'; the partials are still there
        torch.cuda.synchronize()
    o_gpu = s.out.float().cpu().numpy()
    lat_gpu = s.o_latent.cpu().numpy()
    lse_gpu = s.lse.cpu().numpy()
    hsel = slice(None) if heads is None else list(heads)
    o_all, o_ref_all, lat_all, lat_ref_all = [], [], [], []
    for b in seqs:
        o_ref, lat_ref, lse_ref = oracle_sequence(inp, b, heads)
        o, lat, lse = o_gpu[b][:, hsel], lat_gpu[b][:, hsel], lse_gpu[b][:, hsel]
        assert np.isfinite(o).all() and np.isfinite(lat).all()
        assert np.abs(lse - lse_ref).max() <= LSE_MAX_ABS, (b, np.abs(lse - lse_ref).max())
        o_all.append(o), o_ref_all.append(o_ref), lat_all.append(lat), lat_ref_all.append(lat_ref)
    o, o_ref = np.concatenate(o_all), np.concatenate(o_ref_all)
    lat, lat_ref = np.concatenate(lat_all), np.concatenate(lat_ref_all)
    assert np.abs(o - o_ref).max() <= O_MAX_ABS, np.abs(o - o_ref).max()
    assert rel_l2(o, o_ref) <= O_REL_L2, rel_l2(o, o_ref)
    assert rel_l2(lat, lat_ref) <= LAT_REL_L2, rel_l2(lat, lat_ref)
    return rel_l2(o, o_ref), rel_l2(lat, lat_ref)


# ------------------------------------------------------------------------ small cases
SMALL = {
    # kv_len = L + n_q spans: a single token, one short of a page, exactly a page, one over,
    # several pages with a ragged tail
    "edges_q1": W.custom("edges_q1", [0, 62, 63, 64, 127, 300], n_q=1),
    "mtp_q4": W.custom("mtp_q4", [0, 1, 61, 124, 200], n_q=4),
    "mtp_q2": W.custom("mtp_q2", [0, 63, 64, 255], n_q=2),
    "long_tail": W.custom("long_tail", [1500, 1029], n_q=1),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_append_bit_exact(name):
    inp = W.generate(SMALL[name], seed=1)
    s = run_session(inp)
    assert np.array_equal(bits(s.cache), oracle_cache_image(inp))


def test_absorb_q_parity():
    inp = W.generate(W.custom("absorb", [5, 70, 4000], n_q=3), seed=2)
    s = run_session(inp)
    pos = inp.prior_lens.numpy()[:, None] + np.arange(3)[None, :]
    ref = O.absorb_query(O.bf16_bits_to_f64(bits(inp.q_nope)), O.bf16_bits_to_f64(bits(inp.q_rope)),
                         O.bf16_bits_to_f64(bits(inp.w_uk)), pos)
    got = s.q_abs.float().cpu().numpy()
    tol = 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max()
    assert (np.abs(got - ref) <= tol).all(), np.abs(got - ref).max()


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("split_pages", [0, 1, 3])
def test_decode_parity_small(name, split_pages):
    inp = W.generate(SMALL[name], seed=3)
    s = run_session(inp, split_pages=split_pages)
    check_outputs(s, inp, range(inp.batch))


@pytest.mark.parametrize("split_pages", [0, 1, 3, 1000])
def test_fused_finish_matches_combine_then_out_absorb(split_pages):
    """mla_combine_out_absorb performs the merge with the same float32 operations
    as mla_decode_combine and the product as mla_out_absorb: equal bit for bit."""
    inp = W.generate(W.custom("fused", [0, 63, 700, 2500, 64], n_q=2), seed=6)
    a = run_session(inp, split_pages=split_pages, fused_finish=True)
    b = run_session(inp, split_pages=split_pages, fused_finish=False)
    assert np.array_equal(bits(a.out), bits(b.out))
    assert np.array_equal(a.lse.cpu().numpy().view(np.uint32), b.lse.cpu().numpy().view(np.uint32))


def test_append_on_side_stream_matches_in_order():
    inp = W.generate(W.custom("overlap", [10, 64, 333], n_q=3), seed=7)
    a = run_session(inp, overlap_append=True)
    b = run_session(inp, overlap_append=False)
    assert np.array_equal(bits(a.cache), bits(b.cache))
    assert np.array_equal(bits(a.out), bits(b.out))


@pytest.mark.parametrize("lens,n_q", [([10, 64, 333], 3), ([0, 63, 127, 4000], 1), ([5, 200], 4)])
def test_fused_append_absorb_matches_separate_calls(lens, n_q):
    """mla_append_absorb_q writes the cache rows and q_abs of mla_append_kv followed
    by mla_absorb_q, bit for bit (and so the step's outputs)."""
    inp = W.generate(W.custom("prologue", lens, n_q=n_q), seed=11)
    a = run_session(inp, fused_prologue=True)
    b = run_session(inp, fused_prologue=False)
    assert a.stage_names()[0] == "append_absorb" and b.stage_names()[:2] == ["append", "absorb"]
    assert a.launches_per_step() == b.launches_per_step() - 1
    for x, y in [(a.cache, b.cache), (a.q_abs, b.q_abs), (a.out, b.out)]:
        assert np.array_equal(bits(x), bits(y))


@pytest.mark.parametrize("level", [0, 2])
def test_graph_replay_matches_eager_steps(level):
    """A step captured as a CUDA graph gives the eager step's bits, and picks up new
    step inputs written into the session's buffers between replays."""
    from mla_absorbed_decode_absorb_gb300 import ops
    before = ops.mla_get_launch_overlap()
    ops.mla_set_launch_overlap(level)
    try:
        inp = W.generate(W.custom("graph", [5, 700, 4000], n_q=2), seed=14)
        s = run_session(inp)
        eager = bits(s.out).copy()
        g = s.capture()
        s.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ops.mla_get_device_status() == ops.MLA_OK
        assert np.array_equal(bits(s.out), eager)
        # new step inputs through the same graph, against an eager step on them
        gen = torch.Generator().manual_seed(15)
        for t in (s.q_nope, s.q_rope, s.c_new, s.k_new):
            t.copy_((torch.randn(t.shape, generator=gen) * 0.5).to(t.dtype))
        g.replay()
        torch.cuda.synchronize()
        assert ops.mla_get_device_status() == ops.MLA_OK
        replayed = (bits(s.q_abs).copy(), bits(s.out).copy())
        assert not np.array_equal(replayed[1], eager)
        s.step()
        torch.cuda.synchronize()
        assert np.array_equal(bits(s.q_abs), replayed[0])
        assert np.array_equal(bits(s.out), replayed[1])
    finally:
        ops.mla_set_launch_overlap(before)


def test_launch_overlap_levels_give_identical_results():
    """Programmatic dependent launch only moves prologues (and, at level 2, the
    weight reads) ahead of the previous kernel's completion: same bits."""
    from mla_absorbed_decode_absorb_gb300 import ops
    inp = W.generate(W.custom("pdl", [5, 700, 4000], n_q=2), seed=8)
    before = ops.mla_get_launch_overlap()
    try:
        runs = []
        for level in (0, 1, 2):
            ops.mla_set_launch_overlap(level)
            assert ops.mla_get_launch_overlap() == level
            s = run_session(inp, split_pages=3)
            s.step()  # a second step: every launch now follows one of ours
            torch.cuda.synchronize()
            assert ops.mla_get_device_status() == ops.MLA_OK
            runs.append((bits(s.q_abs), bits(s.out), s.lse.cpu().numpy().view(np.uint32), bits(s.cache)))
        for r in runs[1:]:
            for x, y in zip(r, runs[0]):
                assert np.array_equal(x, y)
        with pytest.raises(ops.MLAError):
            ops.mla_set_launch_overlap(3)
    finally:
        ops.mla_set_launch_overlap(before)


# More shapes under the automatic plan: many short sequences, ragged lengths with
# two queries each, a uniform batch of page-aligned sequences.
SHAPES = {
    "many_short": W.custom("many_short", [0, 5, 63, 64, 70, 127, 128, 200] * 12, n_q=1),
    "ragged_q2": W.custom("ragged_q2", [3000, 40, 1000, 2500, 7, 4095] * 6, n_q=2),
    "uniform_aligned": W.custom("uniform_aligned", [2047] * 40, n_q=1),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_decode_parity_shapes(name):
    inp = W.generate(SHAPES[name], seed=9)
    s = run_session(inp, split_pages=0, fused_finish=False)
    check_outputs(s, inp, range(inp.batch), heads=[0, 63, 127])
    f = run_session(inp, split_pages=0, fused_finish=True)
    assert np.array_equal(bits(f.out), bits(s.out))


SHORT = {
    # at most two (sequence, query) units over at most 1024 tokens: a single token, a
    # page, a page and one, the 1024-token limit, two queries of one sequence, two
    # sequences of different lengths
    "short_kv1": W.custom("short_kv1", [0], n_q=1),
    "short_page": W.custom("short_page", [63], n_q=1),
    "short_page_plus1": W.custom("short_page_plus1", [64], n_q=1),
    "short_kv1024": W.custom("short_kv1024", [1023], n_q=1),
    "short_q2": W.custom("short_q2", [500], n_q=2),
    "short_b2": W.custom("short_b2", [10, 700], n_q=1),
}


@pytest.mark.parametrize("name", sorted(SHORT))
def test_short_context_path(name):
    """Short contexts with an automatic split run the short-context kernel (one CTA
    per 8 heads, no split): every head against the oracle, and close to the 2-CTA
    split kernel on the same inputs (forced by an explicit split; both round P to
    bf16 against their own running max, and the split kernel also exchanges fp16
    partial scores)."""
    from mla_absorbed_decode_absorb_gb300 import ops
    inp = W.generate(SHORT[name], seed=31)
    s = run_session(inp, split_pages=0, fused_finish=False)
    assert s.num_splits == 1 and ops.mla_decode_uses_short_path(s.B, s.n_q, s.max_kv_len, 0)
    o_err, lat_err = check_outputs(s, inp, range(inp.batch))
    t = run_session(inp, split_pages=1000, fused_finish=False)
    assert not ops.mla_decode_uses_short_path(t.B, t.n_q, t.max_kv_len, 1000)
    d = rel_l2(s.o_latent.cpu().numpy(), t.o_latent.cpu().numpy())
    print(f"{name}: rel-L2 O {o_err:.3e} O' {lat_err:.3e}; against the split kernel {d:.3e}")
    assert d < 3e-3


def test_split_count_invariance():
    """Split count changes only rounding: P is a bf16 MMA operand and each split
    rounds it against its own running max, so two split layouts differ by about
    two independent bf16 roundings of the weights (rms 2^-9/sqrt(3) each, about
    1.6e-3 relative in L2); a split's partial O' is stored in bf16 (one more such
    rounding, which a single split, writing O' in fp32, does not have), and the
    merge itself is exact up to fp32."""
    inp = W.generate(W.custom("splits", [700, 1000, 64], n_q=2), seed=4)
    ref = run_session(inp, split_pages=1000)
    assert ref.num_splits == 1
    for sp in [1, 2, 5]:
        s = run_session(inp, split_pages=sp, fused_finish=False)
        assert s.num_splits > 1
        assert rel_l2(s.o_latent.cpu().numpy(), ref.o_latent.cpu().numpy()) < 3e-3
        assert np.abs(s.lse.cpu().numpy() - ref.lse.cpu().numpy()).max() < 2e-3


def test_split_partials_in_the_workspace():
    """The split kernel leaves every split's partial in the workspace: O' over the
    split's visible tokens, normalised within the split, in bf16 at rows
    ((t * S + s) * 128 + h) of 512 (t = b * n_q + j), then the splits' log-sum-exps
    in float32; a split with no visible token has lse -inf and a zero row.  Each
    against the oracle's partial over the same token range (FlashMLA point 3 of
    "DeepSeek-MLA-Principle": per-block results merged by their log-sum-exps)."""
    inp = W.generate(W.custom("partials", [700, 130, 0], n_q=2), seed=12)
    s = run_session(inp, split_pages=3)  # the fused finish reads the partials, it does not move them
    S, B, n_q = s.num_splits, inp.batch, inp.n_q
    assert S == 4
    rows = B * n_q * S * 128
    ws = s.workspace.cpu()
    part = ws[:rows * 512 * 2].view(torch.bfloat16).float().numpy().reshape(B, n_q, S, 128, 512)
    lse = ws[rows * 512 * 2:rows * 512 * 2 + rows * 4].view(torch.float32).numpy().reshape(B, n_q, S, 128)
    span = 3 * 64
    w_uk = O.bf16_bits_to_f64(bits(inp.w_uk))
    w_uv = O.bf16_bits_to_f64(bits(inp.w_uv))
    seen_empty = seen_full = 0
    for b in range(B):
        c_bits, k_bits = (bits(x) for x in inp.sequence(b))
        c = O.bf16_bits_to_f64(c_bits)
        kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(c_bits.shape[0])))
        q_nope = O.bf16_bits_to_f64(bits(inp.q_nope[b]))
        q_rope = O.bf16_bits_to_f64(bits(inp.q_rope[b]))
        for sp in range(S):
            _, lat_ref, lse_ref = O.decode_absorbed(q_nope, q_rope, w_uk, w_uv, c, kr, int(inp.prior_lens[b]),
                                                    token_range=(sp * span, (sp + 1) * span))
            for j in range(n_q):
                if np.isneginf(lse_ref[j]).all():
                    assert np.isneginf(lse[b, j, sp]).all() and not part[b, j, sp].any(), (b, j, sp)
                    seen_empty += 1
                    continue
                assert np.abs(lse[b, j, sp] - lse_ref[j]).max() <= LSE_MAX_ABS, (b, j, sp)
                assert rel_l2(part[b, j, sp], lat_ref[j]) <= LAT_REL_L2, (b, j, sp, rel_l2(part[b, j, sp], lat_ref[j]))
                seen_full += 1
    assert seen_empty > 0 and seen_full > 0


def test_out_of_range_page_is_reported():
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession
    inp = W.generate(W.custom("bad", [100, 100], n_q=1), seed=5)
    s = DecodeSession(inp)
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    bad = s.page_table.clone()
    bad[1, 1] = inp.num_pages + 7   # past the pool
    s.page_table = bad
    s.step()
    assert ops.mla_get_device_status() == ops.MLA_ERR_BOUNDS
    assert ops.mla_get_device_status() == ops.MLA_OK  # read-and-clear
    s.page_table = inp.page_table.to(s.device)
    s.step()
    assert ops.mla_get_device_status() == ops.MLA_OK


def test_wait_timeout_is_reported_and_context_survives():
    """A bounded wait on a barrier nothing completes gives up, reports MLA_ERR_TIMEOUT
    through the status word, and later work on the same context is unaffected."""
    from mla_absorbed_decode_absorb_gb300 import ops
    import time
    assert ops.mla_get_device_status() == ops.MLA_OK
    t0 = time.perf_counter()
    assert ops.lib.mla_selftest_wait_timeout(20_000_000, 0) == ops.MLA_OK   # 20 ms
    torch.cuda.synchronize()
    assert 0.015 < time.perf_counter() - t0 < 1.0
    assert ops.mla_get_device_status() == ops.MLA_ERR_TIMEOUT
    assert ops.mla_get_device_status() == ops.MLA_OK  # read-and-clear
    assert ops.lib.mla_selftest_wait_timeout(0, 0) == ops.MLA_ERR_INVALID_ARG
    inp = W.generate(W.custom("after_timeout", [100, 64], n_q=1), seed=16)
    s = run_session(inp)  # asserts a clean status itself
    check_outputs(s, inp, range(inp.batch))


def test_invalid_arguments_raise():
    from mla_absorbed_decode_absorb_gb300 import ops
    x = torch.zeros(1, 1, 512, dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        ops.mla_append_kv(x, x, None, None, None, None)
    q = torch.zeros(1, 9, 128, 128, dtype=torch.bfloat16, device="cuda")
    r = torch.zeros(1, 9, 128, 64, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = torch.zeros(128, 128, 512, dtype=torch.bfloat16, device="cuda")
    rope = ops.rope_table(16)
    with pytest.raises(ops.MLAError):
        ops.mla_absorb_q(q, r, lens, w, rope)   # n_q = 9 > MLA_MAX_NQ


# ------------------------------------------------------------------------ full-size workloads
FULL = ["tiny_b1_l256", "batched_b32_l4096", "ragged_b128_l1024_8192", "long_b8_l32768", "mtp_b64_l8192_q4"]


def oracle_sequence_absorbed(inp: W.Inputs, b: int, w_uk, w_uv):
    """The oracle's absorbed fp64 form for sequence b, all heads (tied to the plain
    definition by the absorption-identity pins)."""
    c_bits, k_bits = (bits(x) for x in inp.sequence(b))
    kv = c_bits.shape[0]
    c = O.bf16_bits_to_f64(c_bits)
    kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(kv)))
    return O.decode_absorbed(O.bf16_bits_to_f64(bits(inp.q_nope[b])), O.bf16_bits_to_f64(bits(inp.q_rope[b])),
                             w_uk, w_uv, c, kr, int(inp.prior_lens[b]))


@pytest.mark.parametrize("name", FULL)
def test_full_workload_every_sequence_and_head(name):
    """The five benchmark workloads at full size, in the bench's launch configuration.

    Every sequence, query and head against the oracle's absorbed fp64 form (O, O'
    and lse; relative L2 per sequence as well as overall, so that one mis-gathered
    page in one sequence of many cannot hide in the aggregate); the plain
    non-absorbed definition on sampled sequences and heads; the cache rows of the
    sampled sequences bit for bit and this step's rows of every sequence.
    """
    wl = W.WORKLOADS[name]
    inp = W.generate(wl, seed=0)
    s = run_session(inp)
    if s.fused_finish and s.num_splits > 1:
        s.combine()
        torch.cuda.synchronize()
    o_gpu = s.out.float().cpu().numpy()
    lat_gpu = s.o_latent.cpu().numpy()
    lse_gpu = s.lse.cpu().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(lat_gpu).all() and np.isfinite(lse_gpu).all()
    w_uk, w_uv = O.bf16_bits_to_f64(bits(inp.w_uk)), O.bf16_bits_to_f64(bits(inp.w_uv))
    num = {"o": 0.0, "lat": 0.0}
    den = {"o": 0.0, "lat": 0.0}
    worst = {"o": 0.0, "lat": 0.0, "lse": 0.0, "o_abs": 0.0}
    for b in range(inp.batch):
        o_ref, lat_ref, lse_ref = oracle_sequence_absorbed(inp, b, w_uk, w_uv)
        for key, got, ref in (("o", o_gpu[b], o_ref), ("lat", lat_gpu[b], lat_ref)):
            d2, r2 = float(((got - ref) ** 2).sum()), float((ref ** 2).sum())
            num[key] += d2
            den[key] += r2
            worst[key] = max(worst[key], (d2 / r2) ** 0.5)
        worst["lse"] = max(worst["lse"], float(np.abs(lse_gpu[b] - lse_ref).max()))
        worst["o_abs"] = max(worst["o_abs"], float(np.abs(o_gpu[b] - o_ref).max()))
    print(f"{name}: rel-L2 O {(num['o'] / den['o']) ** 0.5:.3e} O' {(num['lat'] / den['lat']) ** 0.5:.3e}; "
          f"worst sequence O {worst['o']:.3e} O' {worst['lat']:.3e}; max |dlse| {worst['lse']:.3e}; "
          f"max |dO| {worst['o_abs']:.3e}")
    assert worst["o"] <= O_REL_L2 and worst["lat"] <= LAT_REL_L2, worst
    assert worst["lse"] <= LSE_MAX_ABS and worst["o_abs"] <= O_MAX_ABS, worst
    # the plain definition on a sample (first, middle, last sequence; three heads)
    seqs = sorted({0, inp.batch // 2, inp.batch - 1})
    check_outputs(s, inp, seqs, [0, 41, 127] if inp.batch > 1 else None)
    cache = s.cache
    pt = inp.page_table.numpy()
    for b in seqs:
        kv = int(inp.kv_lens[b])
        rows = bits(cache[torch.as_tensor(pt[b][np.arange(kv) // 64]).long().to(cache.device),
                          torch.as_tensor(np.arange(kv) % 64).to(cache.device)])
        c_bits, k_bits = (bits(x) for x in inp.sequence(b))
        assert np.array_equal(rows[:, :512], c_bits)
        assert np.array_equal(rows[:, 512:], O.rope_key_bf16_bits(k_bits, np.arange(kv)))
    # this step's new rows of every sequence
    c_new, k_new = inp.new_tokens()
    pos = inp.prior_lens.numpy()[:, None] + np.arange(inp.n_q)[None, :]
    pages = np.take_along_axis(pt, pos // 64, axis=1)
    rows = bits(cache[torch.as_tensor(pages).long().to(cache.device), torch.as_tensor(pos % 64).to(cache.device)])
    assert np.array_equal(rows[..., :512], bits(c_new))
    assert np.array_equal(rows[..., 512:].reshape(-1, 64),
                          O.rope_key_bf16_bits(bits(k_new).reshape(-1, 64), pos.reshape(-1)))
