"""Pins the CPU oracle to what the pages and the mathematics fix (no GPU).

Each check here is independent of the oracle's own formulas: closed forms,
textbook identities computed another way (RoPE as a complex rotation, the score
from explicit loops over eq. (2)), invariants, and numbers printed on the pages.
``test_planted_mistakes`` runs the same checks against deliberately broken
copies of oracle functions to show that each kind of slip is caught.
"""

import cmath
import json
import math
import os

import numpy as np
import torch

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(rng, n_h=2, d_h=4, d_c=8, d_r=4, kv=5, n_q=1):
    return dict(
        q_nope=rng.normal(size=(n_q, n_h, d_h)), q_rope=rng.normal(size=(n_q, n_h, d_r)),
        w_uk=rng.normal(size=(n_h, d_h, d_c)), w_uv=rng.normal(size=(n_h, d_h, d_c)),
        c=rng.normal(size=(kv, d_c)), kr=rng.normal(size=(kv, d_r)))


def relerr(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ----------------------------------------------------------------- independent references
def rope_complex(x, pos):
    """Half-split RoPE written as rotation of z_i = x_i + i x_{i+half} by pos*theta_i."""
    half = len(x) // 2
    out = [0.0] * len(x)
    for i in range(half):
        theta_i = math.exp(-math.log(10000.0) * i / half)
        z = complex(x[i], x[i + half]) * cmath.exp(1j * pos * theta_i)
        out[i], out[i + half] = z.real, z.imag
    return out


def score_loops(q_nope_h, q_rope_h, w_uk_h, c_t, kr_t, pos):
    """q.k / sqrt(d_h + d_R) with k^C_i = sum_m W_UK[h][i][m] c_m (eq. (2)), by loops."""
    d_h, d_c = len(w_uk_h), len(w_uk_h[0])
    kc = [sum(w_uk_h[i][m] * c_t[m] for m in range(d_c)) for i in range(d_h)]
    qr = rope_complex(list(q_rope_h), pos)
    dot = sum(q_nope_h[i] * kc[i] for i in range(d_h)) + sum(qr[i] * kr_t[i] for i in range(len(qr)))
    return dot / math.sqrt(d_h + len(qr))


def value_loops(w_uv_h, c_t):
    return [sum(w_uv_h[i][m] * c_t[m] for m in range(len(c_t))) for i in range(len(w_uv_h))]


# ----------------------------------------------------------------- check functions
def check_rope_unit_vectors(rope=O.rope_f64):
    """e_i rotated at position p has components (cos p*theta_i, sin p*theta_i) in (i, i+32)."""
    for i, p in [(0, 1), (0, 7), (16, 100), (31, 12345)]:
        theta = 10000.0 ** (-i / 32)
        e = np.zeros(64)
        e[i] = 1.0
        r = rope(e, p)
        want = np.zeros(64)
        want[i], want[i + 32] = math.cos(p * theta), math.sin(p * theta)
        if not np.allclose(r, want, atol=1e-12):
            return False
        e = np.zeros(64)
        e[i + 32] = 1.0
        r = rope(e, p)
        want = np.zeros(64)
        want[i], want[i + 32] = -math.sin(p * theta), math.cos(p * theta)
        if not np.allclose(r, want, atol=1e-12):
            return False
    return True


def check_two_tokens(decode=O.decode_mha, seed=3):
    """kv = 2: alpha_0 = sigmoid(s_0 - s_1), o = alpha_0 v_0 + (1 - alpha_0) v_1."""
    rng = np.random.default_rng(seed)
    p = tiny(rng, kv=2)
    o, o_lat, lse = decode(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=1)
    for h in range(2):
        s = [score_loops(p["q_nope"][0, h], p["q_rope"][0, h], p["w_uk"][h], p["c"][t], p["kr"][t], 1)
             for t in range(2)]
        a0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        v = [value_loops(p["w_uv"][h], p["c"][t]) for t in range(2)]
        want_o = [a0 * v[0][i] + (1 - a0) * v[1][i] for i in range(len(v[0]))]
        want_lat = a0 * p["c"][0] + (1 - a0) * p["c"][1]
        want_lse = max(s) + math.log(math.exp(s[0] - max(s)) + math.exp(s[1] - max(s)))
        if not (np.allclose(o[0, h], want_o, rtol=1e-12, atol=1e-12)
                and np.allclose(o_lat[0, h], want_lat, rtol=1e-12, atol=1e-12)
                and abs(lse[0, h] - want_lse) < 1e-12):
            return False
    return True


def check_absorbed_identity(mha=O.decode_mha, absorbed=O.decode_absorbed, seed=1):
    rng = np.random.default_rng(seed)
    for kv, n_q in [(1, 1), (2, 1), (5, 1), (3, 2), (5, 3)]:
        p = tiny(rng, kv=kv, n_q=n_q)
        a = mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=kv - n_q)
        b = absorbed(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=kv - n_q)
        for x, y in zip(a, b):
            if relerr(x, y) > 1e-10:
                return False
    return True


# ----------------------------------------------------------------- tests
def test_rope_closed_form_unit_vectors():
    assert check_rope_unit_vectors()


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(0)
    for pos in [0, 1, 3, 4096, 32768]:
        x = rng.normal(size=64)
        assert np.allclose(O.rope_f64(x, pos), rope_complex(list(x), pos), atol=1e-12)


def test_rope_is_rotation():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(10, 64))
    pos = np.arange(10) * 977
    r = O.rope_f64(x, pos)
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.array_equal(O.rope_f64(x, np.zeros(10, dtype=int)), x)


def test_rope_relative_position():
    """<R_i q, R_j k> = <q, R_{j-i} k>."""
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=64), rng.normal(size=64)
    for i, j in [(0, 5), (5, 0), (100, 4196), (4096, 4097), (30000, 2)]:
        lhs = O.rope_f64(q, i) @ O.rope_f64(k, j)
        rhs = q @ O.rope_f64(k, j - i)
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_absorbed_equals_non_absorbed_tiny():
    assert check_absorbed_identity()


def test_absorbed_equals_non_absorbed_full_dims():
    rng = np.random.default_rng(4)
    n_h, kv, n_q = 128, 8, 2
    q_nope = rng.normal(size=(n_q, n_h, 128))
    q_rope = rng.normal(size=(n_q, n_h, 64))
    w_uk = rng.normal(scale=0.02, size=(n_h, 128, 512))
    w_uv = rng.normal(scale=0.02, size=(n_h, 128, 512))
    c, kr = rng.normal(size=(kv, 512)), rng.normal(size=(kv, 64))
    heads = [0, 77, 127]
    a = O.decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, kv - n_q, heads)
    b = O.decode_absorbed(q_nope, q_rope, w_uk, w_uv, c, kr, kv - n_q, heads)
    for x, y in zip(a, b):
        assert relerr(x, y) <= 1e-10


def test_decompressed_keys_obey_the_absorption_identity():
    """q^C . K[t, h] = (W_UK[h]^T q^C) . c_t (the absorbed query of absorb_query, a
    separate code path), and V[t, h] . u = c_t . (W_UV[h]^T u), for every t and h."""
    rng = np.random.default_rng(12)
    n_h, kv = 4, 9
    w_uk = rng.normal(scale=0.02, size=(n_h, 128, 512))
    w_uv = rng.normal(scale=0.02, size=(n_h, 128, 512))
    c = rng.normal(size=(kv, 512))
    q_nope = rng.normal(size=(n_h, 128))
    q_rope = rng.normal(size=(n_h, 64))
    k, v = O.decompress_kv(c, w_uk, w_uv)
    assert k.shape == (kv, n_h, 128) and v.shape == (kv, n_h, 128)
    q_abs = O.absorb_query(q_nope[None], q_rope[None], w_uk, np.array([3]))[0]   # [n_h, 576]
    lhs = np.einsum("thd,hd->th", k, q_nope)
    rhs = c @ q_abs[:, :512].T
    assert relerr(lhs, rhs) <= 1e-12
    u = rng.normal(size=(n_h, 128))
    lhs_v = np.einsum("thd,hd->th", v, u)
    rhs_v = np.stack([c @ (w_uv[h].T @ u[h]) for h in range(n_h)], axis=1)
    assert relerr(lhs_v, rhs_v) <= 1e-12
    # the decompressed keys and values give decode_mha's result for a many-query chunk
    kr = rng.normal(size=(kv, 64))
    qn = rng.normal(size=(5, n_h, 128))
    qr = rng.normal(size=(5, n_h, 64))
    o, _, lse = O.decode_mha(qn, qr, w_uk, w_uv, c, kr, prior_len=kv - 5)
    for j in range(5):
        pos = kv - 5 + j
        for h in range(n_h):
            q = np.concatenate([qn[j, h], O.rope_f64(qr[j, h], pos)])
            keys = np.concatenate([k[:pos + 1, h], kr[:pos + 1]], axis=1)
            sc = keys @ q / np.sqrt(192.0)
            a = np.exp(sc - sc.max())
            assert relerr(o[j, h], (a / a.sum()) @ v[:pos + 1, h]) <= 1e-12
            assert abs(lse[j, h] - (sc.max() + np.log(a.sum()))) <= 1e-12


def check_softmax_weights(decode=O.decode_mha, seed=5):
    """decode_mha's own weights, read out through its latent output: with one-hot
    latent rows c_t = e_t, O' = sum_t alpha_t e_t is the weight vector itself.  Each
    row must be >= 0, sum to 1, vanish past the query's position, and equal the
    softmax of the scores computed by explicit loops over eq. (2)."""
    rng = np.random.default_rng(seed)
    kv, n_q, d_c = 7, 7, 8
    p = tiny(rng, kv=kv, n_q=n_q, d_c=d_c)
    p["c"] = np.eye(kv, d_c)
    _, o_lat, _ = decode(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=0)
    for j in range(n_q):          # query j sits at position j and sees tokens 0..j
        for h in range(2):
            a = o_lat[j, h]
            if (a < 0).any() or abs(a.sum() - 1.0) > 1e-14 or np.abs(a[j + 1:]).max(initial=0.0) != 0.0:
                return False
            s = [score_loops(p["q_nope"][j, h], p["q_rope"][j, h], p["w_uk"][h], p["c"][t], p["kr"][t], j)
                 for t in range(j + 1)]
            e = [math.exp(x - max(s)) for x in s]
            if not np.allclose(a[:j + 1], [x / sum(e) for x in e], rtol=1e-12, atol=1e-15):
                return False
    return True


def test_softmax_rows_sum_to_one():
    assert check_softmax_weights()


def check_out_absorb(out_absorb=O.out_absorb, seed=21):
    """O[..., h, d] = sum_m O'[..., h, m] W_UV[h, d, m] ([N1] final einsum 'bhm,hdm->bhd')
    by explicit loops, on a non-square case with leading batch/query axes."""
    rng = np.random.default_rng(seed)
    B, n_q, n_h, d_v, d_c = 2, 3, 3, 5, 7
    o_lat = rng.normal(size=(B, n_q, n_h, d_c))
    w_uv = rng.normal(size=(n_h, d_v, d_c))
    got = out_absorb(o_lat, w_uv)
    if got.shape != (B, n_q, n_h, d_v):
        return False
    for b in range(B):
        for j in range(n_q):
            for h in range(n_h):
                want = value_loops(w_uv[h], o_lat[b, j, h])
                if not np.allclose(got[b, j, h], want, rtol=1e-13, atol=1e-13):
                    return False
    return True


def test_out_absorb_matches_explicit_loops():
    assert check_out_absorb()


def test_out_absorb_of_the_latent_output_is_the_output():
    """Value absorption ([DP] "3) MLA 中怎么吸收"): W_UV applied to O' = sum alpha c gives
    decode_mha's non-absorbed O = sum alpha W_UV c."""
    rng = np.random.default_rng(22)
    p = tiny(rng, kv=6, n_q=3, d_h=5, d_c=9)
    o, o_lat, _ = O.decode_mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=3)
    assert relerr(O.out_absorb(o_lat, p["w_uv"]), o) <= 1e-12


def check_absorb_query(absorb=O.absorb_query, seed=23):
    """The absorbed query of every token of a multi-token, multi-sequence step:
    latent half q~[m] = sum_d q^C[d] W_UK[h, d, m] by loops ([N1] 'bhd,hdm->bhm'),
    position half RoPE(q^R) at position L_b + j as a complex rotation ([DP] eq. (8))."""
    rng = np.random.default_rng(seed)
    B, n_q, n_h, d_h, d_c, d_r = 3, 4, 2, 3, 5, 8
    q_nope = rng.normal(size=(B, n_q, n_h, d_h))
    q_rope = rng.normal(size=(B, n_q, n_h, d_r))
    w_uk = rng.normal(size=(n_h, d_h, d_c))
    prior = np.array([0, 17, 4093])
    pos = prior[:, None] + np.arange(n_q)[None, :]
    got = absorb(q_nope, q_rope, w_uk, pos)
    if got.shape != (B, n_q, n_h, d_c + d_r):
        return False
    for b in range(B):
        for j in range(n_q):
            for h in range(n_h):
                lat = [sum(q_nope[b, j, h, d] * w_uk[h, d, m] for d in range(d_h)) for m in range(d_c)]
                rot = rope_complex(list(q_rope[b, j, h]), int(pos[b, j]))
                if not (np.allclose(got[b, j, h, :d_c], lat, rtol=1e-13, atol=1e-13)
                        and np.allclose(got[b, j, h, d_c:], rot, rtol=1e-12, atol=1e-12)):
                    return False
    return True


def test_absorb_query_latent_and_rope_halves():
    assert check_absorb_query()


def test_one_token_closed_form():
    """kv = 1: alpha = 1, O' = c_0 exactly, O = W_UV c_0, lse = s_0."""
    rng = np.random.default_rng(6)
    p = tiny(rng, kv=1)
    o, o_lat, lse = O.decode_mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=0)
    for h in range(2):
        assert np.array_equal(o_lat[0, h], p["c"][0])
        assert np.allclose(o[0, h], value_loops(p["w_uv"][h], p["c"][0]), rtol=1e-13, atol=1e-13)
        s0 = score_loops(p["q_nope"][0, h], p["q_rope"][0, h], p["w_uk"][h], p["c"][0], p["kr"][0], 0)
        assert abs(lse[0, h] - s0) < 1e-12


def test_two_token_closed_form():
    assert check_two_tokens()


def test_constant_cache_gives_the_constant():
    rng = np.random.default_rng(7)
    p = tiny(rng, kv=6)
    p["c"][:] = p["c"][0]
    o, o_lat, _ = O.decode_mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], prior_len=5)
    for h in range(2):
        assert np.allclose(o_lat[0, h], p["c"][0], rtol=1e-14, atol=1e-14)
        assert np.allclose(o[0, h], value_loops(p["w_uv"][h], p["c"][0]), rtol=1e-12, atol=1e-12)


def test_score_splits_into_content_and_rope():
    """The 192-wide dot equals content (q~ . c) plus rope (q^R . k^R) terms."""
    rng = np.random.default_rng(8)
    p = tiny(rng, kv=1)
    qr = O.rope_f64(p["q_rope"][0, 0], 0)
    full = np.concatenate([p["q_nope"][0, 0], qr]) @ np.concatenate([p["w_uk"][0] @ p["c"][0], p["kr"][0]])
    q_t = p["w_uk"][0].T @ p["q_nope"][0, 0]
    assert abs(full - (q_t @ p["c"][0] + qr @ p["kr"][0])) < 1e-12


def test_split_combine_invariance():
    rng = np.random.default_rng(9)
    kv, n_q = 23, 3
    p = tiny(rng, kv=kv, n_q=n_q)
    args = (p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], kv - n_q)
    full = O.decode_mha(*args)
    for cuts in [(0, 23), (0, 7, 23), (0, 5, 11, 20, 21, 23), (0, 21, 22, 23)]:
        parts = [O.decode_absorbed(*args, token_range=(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
        o_lat, lse = O.combine_splits([x[1] for x in parts], [x[2] for x in parts])
        assert relerr(o_lat, full[1]) <= 1e-12
        assert np.abs(lse - full[2]).max() <= 1e-12


def test_causal_among_new_tokens():
    """Query j sees tokens 0..L+j: changing token L+1 moves queries j >= 1 only."""
    rng = np.random.default_rng(10)
    kv, n_q = 9, 3
    p = tiny(rng, kv=kv, n_q=n_q)
    L = kv - n_q
    a = O.decode_mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], L)
    c2, kr2 = p["c"].copy(), p["kr"].copy()
    c2[L + 1] += 1.0
    kr2[L + 1] -= 1.0
    b = O.decode_mha(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], c2, kr2, L)
    assert np.array_equal(a[0][0], b[0][0]) and np.array_equal(a[1][0], b[1][0])
    assert not np.allclose(a[0][1], b[0][1]) and not np.allclose(a[0][2], b[0][2])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    x = rng.normal(size=4096).astype(np.float32) * np.float32(3.0)
    # exact ties: a bf16 value plus half an ulp, both parities of the kept bit
    base = (rng.integers(0, 2**15, size=512).astype(np.uint32) << 16)
    ties = (base | np.uint32(0x8000)).view(np.float32)
    ties = ties[np.isfinite(ties)]  # NaN payloads are not part of the recipe
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1e-40, 3.4e38, -3.4e38, np.inf, -np.inf])])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), want)


def test_rope_table_is_float32_of_libm():
    cos, sin = O.rope_table_f32(4096)
    pos = np.arange(4096)[:, None]
    ang = pos * O.rope_inv_freq(64)
    for exact, got in [(np.cos(ang), cos), (np.sin(ang), sin)]:
        ulp = np.spacing(np.abs(exact).astype(np.float32))
        assert (np.abs(got.astype(np.float64) - exact) <= ulp).all()


def test_rope_key_bits_within_one_bf16_ulp():
    rng = np.random.default_rng(12)
    k = torch.randn(2000, 64, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    bits = k.view(torch.int16).numpy().view(np.uint16)
    pos = rng.integers(0, 40000, size=2000)
    got = O.bf16_bits_to_f64(O.rope_key_bf16_bits(bits, pos))
    exact = O.rope_f64(O.bf16_bits_to_f64(bits), pos)
    ulp = np.abs(exact) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - exact) <= ulp).all()


def test_append_layout():
    rng = np.random.default_rng(13)
    P, B, n_new = 7, 2, 3
    sentinel = np.uint16(0x7FC0)
    cache = np.full((P, 64, 576), sentinel, dtype=np.uint16)
    pt = np.array([[5, 2, -1], [0, 6, 3]], dtype=np.int32)
    lens = np.array([62, 127])
    c_new = rng.integers(0, 0x7F00, size=(B, n_new, 512)).astype(np.uint16)
    k_new = torch.randn(B, n_new, 64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = O.append_kv(cache, c_new, k_new, lens, pt)
    placed = {(5, 62): (0, 0), (5, 63): (0, 1), (2, 0): (0, 2), (6, 63): (1, 0), (3, 0): (1, 1), (3, 1): (1, 2)}
    for (page, slot), (b, j) in placed.items():
        assert np.array_equal(out[page, slot, :512], c_new[b, j])
        rot = O.rope_key_bf16_bits(k_new[b, j][None], np.array([lens[b] + j]))[0]
        assert np.array_equal(out[page, slot, 512:], rot)
    mask = np.ones((P, 64), bool)
    for page, slot in placed:
        mask[page, slot] = False
    assert (out[mask] == sentinel).all()
    c, kr = O.gather_sequence(out, pt[1], 130)
    assert np.array_equal(c[127], O.bf16_bits_to_f64(c_new[1, 0]))


def test_pages_numbers():
    from mla_absorbed_decode_absorb_gb300 import accounting as A
    from mla_absorbed_decode_absorb_gb300 import workloads as W
    g = json.load(open(os.path.join(GOLDEN, "pages_numbers.json")))
    d = g["dims"]["value"]
    assert (W.N_HEADS, W.D_NOPE, W.D_ROPE, W.D_LATENT) == (d["n_h"], d["d_h"], d["d_h_rope"], d["d_c"])
    assert W.D_NOPE + W.D_ROPE == g["score_scale_dim"]["value"]
    assert W.PAGE == g["page_size"]["value"]
    assert A.cache_scalars_per_token() == g["cache_scalars_per_token"]["value"]
    assert A.mha_cache_scalars_per_token() == g["mha_cache_scalars_per_token"]["value"]
    ratio = A.mha_cache_scalars_per_token() / A.cache_scalars_per_token()
    assert abs(ratio - g["compression_ratio"]["value"]) <= g["compression_ratio"]["abs_tol"]
    assert 4096 * A.cache_bytes_per_token(2) == g["mla_step_read_bytes_L4096_fp16"]["value"]
    assert A.step_cache_bytes([4096]) == g["mla_step_read_bytes_L4096_fp16"]["value"]
    assert 4096 * A.mha_cache_scalars_per_token() * 2 == g["mha_step_read_bytes_L4096_fp16"]["value"]
    for key, fn in [("mla_history_multiplies_L4096", A.mla_history_macs),
                    ("mha_history_multiplies_L4096", A.mha_history_macs)]:
        v = g[key]["value"]
        assert abs(fn(4096) - v) <= g[key]["rel_tol"] * v
    assert 4096 * W.N_HEADS * W.D_NOPE * 2 == g["non_absorbed_kv_elements_L4096"]["value"]
    # one query against kv tokens: 2 FLOP per MAC of the history interaction
    assert A.step_attention_flops([4097], 1) == 2 * A.mla_history_macs(4097)


# ----------------------------------------------------------------- planted mistakes
def _rope_wrong_sign(x, pos):
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    ang = np.asarray(pos, np.float64)[..., None] * O.rope_inv_freq(2 * h)
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[..., :h] * c + x[..., h:] * s, x[..., h:] * c - x[..., :h] * s], -1)


def _rope_wrong_freq(x, pos):
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    ang = np.asarray(pos, np.float64)[..., None] * (10000.0 ** (-np.arange(h) / (2 * h)))
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[..., :h] * c - x[..., h:] * s, x[..., h:] * c + x[..., :h] * s], -1)


def test_planted_mistakes(monkeypatch):
    # wrong rotation direction / frequency: the unit-vector closed form catches it
    assert not check_rope_unit_vectors(_rope_wrong_sign)
    assert not check_rope_unit_vectors(_rope_wrong_freq)

    # wrong sign inside the oracle's RoPE: the 2-token closed form catches it
    monkeypatch.setattr(O, "rope_f64", _rope_wrong_sign)
    assert not check_two_tokens()
    monkeypatch.undo()

    # wrong scale (1/sqrt(d_h) instead of 1/sqrt(d_h + d_R))
    real_sqrt = math.sqrt

    class _M:
        def __getattr__(self, k):
            return getattr(math, k)

        @staticmethod
        def sqrt(x):
            return real_sqrt(x - 4)  # d_R = 4 in the tiny problem
    monkeypatch.setattr(O, "math", _M())
    assert not check_two_tokens()
    monkeypatch.undo()

    # transposed up-projection operand (square tiny dims so shapes still fit)
    def mha_transposed(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len, heads=None):
        return O.decode_mha(q_nope, q_rope, np.swapaxes(w_uk, 1, 2), w_uv, c, kr, prior_len, heads)

    def tiny_square(rng, **kw):
        return tiny(rng, n_h=2, d_h=8, d_c=8, d_r=4, **kw)
    rng = np.random.default_rng(1)
    p = tiny_square(rng, kv=4)
    a = mha_transposed(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], 3)
    b = O.decode_absorbed(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["c"], p["kr"], 3)
    assert relerr(a[0], b[0]) > 1e-6

    # a dropped RoPE term (score without the position part)
    def mha_no_rope(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len, heads=None):
        return O.decode_mha(q_nope, q_rope, w_uk, w_uv, c, np.zeros_like(kr), prior_len, heads)
    assert not check_two_tokens(decode=mha_no_rope)
    assert not check_absorbed_identity(mha=mha_no_rope)

    # the softmax weights: a wrong scale or a dropped RoPE term moves them off the loop scores
    assert not check_softmax_weights(decode=mha_no_rope)

    # out_absorb: the wrong head's weights, or W_UV's output and latent axes swapped on a square slice
    assert not check_out_absorb(lambda o, w: O.out_absorb(o, np.roll(w, 1, axis=0)))
    assert not check_out_absorb(lambda o, w: np.einsum("...hm,hmd->...hd", o[..., :5],
                                                       np.asarray(w)[:, :, :5]))

    # absorb_query: RoPE at position pos - 1, no RoPE at all, or W_UK's rows for the wrong head
    assert not check_absorb_query(lambda qn, qr, w, pos: O.absorb_query(qn, qr, w, np.asarray(pos) - 1))
    assert not check_absorb_query(lambda qn, qr, w, pos: O.absorb_query(qn, qr, w, np.zeros_like(pos)))
    assert not check_absorb_query(lambda qn, qr, w, pos: O.absorb_query(qn, qr, np.roll(w, 1, axis=0), pos))

    # a causal off-by-one (query sees one token too few)
    def mha_off_by_one(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len, heads=None):
        return O.decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len - 1, heads)
    assert not check_two_tokens(decode=mha_off_by_one)


# ------------------------------------------------------------------------ FP8 latent cache
def test_e4m3_decode_follows_the_format():
    """Values of E4M3 codes from the format's definition (bias 7, 3 mantissa bits,
    subnormals, no infinities, S.1111.111 NaN), cross-checked with torch's float8_e4m3fn."""
    codes = np.arange(256, dtype=np.uint8)
    v = O.e4m3_decode(codes)
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0x7E] == 448.0
    assert v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9 and v[0x01] == 2.0 ** -9
    assert v[0xB8] == -1.0 and v[0xFE] == -448.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isnan(v).sum() == 2
    assert np.all(np.diff(v[:0x7F]) > 0)           # codes 0x00 .. 0x7E are in increasing order
    t = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(v), np.isnan(t))
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])


def test_e4m3_encode_rounds_to_nearest_even_and_saturates():
    cases = [(1.0625, 0x38), (1.1875, 0x3A), (1.0626, 0x39), (448.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E),
             (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (2.0 ** -9, 0x01), (-1.0, 0xB8), (-1e6, 0xFE),
             (0.0, 0x00), (-0.0, 0x80), (240.0, 0x77), (248.0, 0x78)]
    x = np.array([v for v, _ in cases], dtype=np.float32)
    assert O.f32_to_e4m3_codes(x).tolist() == [c for _, c in cases]
    assert O.f32_to_e4m3_codes(np.array([np.nan], np.float32))[0] == 0x7F
    finite = np.arange(0x7F, dtype=np.uint8)        # every finite code round-trips, both signs
    assert np.array_equal(O.f32_to_e4m3_codes(O.e4m3_decode(finite).astype(np.float32)), finite)
    neg = (finite | 0x80).astype(np.uint8)
    assert np.array_equal(O.f32_to_e4m3_codes(O.e4m3_decode(neg).astype(np.float32)), neg)
    rng = np.random.default_rng(11)
    y = (rng.standard_normal(50000) * np.exp2(rng.integers(-12, 9, 50000))).astype(np.float32)
    y = np.clip(y, -448, 448).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.f32_to_e4m3_codes(y), ref)


def _fp8_images(P):
    return (np.full((P, 64, 512), 0x7F, np.uint8), np.full((P, 64), np.nan, np.float32),
            np.full((P, 64, 64), 0x7E00, np.uint16))


def test_fp8_append_stores_within_the_format_bounds():
    """Placement as the bf16 append; the scale is max(amax / 448, 2^-10); the largest
    latent value maps to +-448 exactly; every dequantised value is within half an E4M3
    step; the stored key gives back k^R within half an f16 step; other slots untouched."""
    rng = np.random.default_rng(12)
    B, n, P = 4, 3, 12
    c = rng.standard_normal((B, n, 512)).astype(np.float32)
    c[1, 0] = 0.0                     # an all-zero latent: the scale floor
    c[2, 1] *= 1e-4                   # tiny latent: the floor again, codes below 448
    c[3, 2] *= 300.0                  # large latent
    c_bits = O.f32_to_bf16_bits(c)
    k_bits = O.f32_to_bf16_bits(rng.standard_normal((B, n, 64)).astype(np.float32))
    lens = np.array([0, 62, 64, 125])
    pt = rng.permutation(P).reshape(B, 3)
    c8, sc, kr = O.append_kv_fp8(*_fp8_images(P), c_bits, k_bits, lens, pt)
    cv = O.bf16_bits_to_f64(c_bits)
    written = np.zeros((P, 64), bool)
    for b in range(B):
        for j in range(n):
            pos = lens[b] + j
            pg, sl = pt[b, pos // 64], pos % 64
            written[pg, sl] = True
            amax = np.abs(cv[b, j]).max()
            s = np.float32(max(np.float32(amax) / np.float32(448.0), np.float32(2.0 ** -10)))
            assert sc[pg, sl] == s
            deq = float(s) * O.e4m3_decode(c8[pg, sl])
            step = np.where(np.abs(cv[b, j]) / s >= 2.0 ** -6, np.abs(cv[b, j]) * 2.0 ** -4, float(s) * 2.0 ** -10)
            assert np.all(np.abs(deq - cv[b, j]) <= step * (1 + 1e-6))
            if amax / 448 >= 2.0 ** -10:
                assert np.abs(O.e4m3_decode(c8[pg, sl])).max() == 448.0
            r = O.rope_key_f32(k_bits[b, j][None], np.array([pos]))[0].astype(np.float64)
            kd = float(s) * kr[pg, sl].view(np.float16).astype(np.float64)
            assert np.all(np.abs(kd - r) <= np.abs(r) * 2.0 ** -11 * (1 + 1e-6) + float(s) * 2.0 ** -25)
    assert np.all(c8[~written] == 0x7F) and np.all(np.isnan(sc[~written])) and np.all(kr[~written] == 0x7E00)
    assert sc[pt[1, 0], 62] == np.float32(2.0 ** -10) and np.all(c8[pt[1, 0], 62] == 0)


def test_fp8_cache_attention_stays_near_the_bf16_result():
    """The definition on the dequantised FP8 cache against the same on the bf16 cache:
    the latent output moves by the quantisation error (about 2^-5 relative per value,
    averaged over the attended tokens), the log-sum-exp by a few hundredths."""
    rng = np.random.default_rng(13)
    H, kv = 4, 200
    c = rng.standard_normal((kv, 512)).astype(np.float32)
    k_pe = rng.standard_normal((kv, 64)).astype(np.float32)
    c_bits, k_bits = O.f32_to_bf16_bits(c), O.f32_to_bf16_bits(k_pe)
    pt = np.arange(4)[None]
    c8, sc, kr = O.append_kv_fp8(*_fp8_images(4), c_bits[None], k_bits[None], [0], pt)
    cq, kq = O.gather_sequence_fp8(c8, sc, kr, pt[0], kv)
    cb = O.bf16_bits_to_f64(c_bits)
    kb = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(kv)))
    q_nope = rng.standard_normal((1, H, 128))
    q_rope = rng.standard_normal((1, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) * 0.02
    w_uv = rng.standard_normal((H, 128, 512)) * 0.02
    o8, lat8, lse8 = O.decode_mha(q_nope, q_rope, w_uk, w_uv, cq, kq, kv - 1)
    ob, latb, lseb = O.decode_mha(q_nope, q_rope, w_uk, w_uv, cb, kb, kv - 1)
    rel = np.linalg.norm(lat8 - latb) / np.linalg.norm(latb)
    assert 1e-4 < rel < 4e-2, rel
    assert np.abs(lse8 - lseb).max() < 5e-2


# ------------------------------------------------------------------------ decode layer
def test_linear_is_x_times_w_transposed():
    """y[t, n] = sum_k x[t, k] w[n, k] by explicit loops on a non-square case."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((3, 5))
    w = rng.standard_normal((4, 5))
    ref = np.array([[sum(x[t, k] * w[n, k] for k in range(5)) for n in range(4)] for t in range(3)])
    assert np.allclose(O.linear(x, w), ref, rtol=1e-14, atol=1e-14)


def test_decode_layer_single_token_closed_form():
    """A first token attends only to itself (alpha = 1), so the per-head output is
    W_UV[h] c with c = W_DKV x, and the layer output is its concatenation times W_O^T,
    whatever the query side."""
    rng = np.random.default_rng(22)
    d, dc, dr, dq, H, dh = 16, 8, 4, 6, 2, 4
    x = rng.standard_normal((1, d))
    w_dkv, w_kr, w_dq = rng.standard_normal((dc, d)), rng.standard_normal((dr, d)), rng.standard_normal((dq, d))
    w_uq, w_qr = rng.standard_normal((H * dh, dq)), rng.standard_normal((H * dr, dq))
    w_uk, w_uv = rng.standard_normal((H, dh, dc)), rng.standard_normal((H, dh, dc))
    w_o = rng.standard_normal((d, H * dh))
    y, o = O.decode_layer(x, w_dkv, w_kr, w_dq, w_uq, w_qr, w_uk, w_uv, w_o, np.zeros((0, dc)), np.zeros((0, dr)), 0,
                          cache_bf16_rows=False)
    c = w_dkv @ x[0]
    o_ref = np.stack([w_uv[h] @ c for h in range(H)])
    assert np.allclose(o[0], o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(y[0], w_o @ o_ref.reshape(-1), rtol=1e-12, atol=1e-12)
    # the query side matters once there are two tokens: changing W_UQ changes the output
    hist_c, hist_k = rng.standard_normal((1, dc)), rng.standard_normal((1, dr))
    y1, _ = O.decode_layer(x, w_dkv, w_kr, w_dq, w_uq, w_qr, w_uk, w_uv, w_o, hist_c, hist_k, 1, cache_bf16_rows=False)
    y2, _ = O.decode_layer(x, w_dkv, w_kr, w_dq, 2 * w_uq, w_qr, w_uk, w_uv, w_o, hist_c, hist_k, 1,
                           cache_bf16_rows=False)
    assert np.abs(y1 - y2).max() > 1e-6
