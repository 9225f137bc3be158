"""CPU oracle for absorbed MLA decode.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path and
imports nothing from it; both sides only consume the same seeded inputs.

Sources (three web pages on MLA weight absorption):

* [MA]  "MLA 矩阵吸收 & 吸收分离 原理详解" (chang-wenbin.github.io, MLA_Matrix_Absorption)
* [DP]  "DeepSeek-MLA-Principle" (senjlearning.space)
* [N1]  "DeepSeek MLA 架构详解：多头潜向量注意力如何将 KV Cache 降低 93%" (explore.n1n.ai)

What it computes: the plain, *non-absorbed* definition of one MLA decode step
([DP] §2 "注意力计算", equations (2)/(5), (4), (9), the scaled score, the softmax
and (10)): per head, decompress ``k_t = [W_UK[h] c_t ; k^R_t]`` and
``v_t = W_UV[h] c_t`` for every visible cached token, score with the 192-wide
query ``[q^C ; RoPE(q^R)]`` scaled by ``1/sqrt(d_h + d_h^R)``, softmax over the
visible tokens, and sum the values.  It also returns the latent output
``O' = sum_t alpha_t c_t`` and the log-sum-exp of the scores, which the absorbed
path produces along the way.  Everything is float64 on values read back from
the bf16 cache image that :func:`append_kv` builds.

The absorbed fp64 form ([DP] "3) MLA 中怎么吸收", key and value absorption;
[MA] §2.1, §4.1) is here only to cross-check the identity.

Readings where the pages leave a step open (each listed in the design notes):

* the tokens appended this step are attended to: query ``j`` of a sequence with
  ``L`` prior tokens sits at position ``L + j`` and sees tokens ``0 .. L + j``;
* RoPE is the half-split ("rotate half") form of [N1] ``apply_rope``:
  ``inv_freq_i = theta^(-i/half)``, ``theta = 10000``, ``half = d_R / 2``,
  ``out[i] = x[i] cos - x[i+half] sin``, ``out[i+half] = x[i+half] cos + x[i] sin``;
* the cache holds the rotated key ``k^R`` in bf16 ([N1] rotates before the append);
  its exact bf16 bits follow a fixed fp32 recipe (:func:`rope_key_bf16_bits`).
"""

from __future__ import annotations

import math
from functools import lru_cache

import numpy as np

THETA = 10000.0
PAGE = 64


# --------------------------------------------------------------------------- bf16
def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 to bf16, round-to-nearest-even (NaN stays a quiet NaN)."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


# --------------------------------------------------------------------------- RoPE
def rope_inv_freq(d_rope: int) -> np.ndarray:
    """inv_freq_i = theta^(-i/half), i = 0 .. half-1 ([N1] apply_rope)."""
    half = d_rope // 2
    return np.array([THETA ** (-(i / half)) for i in range(half)], dtype=np.float64)


def rope_f64(x, pos) -> np.ndarray:
    """Exact (float64) half-split RoPE of ``x[..., d_R]`` at integer positions ``pos``.

    [DP] eq. (3) and (8) apply RoPE to the decoupled key/query branch; the
    rotation itself is [N1] ``apply_rope``: ``x*cos + rotate_half(x)*sin`` with
    ``rotate_half(x) = [-x2, x1]``.
    """
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(2 * half)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


@lru_cache(maxsize=8)
def rope_table_f32(n_pos: int, d_rope: int = 64) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin of ``pos * inv_freq_i`` computed in float64 by libm, rounded to float32.

    This is the fixed table the bit-exact append recipe rotates with: angle in
    double (``pos`` times ``10000^(-i/32)`` from ``pow``), ``cos``/``sin`` in double,
    one rounding to float32.
    """
    half = d_rope // 2
    inv = [THETA ** (-(i / half)) for i in range(half)]
    cos = np.empty((n_pos, half), dtype=np.float32)
    sin = np.empty((n_pos, half), dtype=np.float32)
    for p in range(n_pos):
        cos[p] = [math.cos(p * f) for f in inv]
        sin[p] = [math.sin(p * f) for f in inv]
    return cos, sin


def rope_key_bf16_bits(k_pe_bits, pos) -> np.ndarray:
    """Rotated key as the cache stores it: the fixed fp32 recipe, then bf16.

    ``k_pe_bits`` is ``[n, d_R]`` bf16 bits (pre-RoPE), ``pos`` is ``[n]``.  With
    ``c, s`` from :func:`rope_table_f32`, each output is one float32 product per
    term and one float32 add/subtract, every step rounded (no fused multiply-add),
    then rounded to bf16 (nearest even):
    ``r1 = (x1*c) - (x2*s)``, ``r2 = (x2*c) + (x1*s)``.
    """
    return f32_to_bf16_bits(rope_key_f32(k_pe_bits, pos))


def rope_key_f32(k_pe_bits, pos) -> np.ndarray:
    """The float32 rotated key of :func:`rope_key_bf16_bits` before its bf16 rounding."""
    x = bf16_bits_to_f32(k_pe_bits)
    pos = np.asarray(pos, dtype=np.int64)
    half = x.shape[-1] // 2
    need = int(pos.max()) + 1 if pos.size else 1
    cos_t, sin_t = rope_table_f32(-(-need // 4096) * 4096, 2 * half)
    c, s = cos_t[pos], sin_t[pos]
    x1, x2 = x[..., :half], x[..., half:]
    r1 = np.subtract(np.multiply(x1, c, dtype=np.float32), np.multiply(x2, s, dtype=np.float32), dtype=np.float32)
    r2 = np.add(np.multiply(x2, c, dtype=np.float32), np.multiply(x1, s, dtype=np.float32), dtype=np.float32)
    return np.concatenate([r1, r2], axis=-1)


# --------------------------------------------------------------------------- paged cache
def append_kv(cache_bits, c_kv_new_bits, k_pe_new_bits, seq_lens_before, page_table) -> np.ndarray:
    """Append n_new tokens per sequence to a paged cache image (returns a new image).

    Token ``j`` of sequence ``b`` sits at position ``pos = seq_lens_before[b] + j``
    and lands in page ``page_table[b][pos // 64]``, slot ``pos % 64``
    ([MA] §6: 64-token pages; [DP] FlashMLA point 4: paged cache with a block
    table).  The row is ``[c_kv ; RoPE(k_pe, pos)]``: the latent is copied, the
    RoPE key is rotated before it is cached ([N1] forward_decode step 1;
    [DP] eq. (3)).  Shapes: cache ``[P, 64, 576]``, c_kv ``[B, n, 512]``,
    k_pe ``[B, n, 64]``, all uint16 bf16 bits.
    """
    out = np.array(cache_bits, dtype=np.uint16, copy=True)
    c_new = np.asarray(c_kv_new_bits, dtype=np.uint16)
    k_new = np.asarray(k_pe_new_bits, dtype=np.uint16)
    B, n_new, d_c = c_new.shape
    if B == 0 or n_new == 0:
        return out
    lens = np.asarray(seq_lens_before, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    pos = lens[:, None] + np.arange(n_new)[None, :]            # [B, n]
    pages = np.take_along_axis(pt, pos // PAGE, axis=1)         # [B, n]
    slots = pos % PAGE
    out[pages, slots, :d_c] = c_new
    out[pages, slots, d_c:] = rope_key_bf16_bits(k_new.reshape(B * n_new, -1), pos.reshape(-1)).reshape(B, n_new, -1)
    return out


def gather_sequence(cache_bits, page_table_row, kv_len: int, d_c: int = 512):
    """Tokens 0..kv_len-1 of one sequence read back from the cache as float64: (c [kv, d_c], k^R [kv, d_R])."""
    t = np.arange(kv_len)
    pages = np.asarray(page_table_row, dtype=np.int64)[t // PAGE]
    rows = np.asarray(cache_bits, dtype=np.uint16)[pages, t % PAGE]
    return bf16_bits_to_f64(rows[:, :d_c]), bf16_bits_to_f64(rows[:, d_c:])


# --------------------------------------------------------------------------- FP8 latent cache
# The pages name FP8 (one byte per value) among the precisions for the cache and
# for "mixed precision with a scaling strategy" ([DP] §7, training and
# inference; [N1] "标准 KV Cache 的显存瓶颈", p_bytes = 1 for FP8) but fix no
# format.  Reading taken here: the 512 latent values of a token are stored as
# OCP FP8 E4M3 codes of c / s with one float32 scale s per token,
# s = max(amax / 448, 2^-10) (448 is E4M3's largest finite value; the floor keeps
# the stored RoPE key in range); the rotated key is stored as float16 of
# k^R / s, so that both parts of the score carry the same factor 1 / s.  The
# attention then works on the dequantised values c = s * E4M3(code) and
# k^R = s * f16(stored).

E4M3_MAX = 448.0
FP8_SCALE_FLOOR = 2.0 ** -10


def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3 codes as float64: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m / 8 * 2^-6); S.1111.111 is NaN; there are no
    infinities, so S.1111.110 = 448 is the largest finite magnitude.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


@lru_cache(maxsize=1)
def _e4m3_positive_grid():
    codes = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: every finite non-negative value
    return codes, e4m3_decode(codes)


def f32_to_e4m3_codes(x) -> np.ndarray:
    """Round float32 values to E4M3, to nearest with ties to the even code, saturating at +-448.

    Brute force over the 127 finite non-negative codes: the nearest value wins;
    on a tie the code with an even last mantissa bit.  NaN maps to 0x7F.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    codes, vals = _e4m3_positive_grid()
    a = np.minimum(np.abs(x), E4M3_MAX)
    d = np.abs(a[..., None] - vals)                   # [..., 127]
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # among tied candidates (at most two adjacent codes) prefer the even code
    even = (codes & 1) == 0
    pick = np.where(cand & even, 1, 0) + np.where(cand, 1, 0)   # 2: tied and even, 1: tied
    idx = pick.argmax(axis=-1)
    out = codes[idx].astype(np.uint8)
    out = np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)   # the sign is kept, also on zero
    out = np.where(np.isnan(x), np.uint8(0x7F), out)
    return out.astype(np.uint8)


def f32_to_f16_bits(x) -> np.ndarray:
    """Round float32 to IEEE binary16 (nearest even, overflow to infinity); bit patterns."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp8_token_scale(c_bits) -> np.ndarray:
    """Per-token scale ``s = max(amax / 448, 2^-10)`` in float32 (one IEEE division)."""
    c = bf16_bits_to_f32(c_bits)
    amax = np.abs(c).max(axis=-1).astype(np.float32)
    s = np.divide(amax, np.float32(E4M3_MAX), dtype=np.float32)
    return np.maximum(s, np.float32(FP8_SCALE_FLOOR)).astype(np.float32)


def append_kv_fp8(c8, scale, kr, c_kv_new_bits, k_pe_new_bits, seq_lens_before, page_table):
    """Append n_new tokens per sequence to an FP8 paged cache (returns new images).

    Images: ``c8 [P, 64, 512]`` uint8 E4M3 codes, ``scale [P, 64]`` float32,
    ``kr [P, 64, 64]`` uint16 float16 bits.  Token placement as :func:`append_kv`.
    Per token: ``s`` by :func:`fp8_token_scale`; code_i = E4M3(float32(c_i / s))
    (one IEEE division each, then :func:`f32_to_e4m3_codes`); the stored key is
    f16(float32(r / s)) for the float32 rotated key ``r`` of :func:`rope_key_f32`.
    """
    c8 = np.array(c8, dtype=np.uint8, copy=True)
    scale = np.array(scale, dtype=np.float32, copy=True)
    kr = np.array(kr, dtype=np.uint16, copy=True)
    c_new = np.asarray(c_kv_new_bits, dtype=np.uint16)
    k_new = np.asarray(k_pe_new_bits, dtype=np.uint16)
    B, n_new, d_c = c_new.shape
    if B == 0 or n_new == 0:
        return c8, scale, kr
    lens = np.asarray(seq_lens_before, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    pos = lens[:, None] + np.arange(n_new)[None, :]
    pages = np.take_along_axis(pt, pos // PAGE, axis=1)
    slots = pos % PAGE
    s = fp8_token_scale(c_new)                                     # [B, n]
    q = np.divide(bf16_bits_to_f32(c_new), s[..., None], dtype=np.float32)
    c8[pages, slots] = f32_to_e4m3_codes(q)
    scale[pages, slots] = s
    r = rope_key_f32(k_new.reshape(B * n_new, -1), pos.reshape(-1)).reshape(B, n_new, -1)
    kr[pages, slots] = f32_to_f16_bits(np.divide(r, s[..., None], dtype=np.float32))
    return c8, scale, kr


def gather_sequence_fp8(c8, scale, kr, page_table_row, kv_len: int):
    """Dequantised tokens 0..kv_len-1 of one sequence in float64: (c = s E4M3(code), k^R = s f16(stored))."""
    t = np.arange(kv_len)
    pages = np.asarray(page_table_row, dtype=np.int64)[t // PAGE]
    slots = t % PAGE
    s = np.asarray(scale, dtype=np.float32)[pages, slots].astype(np.float64)[:, None]
    c = s * e4m3_decode(np.asarray(c8, dtype=np.uint8)[pages, slots])
    k = s * np.asarray(kr, dtype=np.uint16)[pages, slots].view(np.float16).astype(np.float64)
    return c, k


# --------------------------------------------------------------------------- attention
def _softmax_lse(s: np.ndarray):
    """Max-subtracted softmax and natural log-sum-exp of a score vector ([DP] Softmax_j)."""
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    return e / z, m + math.log(z)


def decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len: int, heads=None):
    """One sequence's decode outputs by the plain definition (non-absorbed, fp64).

    Inputs (float64 or anything numpy converts): ``q_nope [n_q, H, d_h]``,
    ``q_rope [n_q, H, d_R]`` (pre-RoPE), ``w_uk``/``w_uv [H, d_h, d_c]``,
    ``c [kv, d_c]`` and rotated ``kr [kv, d_R]`` of the sequence's cached tokens.
    Query ``j`` is at position ``prior_len + j``.  Returns ``o [n_q, nh, d_v]``
    ([DP] eq. (10): ``o = sum_t alpha_t W_UV[h] c_t``), ``o_lat [n_q, nh, d_c]``
    (``sum_t alpha_t c_t``) and ``lse [n_q, nh]`` (natural log-sum-exp of the
    scaled scores) for the heads in ``heads`` (default: all).
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    n_q, n_h, d_h = q_nope.shape
    d_r = q_rope.shape[-1]
    d_c = c.shape[1]
    heads = list(range(n_h)) if heads is None else list(heads)
    scale = 1.0 / math.sqrt(d_h + d_r)
    o = np.zeros((n_q, len(heads), w_uv.shape[1]))
    o_lat = np.zeros((n_q, len(heads), d_c))
    lse = np.zeros((n_q, len(heads)))
    for hi, h in enumerate(heads):
        k = np.concatenate([c @ w_uk[h].T, kr], axis=1)   # [kv, d_h + d_R]
        v = c @ w_uv[h].T                                 # [kv, d_v]
        for j in range(n_q):
            pos = prior_len + j
            q = np.concatenate([q_nope[j, h], rope_f64(q_rope[j, h], pos)])
            alpha, lse[j, hi] = _softmax_lse((k[:pos + 1] @ q) * scale)
            o[j, hi] = alpha @ v[:pos + 1]
            o_lat[j, hi] = alpha @ c[:pos + 1]
    return o, o_lat, lse


def decompress_kv(c, w_uk, w_uv):
    """The non-absorbed path's first step: per-head keys and values from the latent.

    ``K[t, h] = W_UK[h] c_t`` and ``V[t, h] = W_UV[h] c_t`` ([MA] §2.2 "Non-Absorbed":
    decompress K and V, then standard MHA; [DP] eq. (2) and the value projection)
    for ``c [kv, d_c]`` and ``w_uk``/``w_uv [H, d_h, d_c]``; returns ``K, V [kv, H, d_h]``.
    With the cached ``k^R`` and ``[q^C ; RoPE(q^R)]`` these feed :func:`decode_mha`'s
    per-head attention, which is also the definition of the prefill path for any
    number of new tokens.
    """
    c = np.asarray(c, np.float64)
    k = np.einsum("tm,hdm->thd", c, np.asarray(w_uk, np.float64))
    v = np.einsum("tm,hdm->thd", c, np.asarray(w_uv, np.float64))
    return k, v


def decode_absorbed(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len: int, heads=None,
                    token_range: tuple[int, int] | None = None):
    """The absorbed form in fp64: the cross-check of the absorption identity, and
    (being far cheaper than the plain definition) the full-size reference for
    every sequence and head once that identity is pinned.

    ``q~ = W_UK[h]^T q^C`` ([DP] key absorption; [MA] §2.1 ``Q' = Q W_UK^T``),
    ``score_t = (q~ . c_t + RoPE(q^R) . k^R_t) / sqrt(d_h + d_h^R)`` ([MA] §4.1 score
    split), ``m = sum_t alpha_t c_t`` and ``o = W_UV[h] m`` ([DP] value absorption).
    All selected heads of one query are computed together as matrix products (the
    scores of every head are one ``[T, d_c] x [d_c, H]`` product).  With
    ``token_range=(t0, t1)`` only tokens in ``[t0, t1)`` take part and the result is
    that split's partial: ``o_lat`` normalised within the split and its ``lse``
    (``-inf`` and zeros when the split holds no visible token).
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    c = np.asarray(c, np.float64)
    kr = np.asarray(kr, np.float64)
    n_q, n_h, d_h = q_nope.shape
    d_r = q_rope.shape[-1]
    d_c = c.shape[1]
    heads = list(range(n_h)) if heads is None else list(heads)
    scale = 1.0 / math.sqrt(d_h + d_r)
    t0, t1 = token_range if token_range is not None else (0, c.shape[0])
    w_uk_s, w_uv_s = w_uk[heads], w_uv[heads]
    o = np.zeros((n_q, len(heads), w_uv.shape[1]))
    o_lat = np.zeros((n_q, len(heads), d_c))
    lse = np.full((n_q, len(heads)), -np.inf)
    for j in range(n_q):
        pos = prior_len + j
        hi_t = min(t1, pos + 1)
        if hi_t <= t0:
            continue
        q_t = np.einsum("hd,hdm->hm", q_nope[j, heads], w_uk_s)          # [H, d_c]
        q_r = rope_f64(q_rope[j, heads], pos)                           # [H, d_R]
        s = (c[t0:hi_t] @ q_t.T + kr[t0:hi_t] @ q_r.T) * scale          # [T, H]
        m = s.max(axis=0)
        e = np.exp(s - m)
        z = e.sum(axis=0)
        o_lat[j] = (e / z).T @ c[t0:hi_t]
        lse[j] = m + np.log(z)
        o[j] = np.einsum("hm,hdm->hd", o_lat[j], w_uv_s)
    return o, o_lat, lse


def combine_splits(o_parts, lse_parts):
    """Merge per-split partials by log-sum-exp ([DP] FlashMLA point 3: blocked,
    online-normalised softmax over the history).

    ``o_parts [S, ..., d]`` are split-normalised outputs, ``lse_parts [S, ...]``
    their log-sum-exps (``-inf`` for empty splits).  Returns ``(o, lse)`` with
    ``lse = log sum_s exp(lse_s)`` and ``o = sum_s exp(lse_s - lse) o_s``.
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    m = lse_parts.max(axis=0)
    w = np.exp(lse_parts - m)
    z = w.sum(axis=0)
    lse = m + np.log(z)
    o = (w[..., None] * o_parts).sum(axis=0) / z[..., None]
    return o, lse


def out_absorb(o_lat, w_uv):
    """``O[h] = W_UV[h] O'[h]`` for ``o_lat [..., H, d_c]`` ([N1] final einsum 'bhm,hdm->bhd')."""
    return np.einsum("...hm,hdm->...hd", np.asarray(o_lat, np.float64), np.asarray(w_uv, np.float64))


def linear(x, w):
    """``y = x W^T`` in fp64 for ``x [..., K]`` and an nn.Linear weight ``w [N, K]``
    ([N1] decode listing: the W_DKV, W_KR, W_DQ, W_UQ, W_QR and W_O projections)."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def decode_layer(x, w_dkv, w_kr, w_dq, w_uq, w_qr, w_uk, w_uv, w_o, c_hist, kr_hist, prior_len: int,
                 cache_bf16_rows: bool = True):
    """One sequence's decode layer from the hidden state ([N1] forward_decode).

    ``x [n_q, d_model]`` is the hidden state of the ``n_q`` new tokens at positions
    ``prior_len + j``; ``c_hist [prior_len, 512]`` and ``kr_hist [prior_len, 64]``
    (rotated) are the cached history.  Steps, in the listing's order:
    1. ``c^KV = x W_DKV^T`` and ``k^R = RoPE(x W_KR^T, pos)``, appended to the cache
       (as the bf16 rows the cache format holds, with the fixed RoPE recipe of
       :func:`rope_key_bf16_bits`, when ``cache_bf16_rows``);
    2. ``c^Q = x W_DQ^T``, ``q^C = c^Q W_UQ^T`` and ``q^R = c^Q W_QR^T`` per head;
    3-5. the attention of :func:`decode_mha` (per-head output O);
    then ``y = O W_O^T`` over the concatenated heads.
    Returns ``(y [n_q, d_model], O [n_q, H, d_v])``; everything else in fp64.
    """
    x = np.asarray(x, np.float64)
    n_q = x.shape[0]
    c_new = linear(x, w_dkv)
    k_new = linear(x, w_kr)
    pos = prior_len + np.arange(n_q)
    if cache_bf16_rows:
        c_new = bf16_bits_to_f64(f32_to_bf16_bits(c_new.astype(np.float32)))
        kr_new = bf16_bits_to_f64(rope_key_bf16_bits(f32_to_bf16_bits(k_new.astype(np.float32)), pos))
    else:
        kr_new = rope_f64(k_new, pos)
    c = np.concatenate([np.asarray(c_hist, np.float64).reshape(-1, c_new.shape[1]), c_new])
    kr = np.concatenate([np.asarray(kr_hist, np.float64).reshape(-1, kr_new.shape[1]), kr_new])
    c_q = linear(x, w_dq)
    H, d_h, _ = np.asarray(w_uk).shape
    q_nope = linear(c_q, w_uq).reshape(n_q, H, d_h)
    q_rope = linear(c_q, w_qr).reshape(n_q, H, -1)
    o, _, _ = decode_mha(q_nope, q_rope, w_uk, w_uv, c, kr, prior_len)
    y = linear(o.reshape(n_q, -1), w_o)
    return y, o


def absorb_query(q_nope, q_rope, w_uk, pos):
    """``[W_UK[h]^T q^C ; RoPE(q^R, pos)]`` per head: the 576-wide absorbed query in fp64.

    ``q_nope [..., H, d_h]``, ``q_rope [..., H, d_R]``, ``pos`` broadcast over the
    leading axes ([N1] step 3 einsum 'bhd,hdm->bhm'; [DP] eq. (8) for the RoPE part).
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_t = np.einsum("...hd,hdm->...hm", q_nope, np.asarray(w_uk, np.float64))
    pos = np.asarray(pos)[..., None]
    q_r = rope_f64(q_rope, np.broadcast_to(pos, q_rope.shape[:-1]))
    return np.concatenate([q_t, q_r], axis=-1)
