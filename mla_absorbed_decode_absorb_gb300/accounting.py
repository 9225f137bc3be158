"""Algorithmic byte and FLOP counts of one MLA step, on either path.

These are the figures the roofline is taken against, counted from the problem
statement, not from any kernel:

* each cached token is ``d_c + d_h^R = 512 + 64 = 576`` scalars, 1152 bytes in
  bf16, and is read once per sequence per step (DeepSeek-MLA-Principle, "KV
  cache per token" and the decode HBM-traffic comparison in "那为什么 MLA 仍可能更快");
* per (query token, visible cache token) the absorbed path does
  ``2*n_h*d_c + n_h*d_h^R`` multiply-adds: logits over the 576-wide row and the
  weighted sum over the 512-wide latent (same page, "推理计算：FLOPs 可能增加",
  the MLA history-interaction count), i.e. 139,264 MACs = 278,528 FLOP;
* query token ``j`` of a sequence with ``L`` prior tokens sees ``L + j + 1``
  cache tokens (causal among the new tokens).

The non-absorbed path (a chunk of many new tokens) first decompresses every
cached token into per-head keys and values, ``2 * n_h * d_h * d_c`` MACs per token
([MA] section 2.2, K = c W_UK, V = c W_UV), then does ``n_h * (d_h + d_h^R + d_v)``
MACs per (query token, visible token) (DeepSeek-MLA-Principle section 6, the
non-absorbed L^2 terms: logits over 192 columns and the weighted sum over 128).
"""

from __future__ import annotations

from .workloads import D_LATENT, D_NOPE, D_ROPE, N_HEADS

BF16_BYTES = 2


def cache_scalars_per_token() -> int:
    return D_LATENT + D_ROPE


def mha_cache_scalars_per_token() -> int:
    """Per-token K and V of plain multi-head attention with 128 heads of 128."""
    return 2 * N_HEADS * D_NOPE


# The FP8 latent cache: 512 one-byte E4M3 codes, one float32 scale, 64 float16 key values.
FP8_CACHE_BYTES_PER_TOKEN = D_LATENT + 4 + 2 * D_ROPE


def cache_bytes_per_token(dtype_bytes: int = BF16_BYTES, cache_format: str = "bf16") -> int:
    if cache_format == "fp8":
        return FP8_CACHE_BYTES_PER_TOKEN
    return cache_scalars_per_token() * dtype_bytes


def mla_history_macs(L: int) -> int:
    """Multiply-adds of one query token against L cache tokens (absorbed form)."""
    return 2 * L * N_HEADS * D_LATENT + L * N_HEADS * D_ROPE


def mha_history_macs(L: int) -> int:
    """Multiply-adds of one query token against L cached K/V rows (plain MHA)."""
    return 2 * L * N_HEADS * D_NOPE


def flops_per_token_pair() -> int:
    return 2 * mla_history_macs(1)


def step_cache_bytes(kv_lens, cache_format: str = "bf16") -> int:
    """Cache bytes one decode step reads: every cached token once per sequence."""
    return sum(int(n) for n in kv_lens) * cache_bytes_per_token(cache_format=cache_format)


def step_attention_flops(kv_lens, n_q: int) -> int:
    """Attention FLOPs of one step; query j of a sequence sees kv_len - n_q + j + 1 tokens."""
    tot = 0
    for n in kv_lens:
        L = int(n) - n_q
        for j in range(n_q):
            tot += (L + j + 1) * flops_per_token_pair()
    return tot


def roofline_seconds(kv_lens, n_q: int, hbm_gbs: float, tflops: float) -> tuple[float, str]:
    """Slower of cache bytes at HBM bandwidth and FLOPs at dense bf16 tensor peak."""
    t_mem = step_cache_bytes(kv_lens) / (hbm_gbs * 1e9)
    t_flop = step_attention_flops(kv_lens, n_q) / (tflops * 1e12)
    return (t_mem, "hbm") if t_mem >= t_flop else (t_flop, "tensor")


def decompress_macs_per_token() -> int:
    """K and V of one cached token for all heads: 2 * n_h * d_h * d_c."""
    return 2 * N_HEADS * D_NOPE * D_LATENT


def prefill_pair_macs() -> int:
    """Non-absorbed attention per (query token, visible token): n_h * (d_h + d_h^R + d_v)."""
    return N_HEADS * (D_NOPE + D_ROPE + D_NOPE)


def prefill_attention_flops(kv_lens, n_q: int) -> int:
    tot = 0
    for n in kv_lens:
        L = int(n) - n_q
        pairs = n_q * (L + 1) + n_q * (n_q - 1) // 2  # sum over j of (L + j + 1)
        tot += 2 * pairs * prefill_pair_macs()
    return tot


def decompress_flops(kv_lens) -> int:
    return sum(int(n) for n in kv_lens) * 2 * decompress_macs_per_token()



def layer_weight_bytes(d_model: int, d_q_latent: int = 1536, fold: bool = False) -> int:
    """bf16 bytes of every weight one decode-layer step reads once: W_DKV, W_KR, W_DQ,
    W_UQ, W_QR, W_O ([N1] decode listing) and W_UK, W_UV; with the pre-folds, W_DKV,
    W_KR, W_DQ, W_QK [n_h d_c, d_c'], W_QR and W_OV [d_model, n_h d_c]."""
    hd = N_HEADS * D_NOPE
    head_in = (D_LATENT + D_ROPE + d_q_latent) * d_model
    if fold:
        elems = head_in + N_HEADS * D_LATENT * d_q_latent + N_HEADS * D_ROPE * d_q_latent \
            + d_model * N_HEADS * D_LATENT
    else:
        elems = head_in + (hd + N_HEADS * D_ROPE) * d_q_latent + d_model * hd + 2 * N_HEADS * D_NOPE * D_LATENT
    return elems * BF16_BYTES
