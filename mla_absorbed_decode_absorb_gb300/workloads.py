"""Seeded synthetic workloads for absorbed MLA decode.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no RoPE, no projection, no softmax).  Both the CUDA path and
the CPU oracle consume what it produces, which is why it lives on its own.

Recipe (one ``torch.Generator('cpu')`` per workload, seed 0 by default, drawn in
this fixed order):

1. prior context lengths ``L_b`` (only for ragged workloads: i.i.d. integers,
   uniform on ``[lo, hi]`` inclusive);
2. ``W_UK`` then ``W_UV``, each ``[n_h=128, d_h=128, d_c=512]`` ~ N(0, 0.02) (std);
3. per sequence ``b`` in order, ``c_kv`` ``[L_b + n_q, 512]`` then ``k_pe``
   ``[L_b + n_q, 64]`` ~ N(0, 1); the first ``L_b`` rows are the history, the last
   ``n_q`` rows are the tokens this decode step appends;
4. ``Q_nope`` ``[B, n_q, 128, 128]`` then ``Q_rope`` ``[B, n_q, 128, 64]`` ~ N(0, 1);
5. one random permutation of the page pool, dealt out in order to the
   sequences' page lists, so page tables are shuffled and non-contiguous.

Every floating tensor is drawn in fp32 and rounded to bf16 (round to nearest
even).  ``k_pe`` is the key's RoPE branch *before* rotation; RoPE is applied by
the append step.  The pool holds the pages the sequences need plus 10% spare;
unused page-table entries are -1.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

N_HEADS = 128
D_NOPE = 128
D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE  # 576 scalars per cached token
PAGE = 64
W_STD = 0.02
SPARE_FRACTION = 0.10


@dataclass(frozen=True)
class Workload:
    """One decode-step workload: ``batch`` sequences, ``n_q`` new tokens each."""

    name: str
    batch: int
    n_q: int
    context: int = 0                      # uniform prior length L (when ragged is None)
    ragged: tuple[int, int] | None = None  # inclusive range for i.i.d. uniform L_b
    lengths: tuple[int, ...] | None = None  # explicit L_b (edge-case workloads)
    split_pages: int = 0                  # prescribed KV split size in pages (0 = auto)
    description: str = ""
    cache_format: str = "bf16"            # "bf16" (576 bf16 per token) or "fp8" (E4M3 latent, see ops)
    d_model: int = 0                      # > 0: the whole layer from the hidden state (see LayerInputs)
    fold: bool = False                    # the layer with the weight pre-folds (W_QK, W_OV)


# The five workloads of the benchmark, named by what they are.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_b1_l256", batch=1, n_q=1, context=256,
                 description="B=1, 1 new token, prior context 256"),
        Workload("batched_b32_l4096", batch=32, n_q=1, context=4096,
                 description="B=32, 1 new token each, uniform prior context 4096, shuffled pages"),
        Workload("ragged_b128_l1024_8192", batch=128, n_q=1, ragged=(1024, 8192),
                 description="B=128, prior context i.i.d. uniform in [1024, 8192]"),
        Workload("long_b8_l32768", batch=8, n_q=1, context=32768, split_pages=64,
                 description="B=8, prior context 32768, KV split in 64-page chunks"),
        Workload("mtp_b64_l8192_q4", batch=64, n_q=4, context=8192,
                 description="B=64, 4 causal new query tokens, prior context 8192"),
    ]
}

# Steps with many new tokens per sequence, which take the non-absorbed path
# (chunked prefill after a prior context, and a prompt with no prior context).
PREFILL_WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("chunk_b4_l4096_c512", batch=4, n_q=512, context=4096,
                 description="B=4, a chunk of 512 new tokens each after a prior context of 4096"),
        Workload("prompt_b8_c2048", batch=8, n_q=2048, context=0,
                 description="B=8, a 2048-token prompt each, no prior context"),
        Workload("chunk_b1_l4096_c512", batch=1, n_q=512, context=4096,
                 description="B=1, a chunk of 512 new tokens after 4096 (the chunk case at the size "
                             "a full counter capture handles)"),
        Workload("prompt_b2_c2048", batch=2, n_q=2048, context=0,
                 description="B=2, a 2048-token prompt each (the prompt case at the size a full "
                             "counter capture handles)"),
    ]
}

# The batched decode over the FP8 latent cache (644 bytes per token instead of 1152).
FP8_WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("batched_b32_l4096_fp8", batch=32, n_q=1, context=4096, cache_format="fp8",
                 description="B=32, 1 new token each, uniform prior context 4096, FP8 latent cache"),
    ]
}

# The whole decode layer from the hidden state: the projections of the pages'
# decode listing around the absorbed attention, hidden size 7168 (DeepSeek-V3).
D_MODEL = 7168
D_Q_LATENT = 1536
LAYER_WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("layer_b32_l4096", batch=32, n_q=1, context=4096, d_model=D_MODEL,
                 description="decode layer from the hidden state (d_model 7168): B=32, 1 new token each, "
                             "uniform prior context 4096"),
        Workload("layer_b32_l4096_fold", batch=32, n_q=1, context=4096, d_model=D_MODEL, fold=True,
                 description="the same decode layer with the weight pre-folds W_UK^T W_UQ and W_O W_UV"),
    ]
}

DEFAULT_BENCH_WORKLOAD = "batched_b32_l4096"
# The decode workloads every default bench run reports (the headline one in full,
# the others in its per-workload pass).
DECODE_REPORT_WORKLOADS = tuple(WORKLOADS)


def custom(name: str, lengths, n_q: int = 1, split_pages: int = 0, cache_format: str = "bf16") -> Workload:
    """A workload with explicit prior lengths (parity and edge-case tests)."""
    lengths = tuple(int(x) for x in lengths)
    return Workload(name, batch=len(lengths), n_q=n_q, lengths=lengths, split_pages=split_pages,
                    cache_format=cache_format)


def scaled(wl: Workload, batch: int | None = None, context: int | None = None) -> Workload:
    """The same workload shape with a smaller batch and/or context."""
    return Workload(
        wl.name + "_scaled", batch=batch or wl.batch, n_q=wl.n_q,
        context=context if context is not None else wl.context,
        ragged=None if context is not None else wl.ragged,
        lengths=None, split_pages=wl.split_pages, description="scaled " + wl.description,
        cache_format=wl.cache_format)


@dataclass
class Inputs:
    """CPU tensors of one generated workload (bf16 unless noted)."""

    workload: Workload
    seed: int
    prior_lens: torch.Tensor      # int32 [B]   L_b: tokens already cached
    kv_lens: torch.Tensor         # int32 [B]   L_b + n_q
    w_uk: torch.Tensor            # [128, 128, 512]
    w_uv: torch.Tensor            # [128, 128, 512]
    c_kv: torch.Tensor            # [sum(kv_lens), 512]   rows of sequence b start at tok_offsets[b]
    k_pe: torch.Tensor            # [sum(kv_lens), 64]    pre-RoPE
    tok_offsets: torch.Tensor     # int64 [B + 1]
    q_nope: torch.Tensor          # [B, n_q, 128, 128]
    q_rope: torch.Tensor          # [B, n_q, 128, 64]     pre-RoPE
    page_table: torch.Tensor      # int32 [B, max_pages], -1 where unused
    num_pages: int                # size of the page pool
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.workload.batch

    @property
    def n_q(self) -> int:
        return self.workload.n_q

    def history(self, b: int):
        """(c_kv, k_pe) rows of the first L_b tokens of sequence b."""
        lo = int(self.tok_offsets[b])
        n = int(self.prior_lens[b])
        return self.c_kv[lo:lo + n], self.k_pe[lo:lo + n]

    def new_tokens(self):
        """(c_kv, k_pe) of the n_q tokens appended this step: [B, n_q, 512], [B, n_q, 64]."""
        rows = []
        for b in range(self.batch):
            lo = int(self.tok_offsets[b]) + int(self.prior_lens[b])
            rows.append(torch.arange(lo, lo + self.n_q))
        idx = torch.stack(rows)
        return self.c_kv[idx], self.k_pe[idx]

    def sequence(self, b: int):
        """(c_kv, k_pe) rows of all kv_lens[b] tokens of sequence b."""
        lo = int(self.tok_offsets[b])
        hi = int(self.tok_offsets[b + 1])
        return self.c_kv[lo:hi], self.k_pe[lo:hi]


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def generate(wl: Workload, seed: int = 0) -> Inputs:
    """Draw the workload's inputs with the fixed recipe in the module docstring."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, n_q = wl.batch, wl.n_q
    if wl.lengths is not None:
        prior = torch.tensor(wl.lengths, dtype=torch.int64)
    elif wl.ragged is not None:
        lo, hi = wl.ragged
        prior = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    else:
        prior = torch.full((B,), wl.context, dtype=torch.int64)
    kv = prior + n_q

    w_uk = _bf16(torch.randn(N_HEADS, D_NOPE, D_LATENT, generator=g) * W_STD)
    w_uv = _bf16(torch.randn(N_HEADS, D_NOPE, D_LATENT, generator=g) * W_STD)

    total = int(kv.sum())
    c_kv = torch.empty(total, D_LATENT, dtype=torch.bfloat16)
    k_pe = torch.empty(total, D_ROPE, dtype=torch.bfloat16)
    offsets = torch.zeros(B + 1, dtype=torch.int64)
    pos = 0
    for b in range(B):
        n = int(kv[b])
        c_kv[pos:pos + n] = _bf16(torch.randn(n, D_LATENT, generator=g))
        k_pe[pos:pos + n] = _bf16(torch.randn(n, D_ROPE, generator=g))
        pos += n
        offsets[b + 1] = pos

    q_nope = _bf16(torch.randn(B, n_q, N_HEADS, D_NOPE, generator=g))
    q_rope = _bf16(torch.randn(B, n_q, N_HEADS, D_ROPE, generator=g))

    pages = [(int(n) + PAGE - 1) // PAGE for n in kv]
    need = sum(pages)
    pool = need + int(math.ceil(SPARE_FRACTION * need))
    perm = torch.randperm(pool, generator=g)
    max_pages = max(pages) if pages else 1
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    k = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[k:k + p].to(torch.int32)
        k += p

    return Inputs(workload=wl, seed=seed, prior_lens=prior.to(torch.int32), kv_lens=kv.to(torch.int32),
                  w_uk=w_uk, w_uv=w_uv, c_kv=c_kv, k_pe=k_pe, tok_offsets=offsets,
                  q_nope=q_nope, q_rope=q_rope, page_table=table, num_pages=pool)


# bf16 quiet NaN written into every cache slot no token has been appended to, so
# that a read of an unwritten slot shows up in the output.
CACHE_SENTINEL_BITS = 0x7FC0


def empty_cache(num_pages: int, device="cpu") -> torch.Tensor:
    """A page pool ``[num_pages, 64, 576]`` bf16 filled with the NaN sentinel."""
    t = torch.full((num_pages, PAGE, D_ROW), CACHE_SENTINEL_BITS, dtype=torch.int16, device=device)
    return t.view(torch.bfloat16)


@dataclass
class LayerInputs:
    """The decode-layer inputs: the hidden state of the new tokens and the six
    projection weights (nn.Linear layout [out, in]), next to the attention inputs
    (history, page table, W_UK, W_UV) of :class:`Inputs`, whose own new-token
    latent rows and queries the layer replaces by its projections."""

    base: Inputs
    x: torch.Tensor          # [B, n_q, d_model]
    w_dkv: torch.Tensor      # [512, d_model]
    w_kr: torch.Tensor       # [64, d_model]
    w_dq: torch.Tensor       # [1536, d_model]
    w_uq: torch.Tensor       # [128 * 128, 1536]
    w_qr: torch.Tensor       # [128 * 64, 1536]
    w_o: torch.Tensor        # [d_model, 128 * 128]

    @property
    def workload(self) -> Workload:
        return self.base.workload


def generate_layer(wl: Workload, seed: int = 0) -> LayerInputs:
    """:func:`generate` for the attention inputs, then (second generator, seed + 1)
    the hidden state ~ N(0, 1) and weights ~ N(0, 1 / fan_in), rounded to bf16."""
    base = generate(wl, seed)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    d = wl.d_model
    B, n_q = wl.batch, wl.n_q

    def w(n_out, n_in):
        return _bf16(torch.randn(n_out, n_in, generator=g) / math.sqrt(n_in))
    return LayerInputs(base=base, x=_bf16(torch.randn(B, n_q, d, generator=g)),
                       w_dkv=w(D_LATENT, d), w_kr=w(D_ROPE, d), w_dq=w(D_Q_LATENT, d),
                       w_uq=w(N_HEADS * D_NOPE, D_Q_LATENT), w_qr=w(N_HEADS * D_ROPE, D_Q_LATENT),
                       w_o=w(d, N_HEADS * D_NOPE))
