"""Device-resident decode state for one workload, and one decode step over it.

A :class:`DecodeSession` owns (as torch tensors) the weights, the paged cache
with each sequence's history already appended, the page table, the RoPE table,
the step's inputs and every output/workspace buffer, so that a step is just
these ABI calls with no allocation (three launches with the defaults below):

1. ``mla_append_kv``           -- write this step's n_q tokens into the cache;
2. ``mla_absorb_q``            -- ``q_abs = [q^C W_UK ; RoPE(q^R)]``;
3. ``mla_decode_attn_partial`` -- split attention (per-split partials);
4. ``mla_combine_out_absorb``  -- log-sum-exp merge of the splits and
   ``O = O' W_UV^T`` in one launch.

With ``fused_finish=False`` step 4 is the two separate calls
``mla_decode_combine`` (which also writes the merged O' to ``o_latent``) and
``mla_out_absorb``.  Steps 1 and 2 are independent: by default
(``fused_prologue``) they are the one call ``mla_append_absorb_q`` (or its FP8 form),
so a step is three launches; with ``overlap_append`` step 1 runs on a side
stream forked from the caller's stream and joined before step 3.  By default all launches stay on the caller's stream, where the
library's programmatic dependent launch (``mla_set_launch_overlap``) lets each
kernel's prologue overlap the previous one.

With the workload's ``cache_format`` "fp8" the cache is the FP8 latent cache
(E4M3 codes with one scale per token) and steps 1 and 3 are
``mla_append_kv_fp8`` and ``mla_decode_attn_fp8_partial``; the rest is unchanged.

A step that brings ``PREFILL_MIN_NEW_TOKENS`` (64) or more new tokens per
sequence takes the non-absorbed path instead, as inference engines switch for
prefill and chunked prefill: ``mla_append_kv``, ``mla_decompress_kv`` (per-head
keys and values from the latent cache) and ``mla_prefill_attn`` (causal MHA),
which give the same per-head output ``out``.
"""

from __future__ import annotations

import torch

from . import ops
from .workloads import D_LATENT, D_NOPE, D_ROW, N_HEADS, Inputs, empty_cache


# New tokens per sequence from which a step takes the non-absorbed path (the
# switch point the MLA pages give for prefill / chunked prefill).
PREFILL_MIN_NEW_TOKENS = 64


class StepGraph:
    """A session's step captured once into a CUDA graph (the session's buffers are
    fixed, so every replay runs the same kernels on the current step inputs)."""

    def __init__(self, session, warmup: int = 2):
        self.session = session
        self.stream = torch.cuda.Stream(device=session.device)
        self.stream.wait_stream(torch.cuda.current_stream(session.device))
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):  # lazy one-time setup (attributes, tables) outside the capture
                session.step(self.stream)
        torch.cuda.current_stream(session.device).wait_stream(self.stream)
        torch.cuda.synchronize(session.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            session.step(self.stream)

    def replay(self):
        self.graph.replay()
        return self.session.out


class DecodeSession:
    def __init__(self, inp: Inputs, device="cuda", split_pages: int | None = None, stream=None,
                 fused_finish: bool = True, overlap_append: bool = False, path: str | None = None,
                 fused_prologue: bool = True):
        self.inp = inp
        self.cache_format = inp.workload.cache_format
        if self.cache_format not in ("bf16", "fp8"):
            raise ValueError(f"unknown cache format {self.cache_format!r}")
        self.fused_finish = bool(fused_finish)
        self.overlap_append = bool(overlap_append)
        self.device = torch.device(device)
        wl = inp.workload
        self.B, self.n_q = wl.batch, wl.n_q
        self.split_pages = wl.split_pages if split_pages is None else int(split_pages)
        if path is None:
            # the absorbed kernels take up to MLA_MAX_NQ new tokens per sequence
            small = self.n_q < PREFILL_MIN_NEW_TOKENS and self.n_q <= ops.MLA_MAX_NQ
            path = "absorbed" if small else "non_absorbed"
        if path not in ("absorbed", "non_absorbed"):
            raise ValueError(f"unknown path {path!r}")
        self.path = path
        if self.cache_format == "fp8" and path != "absorbed":
            raise ValueError("the FP8 latent cache is read by the absorbed path only")
        # append + absorb_q as one launch (both on the caller's stream)
        self.fused_prologue = bool(fused_prologue) and path == "absorbed" and not self.overlap_append
        dev = self.device
        self.max_kv_len = int(inp.kv_lens.max()) if self.B else self.n_q
        self.rope = ops.rope_table(self.max_kv_len + 1, dev, stream)
        self.w_uk = inp.w_uk.to(dev)
        self.w_uv = inp.w_uv.to(dev)
        self.page_table = inp.page_table.to(dev)
        # this step's inputs live in one device buffer (typed views into it), so that
        # a caller uploads them with a single copy (see host_step_buffer)
        c_new, k_new = inp.new_tokens()
        self._pack_step_inputs([("c_new", c_new), ("k_new", k_new), ("q_nope", inp.q_nope),
                                ("q_rope", inp.q_rope), ("prior_lens", inp.prior_lens), ("kv_lens", inp.kv_lens)])
        if self.cache_format == "fp8":
            self.cache = None
            self.cache_fp8 = ops.fp8_cache_empty(inp.num_pages, dev)
        else:
            self.cache = empty_cache(inp.num_pages, dev)
        zero = torch.zeros(1, dtype=torch.int32, device=dev)
        for b in range(self.B):
            hc, hk = inp.history(b)
            if hc.shape[0] == 0:
                continue
            if self.cache_format == "fp8":
                ops.mla_append_kv_fp8(hc.to(dev)[None], hk.to(dev)[None], zero, self.page_table[b:b + 1],
                                      self.rope, self.cache_fp8, stream=stream)
            else:
                ops.mla_append_kv(hc.to(dev)[None], hk.to(dev)[None], zero, self.page_table[b:b + 1], self.rope,
                                  self.cache, stream=stream)
        self.lse = torch.empty(self.B, self.n_q, N_HEADS, dtype=torch.float32, device=dev)
        self.out = torch.empty(self.B, self.n_q, N_HEADS, D_NOPE, dtype=torch.bfloat16, device=dev)
        if self.path == "absorbed":
            self.q_abs = torch.empty(self.B, self.n_q, N_HEADS, D_ROW, dtype=torch.bfloat16, device=dev)
            self.o_latent = torch.empty(self.B, self.n_q, N_HEADS, D_LATENT, dtype=torch.float32, device=dev)
            self.workspace = ops.alloc_workspace(self.B, self.n_q, self.max_kv_len, self.split_pages, dev)
            self.num_splits = ops.mla_decode_num_splits(self.B, self.n_q, self.max_kv_len, self.split_pages)
        else:
            kv_shape = (self.B, N_HEADS, self.max_kv_len, D_NOPE)
            self.k_nope = torch.empty(kv_shape, dtype=torch.bfloat16, device=dev)
            self.v = torch.empty(kv_shape, dtype=torch.bfloat16, device=dev)
            self.num_splits = 1
        if self.overlap_append:
            self.side = torch.cuda.Stream(device=dev)
            self._forked = torch.cuda.Event()
            self._appended = torch.cuda.Event()

    _ALIGN = 256

    def _pack_step_inputs(self, named):
        self._layout, off = [], 0
        for name, t in named:
            t = t.contiguous()
            n = t.numel() * t.element_size()
            self._layout.append((name, off, t.dtype, tuple(t.shape), n))
            off = (off + n + self._ALIGN - 1) // self._ALIGN * self._ALIGN
        self.step_buffer = torch.zeros(max(off, 1), dtype=torch.uint8, device=self.device)
        for (name, o, dtype, shape, n), (_, t) in zip(self._layout, named):
            view = self.step_buffer[o:o + n].view(dtype).view(shape)
            view.copy_(t.contiguous())
            setattr(self, name, view)

    def host_step_buffer(self, pin: bool = True) -> torch.Tensor:
        """A host copy of the packed step inputs (same layout as ``step_buffer``)."""
        host = torch.empty(self.step_buffer.shape, dtype=torch.uint8)
        if pin:
            host = host.pin_memory()
        host.copy_(self.step_buffer)
        return host

    def upload(self, host_in: torch.Tensor, stream=None):
        """This step's inputs from a pinned host buffer laid out as ``host_step_buffer``:
        one ``mla_copy_async`` (SM loads over the host link, in the launch-overlap chain)."""
        ops.mla_copy(self.step_buffer, host_in, stream)

    def download(self, host_out: torch.Tensor, stream=None):
        """The step's output ``out`` into a pinned host buffer of the same size."""
        ops.mla_copy(host_out, self.out, stream)

    def _main(self, stream):
        if stream is None:
            return torch.cuda.current_stream(self.device)
        if isinstance(stream, torch.cuda.Stream):
            return stream
        return torch.cuda.ExternalStream(int(stream), device=self.device)

    # individual stages (the bench times them one by one)
    def append(self, stream=None):
        if self.overlap_append:
            self._forked.record(self._main(stream))
            self.side.wait_event(self._forked)
            stream = self.side
        if self.cache_format == "fp8":
            ops.mla_append_kv_fp8(self.c_new, self.k_new, self.prior_lens, self.page_table, self.rope,
                                  self.cache_fp8, stream=stream)
        else:
            ops.mla_append_kv(self.c_new, self.k_new, self.prior_lens, self.page_table, self.rope, self.cache,
                              stream=stream)
        if self.overlap_append:
            self._appended.record(self.side)

    def absorb(self, stream=None):
        ops.mla_absorb_q(self.q_nope, self.q_rope, self.prior_lens, self.w_uk, self.rope, self.q_abs,
                         stream=stream)

    def append_absorb(self, stream=None):
        if self.cache_format == "fp8":
            ops.mla_append_absorb_q_fp8(self.c_new, self.k_new, self.q_nope, self.q_rope, self.prior_lens,
                                        self.page_table, self.w_uk, self.rope, self.cache_fp8, self.q_abs,
                                        stream=stream)
        else:
            ops.mla_append_absorb_q(self.c_new, self.k_new, self.q_nope, self.q_rope, self.prior_lens,
                                    self.page_table, self.w_uk, self.rope, self.cache, self.q_abs, stream=stream)

    def attend_partial(self, stream=None):
        if self.overlap_append:
            self._main(stream).wait_event(self._appended)  # the cache holds the new tokens
        if self.cache_format == "fp8":
            ops.mla_decode_attn_fp8_partial(self.q_abs, self.cache_fp8, self.page_table, self.kv_lens, self.n_q,
                                            self.max_kv_len, self.split_pages, self.workspace, self.o_latent,
                                            self.lse, stream=stream)
        else:
            ops.mla_decode_attn_partial(self.q_abs, self.cache, self.page_table, self.kv_lens, self.n_q,
                                        self.max_kv_len, self.split_pages, self.workspace, self.o_latent,
                                        self.lse, stream=stream)

    def combine(self, stream=None):
        ops.mla_decode_combine(self.B, self.n_q, self.max_kv_len, self.split_pages, self.workspace,
                               self.o_latent, self.lse, stream=stream)

    def project_out(self, stream=None, out=None):
        ops.mla_out_absorb(self.o_latent, self.w_uv, self.out if out is None else out, stream=stream)

    def finish(self, stream=None, out=None):
        ops.mla_combine_out_absorb(self.B, self.n_q, self.max_kv_len, self.split_pages, self.workspace,
                                   self.o_latent, self.w_uv, self.out if out is None else out, self.lse,
                                   stream=stream)

    def decompress(self, stream=None):
        if self.overlap_append:
            self._main(stream).wait_event(self._appended)  # the cache holds the new tokens
        ops.mla_decompress_kv(self.cache, self.page_table, self.kv_lens, self.max_kv_len, self.w_uk, self.w_uv,
                              self.k_nope, self.v, stream=stream)

    def prefill_attn(self, stream=None):
        ops.mla_prefill_attn(self.q_nope, self.q_rope, self.prior_lens, self.rope, self.k_nope, self.v, self.cache,
                             self.page_table, self.kv_lens, self.out, self.lse, stream=stream)

    def stage_names(self) -> list[str]:
        if self.path == "non_absorbed":
            return ["append", "decompress", "prefill_attn"]
        tail = ["finish"] if self.fused_finish else ["combine", "project_out"]
        head = ["append_absorb"] if self.fused_prologue else ["append", "absorb"]
        return head + ["attend_partial"] + tail

    def step(self, stream=None, host_out: torch.Tensor | None = None):
        """One decode step; with ``host_out`` (pinned host memory, the shape of ``out``)
        the result lands there: the out-projection stores it across the host link
        itself, or (other paths) a download follows."""
        names = self.stage_names()
        for name in names[:-1]:
            getattr(self, name)(stream)
        if host_out is not None and names[-1] in ("finish", "project_out"):
            getattr(self, names[-1])(stream, out=host_out)
            return host_out
        getattr(self, names[-1])(stream)
        if host_out is not None:
            self.download(host_out, stream)
            return host_out
        return self.out

    def capture(self, warmup: int = 2) -> "StepGraph":
        """The decode step (its launches and their programmatic dependencies) captured
        as one CUDA graph: ``replay()`` then costs one launch call on the host instead of
        one per kernel, which is what bounds short steps issued back to back."""
        return StepGraph(self, warmup)

    def launches_per_step(self) -> int:
        if self.path == "non_absorbed":
            return 3
        n = 3 if self.fused_prologue else 4
        if self.fused_finish:
            return n
        return n + (1 if self.num_splits > 1 else 0)


class LayerSession:
    """One MLA decode layer from the hidden state, as in the pages' decode listing
    ("DeepSeek MLA 架构详解", forward_decode), on top of a :class:`DecodeSession`:

    1. ``proj_kv``: c_kv = x W_DKV^T and k_pe = x W_KR^T, written straight into the
       decode session's step inputs (so the append stores this step's projections);
    2. ``proj_q``: c_q = x W_DQ^T, then q^C = c_q W_UQ^T and q^R = c_q W_QR^T into
       the step's query inputs;
    3. the decode session's append, absorb_q, split attention and fused finish,
       which give the per-head output O;
    4. ``proj_out``: y = O W_O^T, the layer's output [B, n_q, d_model].

    Every projection is one ``mla_linear`` (plus its split-sum kernel when K is
    split).  The history of every sequence is in the cache before the first step.

    With ``fold=True`` the layer uses the weight pre-folds of the pages ("DeepSeek-
    MLA-Principle", key absorption: q~ = (W_UK[h])^T W_UQ[h] c^Q; "DeepSeek MLA
    架构详解": W^OV[h] = W^O[h] W_UV[h]), prepared once by ``mla_linear`` calls:
    ``proj_q`` writes the query's latent half straight into q_abs (one strided
    linear of c^Q with W_QK [128 * 512, 1536]) and its RoPE half by ``mla_rope_q``
    (no absorb_q); after the attention the merged latent output O' is rounded to
    bf16 and ``proj_out`` is one linear with W_OV [d_model, 128 * 512] (no W_UV
    step).  The folded weights are 201 MB and 940 MB against 66 MB and 252 MB.
    """

    def __init__(self, li, device="cuda", split_pages: int | None = None, stream=None, fold: bool = False):
        self.li = li
        self.fold = bool(fold)
        dev = torch.device(device)
        self.device = dev
        self.dec = DecodeSession(li.base, device=dev, split_pages=split_pages, stream=stream)
        d = self.dec
        self.T = d.B * d.n_q
        self.d_model = li.workload.d_model
        self.x = li.x.to(dev).reshape(self.T, self.d_model)
        self.w_dkv, self.w_kr, self.w_dq = li.w_dkv.to(dev), li.w_kr.to(dev), li.w_dq.to(dev)
        self.w_uq, self.w_qr, self.w_o = li.w_uq.to(dev), li.w_qr.to(dev), li.w_o.to(dev)
        self.c_q = torch.empty(self.T, self.w_dq.shape[0], dtype=torch.bfloat16, device=dev)
        self.y = torch.empty(self.T, self.d_model, dtype=torch.bfloat16, device=dev)
        # step inputs of the decode session, viewed as [tokens, features]
        self._c_new = d.c_new.view(self.T, -1)
        self._k_new = d.k_new.view(self.T, -1)
        self._q_nope = d.q_nope.view(self.T, -1)
        self._q_rope = d.q_rope.view(self.T, -1)
        shapes = [(self.w_dkv, self.d_model), (self.w_kr, self.d_model), (self.w_dq, self.d_model),
                  (self.w_uq, self.c_q.shape[1]), (self.w_qr, self.c_q.shape[1]), (self.w_o, d.out[0].numel() // d.n_q)]
        need = max(ops.mla_linear_workspace_size(self.T, k, w.shape[0]) for w, k in shapes)
        need = max(need, ops.mla_linear_pair_workspace_size(self.T, self.d_model, self.w_dkv.shape[0],
                                                            self.w_kr.shape[0]))
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        # a layer step's input is the hidden state, its result the layer output
        self.step_buffer = self.x
        self.out = self.y
        if self.fold:
            self._prepare_folds(stream)

    def _prepare_folds(self, stream=None):
        """W_QK[(h, m), c] = sum_d W_UK[h, d, m] W_UQ[h*128 + d, c] and
        W_OV[j, (h, m)] = sum_d W_O[j, h*128 + d] W_UV[h, d, m], each by mla_linear calls
        (K = d_h = 128; row blocks of at most 256)."""
        d = self.dec
        H, dh, dc = d.w_uk.shape
        dev = self.device
        dq = self.w_uq.shape[1]
        self.w_qk = torch.empty(H * dc, dq, dtype=torch.bfloat16, device=dev)
        self.w_ov = torch.empty(self.d_model, H * dc, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(16, max(ops.mla_linear_workspace_size(256, dh, n) for n in (dq, dc))),
                         dtype=torch.uint8, device=dev)
        for h in range(H):
            uk_t = d.w_uk[h].t().contiguous()                          # [512, 128]
            uq_t = self.w_uq[h * dh:(h + 1) * dh].t().contiguous()      # [1536, 128]
            for r0 in range(0, dc, 256):
                ops.mla_linear(uk_t[r0:r0 + 256], uq_t, self.w_qk[h * dc + r0:h * dc + r0 + 256], ws, stream)
            o_blk = self.w_o[:, h * dh:(h + 1) * dh].contiguous()       # [d_model, 128]
            uv_t = d.w_uv[h].t().contiguous()                           # [512, 128]
            for r0 in range(0, self.d_model, 256):
                rows = min(256, self.d_model - r0)
                ops.mla_linear_strided(o_blk[r0:r0 + rows], uv_t, self.w_ov[r0:, h * dc:], H * dc, dc, dc, ws,
                                       stream)
        self.o_lat_bf16 = torch.empty(self.T, H * dc, dtype=torch.bfloat16, device=dev)
        need = max(ops.mla_linear_workspace_size(self.T, dq, H * dc),
                   ops.mla_linear_workspace_size(self.T, H * dc, self.d_model))
        if need > self.ws.numel():
            self.ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def host_step_buffer(self, pin: bool = True) -> torch.Tensor:
        host = torch.empty(self.x.shape, dtype=self.x.dtype)
        if pin:
            host = host.pin_memory()
        host.copy_(self.x)
        return host

    def upload(self, host_in: torch.Tensor, stream=None):
        ops.mla_copy(self.x, host_in, stream)

    def download(self, host_out: torch.Tensor, stream=None):
        ops.mla_copy(host_out, self.y, stream)

    def proj_kv(self, stream=None):
        # W_DKV and W_KR read the same hidden state: one launch
        ops.mla_linear_pair(self.x, self.w_dkv, self.w_kr, self._c_new, self._k_new, self.ws, stream)

    def proj_q(self, stream=None):
        ops.mla_linear(self.x, self.w_dq, self.c_q, self.ws, stream)
        if self.fold:
            d = self.dec
            ops.mla_linear_strided(self.c_q, self.w_qk, d.q_abs, N_HEADS * D_ROW, D_LATENT, D_ROW, self.ws, stream)
            ops.mla_linear(self.c_q, self.w_qr, self._q_rope, self.ws, stream)
            ops.mla_rope_q(d.q_rope, d.prior_lens, d.rope, d.q_abs, stream=stream)
            return
        ops.mla_linear(self.c_q, self.w_uq, self._q_nope, self.ws, stream)
        ops.mla_linear(self.c_q, self.w_qr, self._q_rope, self.ws, stream)

    def to_bf16(self, stream=None):
        ops.mla_f32_to_bf16(self.dec.o_latent, self.o_lat_bf16, stream=stream)

    def proj_out(self, stream=None):
        if self.fold:
            ops.mla_linear(self.o_lat_bf16, self.w_ov, self.y, self.ws, stream)
            return
        ops.mla_linear(self.dec.out.view(self.T, -1), self.w_o, self.y, self.ws, stream)

    def stage_names(self) -> list[str]:
        if self.fold:
            return ["proj_kv", "proj_q", "append", "attend_partial", "combine", "to_bf16", "proj_out"]
        return ["proj_kv", "proj_q"] + self.dec.stage_names() + ["proj_out"]

    def __getattr__(self, name):
        # the decode stages (append, absorb, attend_partial, finish, ...) run on the decode session
        return getattr(self.__dict__["dec"], name)

    def step(self, stream=None, host_out: torch.Tensor | None = None):
        for name in self.stage_names():
            getattr(self, name)(stream)
        if host_out is not None:
            self.download(host_out, stream)
            return host_out
        return self.y

    def launches_per_step(self) -> int:
        d = self.d_model
        dq = self.c_q.shape[1]
        if self.fold:
            n = 2 + (1 if self.dec.num_splits > 1 else 0) + 1 + 1   # append, attention, combine, to_bf16, rope_q
            lin = [(self.w_dq, d), (self.w_qk, dq), (self.w_qr, dq), (self.w_ov, self.w_ov.shape[1])]
        else:
            n = self.dec.launches_per_step()
            lin = [(self.w_dq, d), (self.w_uq, dq), (self.w_qr, dq), (self.w_o, self.w_o.shape[1])]
        for w, k in lin:
            n += 1 + (1 if ops.mla_linear_workspace_size(self.T, k, w.shape[0]) else 0)
        # W_DKV and W_KR in one launch (plus its split-K sum)
        n += 1 + (1 if ops.mla_linear_pair_workspace_size(self.T, d, self.w_dkv.shape[0], self.w_kr.shape[0]) else 0)
        return n
