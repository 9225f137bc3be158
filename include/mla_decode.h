/*
 * mla_decode.h -- C ABI of the absorbed Multi-Head Latent Attention decode path
 * for GB300 (sm_103a).
 *
 * The decode step reads only the compressed per-token cache: a 512-wide latent
 * c_kv plus a 64-wide RoPE key shared by all heads, 576 bf16 scalars per token,
 * stored in pages of 64 tokens.  Per-head keys and values are never formed:
 * W_UK is folded into the query and W_UV is applied once to the latent output
 * ("MLA 矩阵吸收 & 吸收分离 原理详解", sections 2.1 and 4.1;
 * "DeepSeek-MLA-Principle", "3) MLA 中怎么吸收", key and value absorption).
 *
 * Fixed dimensions (DeepSeek-V3, "DeepSeek-MLA-Principle" section 3 table):
 *   n_h = 128 heads, d_h = 128 (content part of q/k per head), d_h^R = 64
 *   (RoPE part), d_c = 512 (latent), d_v = 128; score scale 1/sqrt(192);
 *   RoPE theta = 10000, half-split rotation; page size 64 tokens.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major and densely packed as
 *     the shape comments say, owned by the caller.  The library allocates no
 *     memory.  bf16 tensors are passed as their 16-bit patterns (mla_bf16).
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns MLA_ERR_INVALID_ARG (or MLA_ERR_UNSUPPORTED /
 *     MLA_ERR_WORKSPACE) and launches nothing.
 *   - Work is enqueued asynchronously on `stream` (0 = the legacy default
 *     stream).  A launch failure returns MLA_ERR_CUDA.
 *   - Faults found by the kernels themselves (a page id or position out of
 *     range, a bounded wait that ran out) never trap: the kernel skips the
 *     access, records the first such code in a per-device status word and
 *     returns.  mla_get_device_status() reads and clears that word.
 *   - A 16-byte-aligned base address is required for every tensor.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16; /* bit pattern of a bfloat16 value */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, bad size or alignment */
  MLA_ERR_UNSUPPORTED = 2, /* shape outside what the kernels handle */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  MLA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MLA_ERR_TIMEOUT = 5,     /* (device status) a bounded wait ran out */
  MLA_ERR_BOUNDS = 6,      /* (device status) page id / position out of range */
  MLA_ERR_RANGE = 7        /* (device status) a partial attention score exceeded the
                              kernel's exchange range (|q . row| over half a row of at
                              least 65520 * 256 = 1.677e7) or was NaN */
} mla_status;

enum {
  MLA_N_HEADS = 128,
  MLA_D_NOPE = 128,
  MLA_D_LATENT = 512,
  MLA_D_ROPE = 64,
  MLA_D_ROW = 576, /* MLA_D_LATENT + MLA_D_ROPE scalars per cached token */
  MLA_PAGE = 64,
  MLA_MAX_NQ = 8   /* new query tokens per sequence per step */
};

/* Version of this ABI (bumped on any signature change). */
int mla_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(mla_status status);

/*
 * RoPE table.  RoPE is the half-split rotation of "DeepSeek MLA 架构详解"
 * (apply_rope in its decode listing): inv_freq_i = 10000^(-i/32), i < 32,
 * angle = pos * inv_freq_i, out[i] = x[i] cos - x[i+32] sin,
 * out[i+32] = x[i+32] cos + x[i] sin.
 *
 * mla_rope_table_bytes: bytes of a table covering positions [0, max_positions).
 * mla_rope_table_init: fills a caller-owned device buffer `table`
 *   [max_positions][64] float32 (cos of the 32 frequencies, then sin) with the
 *   angles' cos/sin computed in double on the host and rounded once to float.
 *   Blocking: returns after the copy to `table` has completed on `stream`.
 *   The table is an input of mla_append_kv and mla_absorb_q; any position they
 *   rotate must be < max_positions.
 */
size_t mla_rope_table_bytes(int max_positions);
mla_status mla_rope_table_init(float* table, int max_positions, cudaStream_t stream);

/*
 * mla_append_kv -- write n_new tokens per sequence into the paged cache.
 * ("DeepSeek MLA 架构详解", decode listing step 1: rotate the key, then append;
 *  "DeepSeek-MLA-Principle" eq. (3) and FlashMLA point 4, paged cache with a
 *  block table; "MLA 矩阵吸收 …" section 6, page_size = 64.)
 *
 *   c_kv_new        [B, n_new, 512] bf16   latent of the new tokens
 *   k_pe_new        [B, n_new, 64]  bf16   RoPE key of the new tokens, NOT yet rotated
 *   seq_lens_before [B] int32              position of each sequence's first new token
 *   page_table      [B, pt_stride] int32   page ids of each sequence's pages, in order
 *   rope_table      from mla_rope_table_init, covering positions < rope_max_pos
 *   cache           [num_pages, 64, 576] bf16, updated in place
 *
 * Token j of sequence b has position pos = seq_lens_before[b] + j and is written
 * to cache[page_table[b][pos/64]][pos%64] as [c_kv ; RoPE(k_pe, pos)].  The
 * rotation is done in float32 with separately rounded products and sums (no
 * fused multiply-add) and rounded to bf16 to nearest even, so the cache image
 * is reproducible bit for bit.  A token whose position, page slot or page id is
 * out of range is skipped and sets MLA_ERR_BOUNDS in the device status.
 * B >= 0, n_new >= 0 (0 launches nothing).
 */
mla_status mla_append_kv(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                         const int32_t* seq_lens_before, const int32_t* page_table,
                         int pt_stride, const float* rope_table, int rope_max_pos,
                         mla_bf16* cache, int64_t num_pages, int B, int n_new,
                         cudaStream_t stream);

/*
 * mla_absorb_q -- the absorbed query, 576 wide per head.
 * ("MLA 矩阵吸收 …" section 2.1, Q' = Q W_UK^T; "DeepSeek-MLA-Principle"
 *  key absorption q~ = (W_UK[h])^T q^C; "DeepSeek MLA 架构详解" step 3,
 *  einsum 'bhd,hdm->bhm'; RoPE of the query branch, eq. (8).)
 *
 *   q_nope          [B, n_q, 128, 128] bf16  content query q^C per head
 *   q_rope          [B, n_q, 128, 64]  bf16  RoPE query q^R per head, NOT yet rotated
 *   seq_lens_before [B] int32                query j of sequence b is at position
 *                                            seq_lens_before[b] + j
 *   w_uk            [128, 128, 512] bf16     W_UK[h][d][m]
 *   q_abs           [B, n_q, 128, 576] bf16  out: [sum_d q^C[d] W_UK[h][d][:] ; RoPE(q^R)]
 *
 * Accumulation is float32; results are rounded to bf16.  1 <= n_q <= MLA_MAX_NQ.
 */
mla_status mla_absorb_q(const mla_bf16* q_nope, const mla_bf16* q_rope,
                        const int32_t* seq_lens_before, const mla_bf16* w_uk,
                        const float* rope_table, int rope_max_pos, mla_bf16* q_abs,
                        int B, int n_q, cudaStream_t stream);

/*
 * mla_append_absorb_q -- mla_append_kv(c_kv_new, k_pe_new, ..., cache, B, n_new = n_q)
 * and mla_absorb_q(q_nope, q_rope, ..., q_abs, B, n_q) in one launch.
 * (The same two steps as above: "DeepSeek MLA 架构详解" decode listing steps 1
 *  and 3.)  The query side reads nothing the append writes, so the rows are
 * written by warps of the absorbed-query kernel; the cache image and q_abs are
 * bit for bit those of the two separate calls.  Arguments as in those calls,
 * with n_new = n_q; the constraints of both apply (16-byte aligned c_kv_new,
 * cache, q_nope, q_rope, w_uk, q_abs; 1 <= n_q <= MLA_MAX_NQ), and a token out
 * of range sets MLA_ERR_BOUNDS exactly as in mla_append_kv.  A decode step that
 * uses it launches one kernel fewer, and the attention that follows waits for
 * one grid instead of two.
 */
mla_status mla_append_absorb_q(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                               const mla_bf16* q_nope, const mla_bf16* q_rope,
                               const int32_t* seq_lens_before, const int32_t* page_table,
                               int pt_stride, const mla_bf16* w_uk,
                               const float* rope_table, int rope_max_pos,
                               mla_bf16* cache, int64_t num_pages, mla_bf16* q_abs,
                               int B, int n_q, cudaStream_t stream);

/*
 * Split-KV attention over the paged latent cache.
 * ("DeepSeek-MLA-Principle" section 2: score = q.k / sqrt(d_h + d_h^R), softmax,
 *  eq. (10); the absorbed score Q'_nope c^T + Q_rope k_rope^T of "MLA 矩阵吸收 …"
 *  section 4.1; value absorption O' = softmax . c; FlashMLA point 3: blocked,
 *  online-normalised softmax over the history, split-KV.)
 *
 *   q_abs      [B, n_q, 128, 576] bf16 (from mla_absorb_q)
 *   cache      [num_pages, 64, 576] bf16; must already hold the n_q new tokens
 *   page_table [B, pt_stride] int32
 *   kv_lens    [B] int32: cached tokens of each sequence INCLUDING the n_q new
 *              ones; query j of sequence b sees tokens 0 .. kv_lens[b] - n_q + j
 *              (causal among the new tokens); kv_lens[b] >= n_q.
 *   max_kv_len host-side upper bound of kv_lens (sizes the grid without a sync);
 *              a sequence longer than it sets MLA_ERR_BOUNDS.
 *   split_pages pages per KV split (0 = choose automatically: at most 2
 *              (sequence, query) units over at most 1024 cached tokens then run
 *              the short-context kernel, one CTA per 8 heads on warp-level
 *              tensor-core tiles and no split, which mla_decode_uses_short_path
 *              reports; otherwise the split count that fills the GPU with 2-CTA
 *              tcgen05 clusters).
 *   workspace  device scratch of at least mla_decode_workspace_size() bytes,
 *              16-byte aligned (may be NULL when that size is 0); a missing, short
 *              or misaligned workspace returns MLA_ERR_WORKSPACE.
 *   o_latent   [B, n_q, 128, 512] float32 out: O'[h] = sum_t alpha_t c_t
 *   lse        [B, n_q, 128] float32 out (nullable): natural log-sum-exp of the
 *              scaled scores.
 *
 * mla_decode_attn runs the split kernel and, when there is more than one
 * split, the float32 log-sum-exp combine.  The two halves are also exposed
 * separately (same arguments): mla_decode_attn_partial writes per-split partials
 * into the workspace (or the final outputs when there is a single split) and
 * mla_decode_combine merges them (a no-op for a single split).  A split's partial
 * O' rows are stored in bf16: each is normalised within its split, a convex
 * combination of cache rows, so rounding it costs at most half a bf16 ulp of a
 * cache-sized value per element; the partial log-sum-exps and the merge stay
 * float32.
 */
mla_status mla_decode_workspace_size(int B, int n_q, int max_kv_len, int split_pages,
                                     size_t* bytes);
mla_status mla_decode_num_splits(int B, int n_q, int max_kv_len, int split_pages,
                                 int* num_splits);
mla_status mla_decode_uses_short_path(int B, int n_q, int max_kv_len, int split_pages,
                                      int* is_short);
mla_status mla_decode_attn(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                           const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                           int B, int n_q, int max_kv_len, int split_pages,
                           void* workspace, size_t workspace_bytes,
                           float* o_latent, float* lse, cudaStream_t stream);
mla_status mla_decode_attn_partial(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                                   const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                                   int B, int n_q, int max_kv_len, int split_pages,
                                   void* workspace, size_t workspace_bytes,
                                   float* o_latent, float* lse, cudaStream_t stream);
mla_status mla_decode_combine(int B, int n_q, int max_kv_len, int split_pages,
                              const void* workspace, size_t workspace_bytes,
                              float* o_latent, float* lse, cudaStream_t stream);

/*
 * mla_linear -- y = x W^T for a few tokens: the projections around the
 * attention ("DeepSeek MLA 架构详解", decode listing: W_DKV, W_KR, W_DQ, W_UQ,
 * W_QR and W_O are linear layers without bias; "DeepSeek-MLA-Principle"
 * section 2 table for their shapes).
 *
 *   x  [T, K] bf16, 1 <= T <= MLA_LINEAR_MAX_T, K a multiple of 64
 *   w  [N, K] bf16 (the nn.Linear weight layout: one row per output), N >= 1
 *   y  [T, N] bf16 out: y[t][n] = bf16(sum_k x[t][k] w[n][k]), fp32 accumulation
 *   workspace: mla_linear_workspace_size bytes (0 when K is not split), 16-byte
 *              aligned, caller-owned; its contents are scratch.
 *
 * K is split over CTAs when the output alone would not cover the GPU; the
 * split partials are then added in a fixed order by a second kernel, so the
 * result does not depend on timing.  x and w need 16-byte-aligned bases.
 */
#define MLA_LINEAR_MAX_T 256
mla_status mla_linear_workspace_size(int T, int K, int N, size_t* bytes);
mla_status mla_linear(const mla_bf16* x, const mla_bf16* w, mla_bf16* y, int T, int K, int N,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);
/*
 * mla_linear_strided -- mla_linear writing y[t][n] to
 *   y[t * y_ld + (n / seg) * seg_ld + n % seg]
 * (N a multiple of seg, seg_ld >= seg, y_ld >= (N / seg) * seg_ld): e.g. the
 * latent half of q_abs [T, 128, 576] with seg = 512, seg_ld = 576, y_ld = 128 * 576.
 */
mla_status mla_linear_strided(const mla_bf16* x, const mla_bf16* w, mla_bf16* y, int T, int K, int N,
                              int64_t y_ld, int seg, int seg_ld, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);
/*
 * mla_linear_pair -- two projections of the same x in one launch: y0 = x W0^T
 * [T, N0] and y1 = x W1^T [T, N1], each as mla_linear computes it (fp32
 * accumulation; K may be split differently from two separate calls, which
 * only reorders the fp32 sums).  For the pairs of the decode
 * listing that share their input, W_DKV and W_KR of the hidden state: a launch
 * and a split-K sum fewer than two calls, which matters when the weights are
 * small and the projections latency-bound.  workspace: mla_linear_pair_workspace_size
 * bytes (0 when K is not split).  Arguments and errors otherwise as mla_linear.
 */
mla_status mla_linear_pair_workspace_size(int T, int K, int N0, int N1, size_t* bytes);
mla_status mla_linear_pair(const mla_bf16* x, int T, int K, const mla_bf16* w0, int N0, mla_bf16* y0,
                           const mla_bf16* w1, int N1, mla_bf16* y1, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Weight pre-folds ("DeepSeek-MLA-Principle", key absorption: when q^C = W_UQ c^Q
 * the two linear maps combine, q~ = (W_UK[h])^T W_UQ[h] c^Q; "DeepSeek MLA 架构详解":
 * W_UV folded into the output projection, W^OV[h] = W^O[h] W_UV[h], d x d_c).
 * With the folded weights the query's latent half is one mla_linear_strided of
 * c^Q into q_abs, and the layer output one mla_linear of the merged latent
 * output O' (as bf16) with W^OV.  Two helpers complete those steps:
 *
 * mla_rope_q -- the RoPE half of q_abs alone: q_abs[t, h, 512:576] =
 *   RoPE(q_rope[t, h], seq_lens_before[b] + j), the float32 recipe of
 *   mla_absorb_q, bit for bit; arguments as mla_absorb_q.
 * mla_f32_to_bf16 -- dst[i] = bf16(src[i]) (nearest even), n elements.
 */
mla_status mla_rope_q(const mla_bf16* q_rope, const int32_t* seq_lens_before, const float* rope_table,
                      int rope_max_pos, mla_bf16* q_abs, int B, int n_q, cudaStream_t stream);
mla_status mla_f32_to_bf16(const float* src, mla_bf16* dst, int64_t n, cudaStream_t stream);

/*
 * FP8 latent cache.  The pages list FP8 (one byte per value) among the cache
 * precisions, with a scaling strategy ("DeepSeek-MLA-Principle" section 7,
 * mixed precision such as FP16/BF16/FP8 with scaling; "DeepSeek MLA 架构详解",
 * the KV-cache memory formula with p_bytes = 1 for FP8), without fixing a
 * format.  This library's format, per token t at page p, slot k:
 *   cache_c8    [num_pages, 64, 512] uint8    OCP FP8 E4M3 codes of c_t / s_t
 *   cache_scale [num_pages, 64]      float32  s_t = max(amax_t / 448, 2^-10)
 *   cache_kr    [num_pages, 64, 64]  float16  (bits) k^R_t / s_t
 * where amax_t is the largest |c_t[i]| of the token's bf16 latent, 448 the
 * largest finite E4M3 value and k^R_t the rotated key of mla_append_kv.  644
 * bytes per token instead of 1152.  The attention works on the dequantised
 * values c_t = s_t E4M3(code) and k^R_t = s_t f16(stored).
 *
 * mla_append_kv_fp8 -- mla_append_kv for this format.  Each value passes the
 * same float32 steps (so the image is reproducible bit for bit): amax of the
 * bf16 inputs; s_t = max(amax / 448, 2^-10) with one IEEE division; each code
 * = E4M3(c_i / s_t), one IEEE division, then nearest even with saturation at
 * +-448; the key r is rotated as in mla_append_kv (float32, separately rounded
 * products and sums) and stored as f16(r / s_t), one IEEE division, nearest
 * even.  Arguments, placement and errors are those of mla_append_kv.
 *
 * mla_decode_attn_fp8_partial -- mla_decode_attn_partial over this format:
 * same outputs, workspace, split plan and errors (combine and the fused
 * finish calls take its partials unchanged).  Partial scores are exchanged as
 * fp16 of (score over half a row) / 256 as in the bf16 kernel, and P reaches
 * the P V MMA as f16(p_t s_t): a page whose p_t s_t exceeds 65504 (s_t above
 * 255, i.e. a latent value beyond about 114000) overflows.  The query is
 * converted to float16 (exact for 2^-14 <= |q| <= 65504).
 *
 * mla_append_absorb_q_fp8 -- mla_append_absorb_q with this format: the rows of
 * mla_append_kv_fp8 (n_new = n_q) and the q_abs of mla_absorb_q in one launch,
 * bit for bit those of the two separate calls; arguments and errors of both
 * (16-byte aligned c_kv_new, cache_c8, q_nope, q_rope, w_uk, q_abs).
 */
mla_status mla_append_kv_fp8(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                             const int32_t* seq_lens_before, const int32_t* page_table,
                             int pt_stride, const float* rope_table, int rope_max_pos,
                             uint8_t* cache_c8, float* cache_scale, uint16_t* cache_kr,
                             int64_t num_pages, int B, int n_new, cudaStream_t stream);
mla_status mla_append_absorb_q_fp8(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                                   const mla_bf16* q_nope, const mla_bf16* q_rope,
                                   const int32_t* seq_lens_before, const int32_t* page_table,
                                   int pt_stride, const mla_bf16* w_uk,
                                   const float* rope_table, int rope_max_pos,
                                   uint8_t* cache_c8, float* cache_scale, uint16_t* cache_kr,
                                   int64_t num_pages, mla_bf16* q_abs, int B, int n_q,
                                   cudaStream_t stream);
mla_status mla_decode_attn_fp8_partial(const mla_bf16* q_abs, const uint8_t* cache_c8,
                                       const float* cache_scale, const uint16_t* cache_kr,
                                       int64_t num_pages, const int32_t* page_table, int pt_stride,
                                       const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                       int split_pages, void* workspace, size_t workspace_bytes,
                                       float* o_latent, float* lse, cudaStream_t stream);

/*
 * mla_decode_attn_noalloc -- mla_decode_attn for callers that cannot allocate
 * device memory.  (The MLA pages have no counterpart to this call; it exists for
 * deployment.)  Some callers may not call cudaMalloc when they run a decode
 * step: a serving runtime whose device memory is reserved up front by its own
 * pool, a plugin that may only touch the buffers it is handed, or a hot path
 * where allocation is forbidden.  This variant takes no workspace: the split
 * partials live in a 16 MiB array inside the library, which every GPU that loads
 * the library holds until the process exits.
 *
 * Arguments, outputs and semantics are those of mla_decode_attn without
 * `workspace`/`workspace_bytes`.  Limit: the split plan must fit the array,
 * i.e. B * n_q * num_splits <= 127 units of split partials (each 128 x 512
 * bf16 values and 128 floats); a single-split plan needs none.  A larger plan returns
 * MLA_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress with that device current); make that first call before
 * any stream capture.  The looked-up address belongs to the device's context:
 * after cudaDeviceReset it is stale, so do not call this entry point again in
 * that process.  All calls share the one array, so calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race and
 * corrupt each other's partials; the array keeps the last call's contents,
 * which are fully rewritten by each call before they are read.  No memory is
 * allocated or freed by this call.
 */
mla_status mla_decode_attn_noalloc(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                                   const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                                   int B, int n_q, int max_kv_len, int split_pages,
                                   float* o_latent, float* lse, cudaStream_t stream);

/*
 * mla_out_absorb -- O[h] = W_UV[h] O'[h], the value up-projection applied once.
 * ("MLA 矩阵吸收 …" section 2.1, V side: O = (Attn c) W_UV, once per step;
 *  "DeepSeek MLA 架构详解" step 5, einsum 'bhm,hdm->bhd'.)
 *
 *   o_latent [B, n_q, 128, 512] float32 (from mla_decode_attn)
 *   w_uv     [128, 128, 512] bf16   W_UV[h][d][m]
 *   out      [B, n_q, 128, 128] bf16 out: device memory, or pinned host memory
 *            mapped into the device's address space (the kernel then stores the
 *            result across the host link itself: no separate download); 16-byte
 *            aligned; pageable host memory gives MLA_ERR_INVALID_ARG
 *
 * o_latent is rounded to bf16 before the product; accumulation is float32.
 */
mla_status mla_out_absorb(const float* o_latent, const mla_bf16* w_uv, mla_bf16* out,
                          int B, int n_q, cudaStream_t stream);

/*
 * mla_combine_out_absorb -- mla_decode_combine and mla_out_absorb in one launch:
 * out[h] = W_UV[h] O'[h] with O' the log-sum-exp merge of the split partials.
 * (FlashMLA point 3 of "DeepSeek-MLA-Principle": the per-split results of the
 *  blocked softmax are merged by their log-sum-exps; "MLA 矩阵吸收 …" section
 *  2.1, V side: the up-projection W_UV is applied once, after the attention.)
 *
 *   B, n_q, max_kv_len, split_pages, workspace, workspace_bytes: as given to the
 *              mla_decode_attn_partial call whose results are consumed
 *   o_latent   [B, n_q, 128, 512] float32: read only when the plan has a single
 *              split (mla_decode_attn_partial then wrote the final O' there)
 *   w_uv       [128, 128, 512] bf16   W_UV[h][d][m]
 *   out        [B, n_q, 128, 128] bf16 out: device memory or mapped pinned host
 *              memory, as in mla_out_absorb
 *   lse        [B, n_q, 128] float32 out (nullable), written only when there is
 *              more than one split (otherwise the partial call already wrote it)
 *
 * The merged O' is formed in float32 with the same operations in the same order
 * as mla_decode_combine, rounded to bf16 and multiplied as in mla_out_absorb, so
 * `out` equals combine-then-out_absorb bit for bit; O' itself is not written to
 * o_latent.  Errors: MLA_ERR_INVALID_ARG for bad sizes or unaligned pointers,
 * MLA_ERR_WORKSPACE if the workspace is smaller than the plan needs or not 16-byte
 * aligned.
 */
mla_status mla_combine_out_absorb(int B, int n_q, int max_kv_len, int split_pages,
                                  const void* workspace, size_t workspace_bytes, const float* o_latent,
                                  const mla_bf16* w_uv, mla_bf16* out, float* lse, cudaStream_t stream);

/*
 * The non-absorbed path, for a chunk of many new tokens (prefill / chunked
 * prefill).  ("MLA 矩阵吸收 …" section 2.2, Non-Absorbed: decompress K = c W_UK
 * and V = c W_UV, then standard MHA; section 6: engines switch to it when a step
 * brings about 64 new tokens or more; "DeepSeek-MLA-Principle" section 6, the
 * L^2 terms of prefill are ~3x smaller without absorption.)  A step on this path:
 * mla_append_kv for the chunk, mla_decompress_kv, mla_prefill_attn; the result is
 * the same per-head O that the absorbed path's mla_out_absorb produces.
 *
 * mla_decompress_kv -- K[b, h, t, :] = W_UK[h] c_t, V[b, h, t, :] = W_UV[h] c_t for
 * the cached tokens t < kv_lens[b] of every sequence.
 *   cache, num_pages, page_table, pt_stride: as for mla_decode_attn
 *   kv_lens    [B] int32 tokens to decompress per sequence (<= max_kv_len)
 *   w_uk, w_uv [128, 128, 512] bf16
 *   k_nope, v  [B, 128, max_kv_len, 128] bf16 out (head-major).  Rows from
 *              kv_lens[b] up to the next multiple of 128 (within max_kv_len) are
 *              written as zeros; rows beyond that are not touched.
 * Accumulation is float32, results rounded to bf16.  MLA_ERR_UNSUPPORTED when
 * B * 128 * (max_kv_len + 64) does not fit in 31 bits.
 *
 * mla_prefill_attn -- O[b, j, h] = sum_t softmax_t(s) V[b, h, t] with
 * s_t = [q^C ; RoPE(q^R, pos)] . [K[b, h, t] ; k^R_t] / sqrt(192), causal: query j of
 * sequence b sits at pos = seq_lens_before[b] + j and sees tokens 0 .. pos.
 *   q_nope     [B, n_q, 128, 128] bf16; q_rope [B, n_q, 128, 64] bf16, NOT rotated
 *   seq_lens_before [B] int32; kv_lens [B] int32 must equal seq_lens_before + n_q
 *   rope_table, rope_max_pos: from mla_rope_table_init (pos < rope_max_pos)
 *   k_nope, v  as written by mla_decompress_kv (rows past kv_lens[b] up to the next
 *              multiple of 128 must be finite)
 *   cache ...  the cache holding the chunk (its RoPE keys k^R are read from it)
 *   out        [B, n_q, 128, 128] bf16 out; lse [B, n_q, 128] float32 out (nullable,
 *              natural log-sum-exp of the scaled scores)
 * n_q is not limited to MLA_MAX_NQ here.  A sequence whose lengths are
 * inconsistent sets MLA_ERR_BOUNDS and gets zeros.
 */
mla_status mla_decompress_kv(const mla_bf16* cache, int64_t num_pages, const int32_t* page_table, int pt_stride,
                             const int32_t* kv_lens, int B, int max_kv_len, const mla_bf16* w_uk,
                             const mla_bf16* w_uv, mla_bf16* k_nope, mla_bf16* v, cudaStream_t stream);
mla_status mla_prefill_attn(const mla_bf16* q_nope, const mla_bf16* q_rope, const int32_t* seq_lens_before,
                            const float* rope_table, int rope_max_pos, const mla_bf16* k_nope, const mla_bf16* v,
                            int max_kv_len, const mla_bf16* cache, int64_t num_pages, const int32_t* page_table,
                            int pt_stride, const int32_t* kv_lens, int B, int n_q, mla_bf16* out, float* lse,
                            cudaStream_t stream);

/*
 * mla_selftest_wait_timeout -- exercises the failure path of the bounded waits
 * every kernel uses (no counterpart on the MLA pages).  One warp waits on an
 * mbarrier that nothing completes; after limit_ns nanoseconds (1 .. 2e9) of
 * %globaltimer the wait gives up, MLA_ERR_TIMEOUT is recorded in the device
 * status word and the kernel returns: the context stays usable and the next
 * mla_get_device_status reports (and clears) the code.  Nothing faults, traps
 * or hangs.  Asynchronous on `stream`.
 */
mla_status mla_selftest_wait_timeout(int64_t limit_ns, cudaStream_t stream);

/*
 * mla_copy_async -- copy `bytes` from src to dst with the GPU's own loads and
 * stores, as one kernel of this library on `stream`.  (The MLA pages have no
 * counterpart; this moves a step's inputs and outputs.)  Each of dst and src
 * is device memory of the current device, managed memory, or pinned host
 * memory mapped into the device's address space (cudaHostAlloc /
 * cudaHostRegister on a unified-address system: on an NVLink-C2C machine the
 * GPU reads and writes it at link speed); the whole range [p, p + bytes) must
 * lie inside one such allocation, and the two ranges must not overlap, else
 * MLA_ERR_INVALID_ARG (pageable host memory is refused).  Any alignment (16-
 * byte aligned pointers take the vector path).  Ordered on the stream like the
 * other calls and part of the launch-overlap chain (mla_set_launch_overlap):
 * at level 2 a host-memory source is read before the previous kernel of the
 * stream has completed, so the caller must not change it after enqueueing.
 * bytes == 0 does nothing.
 */
mla_status mla_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/*
 * mla_set_launch_overlap / mla_get_launch_overlap -- how consecutive launches
 * of this library on one stream may overlap.  (The MLA pages have no
 * counterpart; this is a launch-latency setting of the GPU runtime.)
 *
 *   0  plain stream order: a kernel starts after the previous one has finished.
 *   1  (default) programmatic dependent launch: a kernel may be scheduled while
 *      the previous kernel of its stream drains and set up its shared memory,
 *      barriers and tensor memory; it reads or writes global memory only after
 *      that kernel has completed and its writes are visible.  Same results and
 *      the same ordering guarantees as 0.
 *   2  as 1, and the weight matrices w_uk (mla_absorb_q) and w_uv
 *      (mla_out_absorb, mla_combine_out_absorb) are read BEFORE the previous
 *      kernel has completed.  Only valid while no work still running on the
 *      stream writes those weights (fixed inference weights).  Likewise
 *      mla_copy_async reads a host-memory source before that point.
 *
 * The level is process-wide and read at each launch.  MLA_ERR_INVALID_ARG for a
 * level outside 0..2.  A launch whose predecessor on the stream is not a kernel
 * (a copy, an event wait) is ordered as in level 0.
 */
mla_status mla_set_launch_overlap(int level);
int mla_get_launch_overlap(void);

/*
 * Device status: synchronizes `stream`, returns the first fault code any kernel
 * of this library recorded on the current device since the last call
 * (MLA_OK if none) and clears it.  MLA_ERR_CUDA if the synchronisation fails.
 */
mla_status mla_get_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
