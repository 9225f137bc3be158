// Value up-projection applied once to the latent output: O[t,h,d] = sum_m O'[t,h,m] W_UV[h,d,m],
// optionally preceded by the split-KV log-sum-exp merge that produces O'.
//
// "MLA 矩阵吸收 …" section 2.1, V side (O = (Attn c) W_UV, done once, independent
// of the history length); "DeepSeek-MLA-Principle" value absorption
// o = W_UV[h] m; "DeepSeek MLA 架构详解" step 5 (einsum 'bhm,hdm->bhd').
// The merge is the one of FlashMLA point 3 ("DeepSeek-MLA-Principle"): with
// split outputs O'_s normalised within their split and natural log-sum-exps
// lse_s, lse = log sum_s exp(lse_s) and O' = sum_s exp(lse_s - lse) O'_s.
//
// tcgen05 version, operands swapped so the large side is M: per head h the CTA
// computes D[d, t] = sum_m W_UV[h][d][m] * O'[t][h][m] with the 128 output
// dimensions d as M and up to 64 query tokens as N.  Both operands are K-major
// (m contiguous).  All of W_UV[h] (128 KB) is requested at once, as eight TMA
// boxes of 64 m x 128 d; while it is in flight the CTA builds O' (merging the
// splits in float32 with the same operations, in the same order, as the
// stand-alone merge kernel) and rounds it to bf16 into shared memory.  One
// chain of 32 MMAs (K = 16 each) accumulates in TMEM.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kNMax = 64;                          // query tokens per CTA
constexpr int kThreads = 256;
constexpr int kChunk = 128 * 128;                  // 128 rows x 64 m (128 B), SW128
constexpr int kSmemA = (kLatent / 64) * kChunk;    // W_UV[h]: 8 chunks, 128 KB

// Tokens of the widest tile (rounded up to the MMA's N granularity of 16), and
// the TMEM columns for its fp32 accumulator (a power of two, at least 32).
__host__ __device__ inline int tile_tokens(int T) { return (min(kNMax, T) + 15) & ~15; }
__host__ __device__ inline uint32_t tmem_cols_for(int nb) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(nb)) c <<= 1;
  return c;
}
constexpr int kTableSplits = 128;  // merge weights kept in shared memory up to this many splits
__host__ __device__ inline int smem_bytes_for(int T, int num_splits) {
  const int nb = tile_tokens(T);
  const int table = num_splits <= kTableSplits ? nb * num_splits : 0;
  return kSmemA + (kLatent / 64) * nb * 128 + 24 + 4 * (2 * kNMax + table) + 1024;
}

// src: O' rows; with src_lse == nullptr, row (t, h) is the fp32 row
// src[(t * 128 + h) * 512] (one source); otherwise num_splits partial rows in bf16,
// src[((t * S + s) * 128 + h) * 512], with log-sum-exps src_lse[(t * S + s) * 128 + h]
// are merged first, and the merged log-sum-exp goes to lse_out[t * 128 + h] (if non-null).
__global__ void __launch_bounds__(kThreads, 1)
out_absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const void* __restrict__ src,
                     const float* __restrict__ src_lse, int num_splits, uint16_t* __restrict__ out, float* __restrict__ lse_out,
                     int T, int* status, bool weights_early) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nb = tile_tokens(T);  // B and TMEM are sized for the widest token tile of this launch
  const uint32_t tmem_cols = tmem_cols_for(nb);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSmemA;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + (kLatent / 64) * nb * 128);
  uint64_t* wbar = bar + 1;                          // W_UV[h] has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  float* s_max = reinterpret_cast<float*>(bar + 3);  // per token: max_s lse_s
  float* s_inv = s_max + kNMax;                      // per token: 1 / sum_s exp(lse_s - max)
  float* s_w = s_inv + kNMax;                        // [token][split] weights (table mode)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kNMax;
  const int nt = min(kNMax, T - t0);
  const int npad = (nt + 15) & ~15;
  const int64_t S = num_splits;

  // A: W_UV[h][d][0 .. 512) -> 8 K-major chunks of 64 m, rows d, by TMA (all in
  // flight at once; possibly requested before the previous kernel has finished)
  auto load_w = [&]() {
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(wbar), kSmemA);
      for (int c = 0; c < kLatent / 64; ++c)
        tma_load_2d(smem_u32(sA + c * kChunk), &tm_w, 64 * c, h * kNope, smem_u32(wbar));
    }
  };
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    mbar_init(smem_u32(wbar), 1);
    fence_mbar_init();
  }
  if (weights_early) load_w();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  grid_dep_wait();
  grid_dep_launch();
  if (!weights_early) load_w();
  // Merge weights: w[t][s] = exp(lse_s - max_s lse_s) (-1 marks an empty split,
  // which is skipped), kept in shared memory for up to kTableSplits splits.
  // They are computed once the first split rows are in flight (the row loads
  // do not depend on them), so the two round trips to memory overlap.
  const bool table = num_splits <= kTableSplits;
  auto merge_weights = [&]() {
    if (tid < nt) {
      const float* ls = src_lse + (static_cast<int64_t>(t0 + tid) * S) * kHeads + h;
      float m = -INFINITY;
      for (int s = 0; s < num_splits; ++s) m = fmaxf(m, ls[s * kHeads]);
      float z = 0.f;
      if (m != -INFINITY)
        for (int s = 0; s < num_splits; ++s) {
          const float l = ls[s * kHeads];
          const float w = l == -INFINITY ? -1.f : expf(l - m);
          if (w >= 0.f) z += w;
          if (table) s_w[tid * num_splits + s] = w;
        }
      s_max[tid] = m;
      s_inv[tid] = 1.f / z;
      if (lse_out != nullptr) lse_out[static_cast<int64_t>(t0 + tid) * kHeads + h] = m == -INFINITY ? m : m + logf(z);
    }
    __syncthreads();
  };
  bool weights_ready = src_lse == nullptr;

  // B: O'[t0 + t][h][0 .. 512) rounded to bf16: 8 K-major chunks of 64, rows t
  // (zero past nt).  Thread (tq, u) = (tid / 64, tid % 64) builds 16-byte unit u
  // (8 consecutive m) of tokens t = tq + 4i, 8 tokens at a time; the rows of
  // two splits (32 loads) are in flight together.
  const int u = tid & 63, tq = tid >> 6;
  for (int i0 = 0; i0 < npad / 4; i0 += 8) {
    float4 a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = b[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (src_lse == nullptr) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = tq + 4 * (i0 + k);
        if (t < nt) {
          const float4* p =
              reinterpret_cast<const float4*>(static_cast<const float*>(src) + (static_cast<int64_t>(t0 + t) * kHeads + h) * kLatent) +
              2 * u;
          a[k] = p[0];
          b[k] = p[1];
        }
      }
    } else {
      for (int s0 = 0; s0 < num_splits; s0 += 2) {
        float4 x[2][8], y[2][8];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int t = tq + 4 * (i0 + k);
            x[j][k] = y[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < nt && s0 + j < num_splits) {
              const int64_t r = (static_cast<int64_t>(t0 + t) * S + s0 + j) * kHeads + h;
              const uint4 q = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + r * kLatent)[u];
              x[j][k] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                    __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
              y[j][k] = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xffff0000u),
                                    __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xffff0000u));
            }
          }
        if (!weights_ready) {
          merge_weights();
          weights_ready = true;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int t = tq + 4 * (i0 + k);
            const int s = s0 + j;
            float w = -1.f;
            if (t < nt && s < num_splits && s_max[t] != -INFINITY) {
              if (table) {
                w = s_w[t * num_splits + s];
              } else {
                const float l = src_lse[(static_cast<int64_t>(t0 + t) * S + s) * kHeads + h];
                w = l == -INFINITY ? -1.f : expf(l - s_max[t]);
              }
            }
            if (w >= 0.f) {
              a[k].x = fmaf(w, x[j][k].x, a[k].x); a[k].y = fmaf(w, x[j][k].y, a[k].y);
              a[k].z = fmaf(w, x[j][k].z, a[k].z); a[k].w = fmaf(w, x[j][k].w, a[k].w);
              b[k].x = fmaf(w, y[j][k].x, b[k].x); b[k].y = fmaf(w, y[j][k].y, b[k].y);
              b[k].z = fmaf(w, y[j][k].z, b[k].z); b[k].w = fmaf(w, y[j][k].w, b[k].w);
            }
          }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = tq + 4 * (i0 + k);
        if (t < nt && s_max[t] != -INFINITY) {
          const float inv = s_inv[t];
          a[k].x *= inv; a[k].y *= inv; a[k].z *= inv; a[k].w *= inv;
          b[k].x *= inv; b[k].y *= inv; b[k].z *= inv; b[k].w *= inv;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = tq + 4 * (i0 + k);
      if (t < npad)
        *reinterpret_cast<uint4*>(sB + (u >> 3) * npad * 128 + sw128(t * 128 + (u & 7) * 16)) =
            make_uint4(pack_bf16x2(a[k].x, a[k].y), pack_bf16x2(a[k].z, a[k].w), pack_bf16x2(b[k].x, b[k].y),
                       pack_bf16x2(b[k].z, b[k].w));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool wok = true;
  if (tid == 0) wok = mbar_wait(smem_u32(wbar), 0, status);  // W_UV[h] has landed
  if (tid == 0 && wok) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16(128, npad, /*a_mn=*/0, /*b_mn=*/0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
    for (int k = 0; k < kLatent / 16; ++k) {
      const uint64_t ad = smem_desc(a0 + (k >> 2) * kChunk + (k & 3) * 32, 16, 1024, kSw128);
      const uint64_t bd = smem_desc(b0 + (k >> 2) * npad * 128 + (k & 3) * 32, 16, 1024, kSw128);
      mma_ss(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
    }
    mma_commit(smem_u32(bar));
  }
  if (tid == 0 && !wok) mbar_arrive(smem_u32(bar));  // no MMA: release the waiters (the result is flagged)
  const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), 0, status));
  tc_fence_after();

  if (ok) {
    // warp w reads TMEM lanes 32 (w % 4) .. + 32 (d), columns (tokens) of half w / 4
    const int d = (warp & 3) * 32 + lane;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    for (int c0 = (warp >> 2) * 16; c0 < npad; c0 += 32) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = c0 + i;
        if (t < nt) out[(static_cast<int64_t>(t0 + t) * kHeads + h) * kNope + d] = f32_to_bf16_bits(__uint_as_float(r[i]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ------------------------------------------------------------------ streamed variant
// For up to kTMaxSplits splits the O' rows come in by TMA as well: a plain
// load of 128 KB per CTA is limited by what L1 can hold in flight next to the
// 128 KB of W_UV in shared memory, while a TMA box lands in shared memory
// directly.  Per CTA (head h, up to kTTokens tokens), latent chunk k (64 m)
// travels through a 5-slot ring as W_UV[h]'s chunk k (a 64 m x 128 d box) and the
// rows (token t, split s) of O' (one box of up to 128 bf16 partial rows, or of
// up to 32 fp32 rows of a single source): the first five
// weight chunks are requested before the previous kernel has finished (where
// the launch allows) and the last three pulled into L2, so that the O' of five
// chunks is in flight at once (two round trips to L2 for the tile, where a
// 3-slot ring of O' beside all of W_UV needed three).  8 combine warps merge
// chunk k (same fp32 operations in the same order as the stand-alone merge) into
// bf16 chunk k of B, and warp 8 issues the chunk's 4 MMAs as soon as it is
// written, then refills the slot once they have finished.
constexpr int kTTokens = 32;                   // tokens per CTA (at most)
constexpr int kTBoxRows = 128;                 // O' rows (token x split) per box
constexpr int kTStages = 5;
constexpr int kTBoxBytes = 64 * 2 * kTBoxRows;  // 16 KB: 128 rows of 64 bf16 partial values
static_assert(kTTokens * 64 * 4 <= kTBoxBytes, "a single source's fp32 rows (one per token) fit the box");
constexpr int kTSlotBytes = kChunk + kTBoxBytes;  // W_UV chunk, then the O' box
constexpr int kTThreads = 288;                 // warps 0-7 merge, warp 8 loads and issues MMAs
constexpr int kTMaxSplits = 16;
constexpr int kTSmemB = (kLatent / 64) * kTTokens * 128;  // 32 KB

struct TBars {
  uint64_t w_full[kTStages];      // the slot's weight chunk has landed
  uint64_t p_full[kTStages];      // the slot's O' box has landed
  uint64_t s_free[kTStages];      // the MMAs of the slot's chunk have finished (its weights are read)
  uint64_t b_full[kLatent / 64];  // chunk k of B written (and box k read) by all 256 merge threads
  uint64_t mma_done;
  uint32_t tmem_slot;
};
constexpr int kTOffRing = 0;
constexpr int kTOffB = kTOffRing + kTStages * kTSlotBytes;
constexpr int kTOffBars = kTOffB + kTSmemB;
constexpr int kTOffTab = kTOffBars + 256;
constexpr int kTSmemBytes = kTOffTab + 4 * (kTTokens * kTMaxSplits + 2 * kTTokens) + 1024;
static_assert(sizeof(TBars) <= 256, "barrier block");
static_assert(kTSmemBytes <= 232448, "shared memory budget");

// Tokens per CTA for S splits: whole tokens' rows fit one box (S = 1: at most
// kTTokens fp32 rows).
__host__ __device__ inline int t_tile(int S) { return min(kTTokens, kTBoxRows / S); }

__global__ void __launch_bounds__(kTThreads, 1)
out_absorb_stream_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
                         const float* __restrict__ src_lse, int num_splits, uint16_t* __restrict__ out,
                         float* __restrict__ lse_out, int T, int* status, bool weights_early) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem + kTOffB;
  uint8_t* ring = smem + kTOffRing;
  TBars& bars = *reinterpret_cast<TBars*>(smem + kTOffBars);
  float* s_w = reinterpret_cast<float*>(smem + kTOffTab);  // [token][split] merge weights
  float* s_inv = s_w + kTTokens * kTMaxSplits;            // per token: 1 / sum_s w
  float* s_max = s_inv + kTTokens;                        // per token: max_s lse_s

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = num_splits;
  const int ntile = t_tile(S);
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * ntile;
  const int nt = min(ntile, T - t0);
  const int npad = (nt + 15) & ~15;
  const uint32_t tmem_cols = 32;  // npad <= 32
  const bool merge = src_lse != nullptr;

  constexpr int kNChunks = kLatent / 64;
  // weight chunk k (64 m x 128 d) into slot k % kTStages
  auto load_w = [&](int k) {
    const int slot = k % kTStages;
    mbar_arrive_expect_tx(smem_u32(&bars.w_full[slot]), kChunk);
    tma_load_2d(smem_u32(ring + slot * kTSlotBytes), &tm_w, 64 * k, h * kNope, smem_u32(&bars.w_full[slot]));
  };
  auto load_w_first = [&]() {
    for (int k = 0; k < kTStages; ++k) load_w(k);
    for (int k = kTStages; k < kNChunks; ++k) tma_prefetch_l2_2d(&tm_w, 64 * k, h * kNope);
  };
  // box k: rows (t0 + t) * S + s, t < ntile, columns [64k, 64k + 64) of head h
  const uint32_t prow_bytes = merge ? 128u : 256u;  // 64 columns of a bf16 partial row, or of an fp32 O' row
  auto load_p = [&](int k) {
    const int slot = k % kTStages;
    mbar_arrive_expect_tx(smem_u32(&bars.p_full[slot]), prow_bytes * ntile * S);  // the whole box, rows past T * S as zeros
    tma_load_3d(smem_u32(ring + slot * kTSlotBytes + kChunk), &tm_p, 64 * k, h, t0 * S, smem_u32(&bars.p_full[slot]));
  };

  if (tid == 256) {
    for (int i = 0; i < kTStages; ++i) {
      mbar_init(smem_u32(&bars.w_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), 1);
      mbar_init(smem_u32(&bars.s_free[i]), 1);
    }
    for (int i = 0; i < kNChunks; ++i) mbar_init(smem_u32(&bars.b_full[i]), 256);
    mbar_init(smem_u32(&bars.mma_done), 1);
    fence_mbar_init();
    if (weights_early) load_w_first();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&bars.tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 8) {
    // ------------------------------------------------ loads and MMAs
    if (lane == 0) {
      if (!weights_early) load_w_first();
      for (int k = 0; k < kTStages; ++k) load_p(k);
      const uint32_t idesc = idesc_bf16(128, npad, /*a_mn=*/0, /*b_mn=*/0);
      const uint32_t b0 = smem_u32(sB);
      bool ok = true;
      for (int k = 0; k < kNChunks && ok; ++k) {
        const int slot = k % kTStages;
        const uint32_t use = (k / kTStages) & 1;
        ok = mbar_wait(smem_u32(&bars.w_full[slot]), use, status) && mbar_wait(smem_u32(&bars.b_full[k]), 0, status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + slot * kTSlotBytes);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t ad = smem_desc(a0 + q * 32, 16, 1024, kSw128);
          const uint64_t bd = smem_desc(b0 + k * npad * 128 + q * 32, 16, 1024, kSw128);
          mma_ss(tmem, ad, bd, idesc, (k | q) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.s_free[slot]));
        if (k + kTStages < kNChunks) {
          // box k has been merged (b_full); the slot is free once these MMAs have read its weights
          ok = mbar_wait(smem_u32(&bars.s_free[slot]), use, status);
          if (!ok) break;
          load_w(k + kTStages);
          load_p(k + kTStages);
        }
      }
      if (ok) mma_commit(smem_u32(&bars.mma_done));
      else mbar_arrive(smem_u32(&bars.mma_done));  // no result: release the epilogue (the status is set)
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ merge: thread (t, u) = 8 m of token t
    const int t = tid >> 3, u = tid & 7;
    if (merge && tid < nt) {
      const float* ls = src_lse + (static_cast<int64_t>(t0 + tid) * S) * kHeads + h;
      float m = -INFINITY;
      for (int s = 0; s < S; ++s) m = fmaxf(m, ls[s * kHeads]);
      float z = 0.f;
      if (m != -INFINITY)
        for (int s = 0; s < S; ++s) {
          const float l = ls[s * kHeads];
          const float w = l == -INFINITY ? -1.f : expf(l - m);
          if (w >= 0.f) z += w;
          s_w[tid * S + s] = w;
        }
      s_max[tid] = m;
      s_inv[tid] = 1.f / z;
      if (lse_out != nullptr) lse_out[static_cast<int64_t>(t0 + tid) * kHeads + h] = m == -INFINITY ? m : m + logf(z);
    }
    named_barrier_sync(1, 256);
    const bool live = t < nt && (!merge || s_max[t] != -INFINITY);
    for (int k = 0; k < kLatent / 64; ++k) {
      const int slot = k % kTStages;
      mbar_wait(smem_u32(&bars.p_full[slot]), (k / kTStages) & 1, status);
      if (t < npad) {
        float a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = 0.f;
        if (live) {
          const uint8_t* box = ring + slot * kTSlotBytes + kChunk;
          for (int s = 0; s < S; ++s) {
            const float w = merge ? s_w[t * S + s] : 1.f;
            if (w >= 0.f) {
              float4 x, y;
              if (merge) {
                const uint4 q = *reinterpret_cast<const uint4*>(box + (t * S + s) * 128 + u * 16);
                x = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
                y = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xffff0000u),
                                __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xffff0000u));
              } else {
                const float4* r = reinterpret_cast<const float4*>(box + (t * S + s) * 256 + u * 32);
                x = r[0];
                y = r[1];
              }
              a[0] = fmaf(w, x.x, a[0]); a[1] = fmaf(w, x.y, a[1]); a[2] = fmaf(w, x.z, a[2]); a[3] = fmaf(w, x.w, a[3]);
              a[4] = fmaf(w, y.x, a[4]); a[5] = fmaf(w, y.y, a[5]); a[6] = fmaf(w, y.z, a[6]); a[7] = fmaf(w, y.w, a[7]);
            }
          }
          if (merge) {
            const float inv = s_inv[t];
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] *= inv;
          }
        }
        *reinterpret_cast<uint4*>(sB + k * npad * 128 + sw128(t * 128 + u * 16)) =
            make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.b_full[k]));
    }
    // ------------------------------------------------ epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 32 (d),
    // columns (tokens) of half w / 4
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.mma_done), 0, status));
    tc_fence_after();
    if (ok) {
      const int d = (warp & 3) * 32 + lane;
      const uint32_t row_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      for (int c0 = (warp >> 2) * 16; c0 < npad; c0 += 32) {
        uint32_t r[16];
        tmem_ld16(row_addr + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int tt = c0 + i;
          if (tt < nt) out[(static_cast<int64_t>(t0 + tt) * kHeads + h) * kNope + d] = f32_to_bf16_bits(__uint_as_float(r[i]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) tmem_dealloc(tmem, tmem_cols);
}

cudaError_t launch_stream(const void* src, const float* src_lse, int num_splits, const uint16_t* w_uv, uint16_t* out,
                          float* lse_out, int T, int* status, cudaStream_t stream) {
  static bool configured[kMaxDevicesLocal] = {};  // the attribute is per device
  const int dev_ = current_device_index();
  if (dev_ < 0) return cudaErrorInvalidDevice;
  if (!configured[dev_]) {
    cudaError_t e = cudaFuncSetAttribute(out_absorb_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev_] = true;
  }
  CUtensorMap tw, tp;
  const int S = num_splits;
  const int ntile = t_tile(S);
  // W_UV as a [128 * 128, 512] matrix: box 64 columns x 128 rows, 128-byte swizzle;
  // O' rows as [T * S][128 heads][512] (bf16 partials when merging, else fp32): box
  // 64 columns x 1 head x (ntile * S) rows
  const uint64_t rows = static_cast<uint64_t>(T) * S;
  const bool merge = src_lse != nullptr;
  if (!merge && S != 1) return cudaErrorInvalidValue;  // fp32 rows: one source only
  if (!make_tmap_bf16_2d(&tw, w_uv, static_cast<uint64_t>(kHeads) * kNope, kLatent, kLatent, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      (merge ? !make_tmap_bf16_3d(&tp, src, kLatent, kHeads, rows, kLatent * 2ull, static_cast<uint64_t>(kHeads) * kLatent * 2ull,
                                  64, 1, static_cast<uint32_t>(ntile * S), CU_TENSOR_MAP_SWIZZLE_NONE)
             : !make_tmap_f32_3d(&tp, src, kLatent, kHeads, rows, kLatent * 4ull, static_cast<uint64_t>(kHeads) * kLatent * 4ull,
                                 64, 1, static_cast<uint32_t>(ntile * S))))
    return cudaErrorInvalidValue;
  dim3 grid(kHeads, (T + ntile - 1) / ntile);
  return launch_kernel(out_absorb_stream_kernel, grid, dim3(kTThreads), kTSmemBytes, stream, tw, tp, src_lse,
                       num_splits, out, lse_out, T, status, launch_overlap() >= 2);
}

cudaError_t launch(const void* src, const float* src_lse, int num_splits, const uint16_t* w_uv, uint16_t* out,
                   float* lse_out, int T, int* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (num_splits <= kTMaxSplits && (reinterpret_cast<uintptr_t>(src) & 15u) == 0)
    return launch_stream(src, src_lse, num_splits, w_uv, out, lse_out, T, status, stream);
  static bool configured[kMaxDevicesLocal] = {};  // the attribute is per device
  const int dev_ = current_device_index();
  if (dev_ < 0) return cudaErrorInvalidDevice;
  if (!configured[dev_]) {
    cudaError_t e = cudaFuncSetAttribute(out_absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes_for(kNMax, kTableSplits));
    if (e != cudaSuccess) return e;
    configured[dev_] = true;
  }
  // W_UV as a [128 * 128, 512] matrix: box 64 columns x 128 rows, 128-byte swizzle
  CUtensorMap tw;
  if (!make_tmap_bf16_2d(&tw, w_uv, static_cast<uint64_t>(kHeads) * kNope, kLatent, kLatent, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  dim3 grid(kHeads, (T + kNMax - 1) / kNMax);
  return launch_kernel(out_absorb_tc_kernel, grid, dim3(kThreads), smem_bytes_for(T, num_splits), stream, tw, src,
                       src_lse, num_splits, out, lse_out, T, status, launch_overlap() >= 2);
}

}  // namespace

cudaError_t launch_out_absorb(const float* o_latent, const uint16_t* w_uv, uint16_t* out, int B, int n_q,
                              int* status, cudaStream_t stream) {
  return launch(o_latent, nullptr, 1, w_uv, out, nullptr, B * n_q, status, stream);
}

cudaError_t launch_combine_out_absorb(const uint16_t* o_part, const float* lse_part, int num_splits,
                                      const uint16_t* w_uv, uint16_t* out, float* lse, int B, int n_q,
                                      int* status, cudaStream_t stream) {
  return launch(o_part, lse_part, num_splits, w_uv, out, lse, B * n_q, status, stream);
}

}  // namespace mla
