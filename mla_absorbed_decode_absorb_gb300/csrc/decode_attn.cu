// Split-KV absorbed attention over the paged latent cache (tcgen05, 2-CTA clusters).
//
// Per (sequence b, query j, split s) and head h, over the split's visible tokens t:
//   score_t = (q_abs[h,0:512] . c_t + q_abs[h,512:576] . kR_t) / sqrt(192)
//   O'_s[h] = sum_t softmax(score)_t c_t,   lse_s[h] = log sum_t exp(score_t)
// ("MLA 矩阵吸收 …" section 4.1: score = Q'_nope c^T + Q_rope k_rope^T, and the
//  V-side absorption O' = softmax . c; "DeepSeek-MLA-Principle" section 2: scale
//  1/sqrt(d_h + d_h^R), eq. (10); FlashMLA point 3: online softmax by block,
//  split-KV; point 4: paged cache.)
//
// All 128 heads share one latent key/value row per token, so the 128 heads are
// the M = 128 rows of both tensor-core contractions: S = Q c^T (K = 576) and
// O' += P c (K = 64 tokens per page).  One cluster of two CTAs handles one
// (sequence, query, split) unit; CTA r in {0, 1}:
//   * owns latent columns [256r, 256r + 256) of O' (256 fp32 TMEM columns);
//   * loads only its 288 columns of each 64-token page: latent [256r, 256r+256)
//     and RoPE [32r, 32r + 32), i.e. 36 KB per page instead of 72 KB;
//   * computes the partial score over those 288 columns and swaps partial S
//     (128 x 64 fp32) with its peer through distributed shared memory, so both
//     CTAs hold the same full S = S_0 + S_1 (bitwise equal: fp addition commutes);
//   * runs the same online softmax as its peer on that S, so both use identical
//     P, running max and sum, and accumulates its half of O' = P c.
// Warp roles: warp 0 issues TMA loads (the query tile once, then a 3-stage ring
// of half-pages; page ids are prefetched 32 at a time), warp 1 allocates TMEM
// and issues tcgen05.mma (QK^T into one of two TMEM score buffers; P V with P
// read from TMEM), warps 6-9 are the exchange warpgroup (per page: read the
// partial scores, swap them with the peer, write the full scores back into
// TMEM), warps 2-5 are the softmax/epilogue warpgroup.  Both warpgroups have one
// thread per head row, and the exchange for page i+1 overlaps the softmax of
// page i.  The softmax keeps a lazily updated reference max: O' in TMEM is
// rescaled only when a page raises a row's max by more than 2^8.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kExchangeWarp0 = 6;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O' half: [0, 256)
constexpr uint32_t kTmemS = 256;  // two score buffers: [256, 320), [320, 384); P aliases their first 32 columns

constexpr int kQChunk = 128 * 128;    // 64 latent columns x 128 heads, 128-byte rows
constexpr int kQRope = 128 * 64;      // 32 RoPE columns x 128 heads, 64-byte rows
constexpr int kQBytes = 4 * kQChunk + kQRope;
constexpr int kPChunk = 64 * 128;     // 64 latent columns x 64 tokens
constexpr int kPRope = 64 * 64;       // 32 RoPE columns x 64 tokens
constexpr int kStageBytes = 4 * kPChunk + kPRope;
constexpr int kXStride = 68;          // floats per exchanged score row (64 + 4 pad: conflict-free v4 access)
constexpr int kXBytes = kSoftmaxThreads * kXStride * 4;
constexpr uint32_t kXTxBytes = kSoftmaxThreads * 64 * 4;

constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kQBytes;
constexpr int kOffX = kOffStage + kStages * kStageBytes;
constexpr int kOffBar = kOffX + kXBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers + 1 KB alignment slack

constexpr float kRescaleLog2 = 8.f;

struct Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full;
  uint64_t s_full[2];   // partial scores of this CTA are in TMEM
  uint64_t s_ready[2];  // full scores are in TMEM
  uint64_t p_full[2];
  uint64_t pv_done;
  uint64_t x_full;
  uint64_t x_free;
  uint64_t x_read;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  float* o_out;
  float* lse_out;
  int* status;
  int64_t num_pages;
  int pt_stride;
  int n_q;
  int max_kv_len;
  int split_pages;
  int num_splits;
};

__device__ __forceinline__ uint32_t bar_addr(uint64_t& b) { return smem_u32(&b); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q128, const __grid_constant__ CUtensorMap tm_q64,
                      const __grid_constant__ CUtensorMap tm_c128, const __grid_constant__ CUtensorMap tm_c64,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int bj = unit / p.num_splits;
  const int split = unit % p.num_splits;
  const int b = bj / p.n_q, j = bj % p.n_q;

  // The unit's token range [t_begin, t_end): identical in both CTAs of the cluster.
  const int kv = p.kv_lens[b];
  const bool bad = kv > p.max_kv_len || kv < p.n_q || (kv + kPage - 1) / kPage > p.pt_stride;
  const int t_begin = split * p.split_pages * kPage;
  const int t_end = bad ? t_begin : min(t_begin + p.split_pages * kPage, kv - p.n_q + j + 1);
  const int page_begin = t_begin / kPage;
  const int n_pages = t_end > t_begin ? (t_end + kPage - 1) / kPage - page_begin : 0;

  if (tid == 0) {
    if (bad && rank == 0) record_status(p.status, MLA_ERR_BOUNDS);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_addr(bars.full[s]), 1);
      mbar_init(bar_addr(bars.empty[s]), 1);
    }
    mbar_init(bar_addr(bars.q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr(bars.s_full[s]), 1);
      mbar_init(bar_addr(bars.s_ready[s]), kSoftmaxThreads);
      mbar_init(bar_addr(bars.p_full[s]), kSoftmaxThreads);
    }
    mbar_init(bar_addr(bars.pv_done), 1);
    mbar_init(bar_addr(bars.x_full), 1);
    mbar_init(bar_addr(bars.x_free), 1);
    mbar_init(bar_addr(bars.x_read), kSoftmaxThreads);  // the 128 exchange threads
    mbar_init(bar_addr(bars.drain), 1);
    bars.abort = 0;
    fence_mbar_init();
    // arm the first exchange phase: 32 KB of the peer's partial scores
    mbar_arrive_expect_tx(bar_addr(bars.x_full), kXTxBytes);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote traffic
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (n_pages > 0) {
      const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride + page_begin;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q128);
        tma_prefetch_desc(&tm_q64);
        tma_prefetch_desc(&tm_c128);
        tma_prefetch_desc(&tm_c64);
        const int q_row = bj * kHeads;
        const uint32_t qb = smem_u32(smem + kOffQ);
        mbar_arrive_expect_tx(bar_addr(bars.q_full), kQBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(qb + c * kQChunk, &tm_q128, 64 * (4 * rank + c), q_row, bar_addr(bars.q_full));
        tma_load_2d(qb + 4 * kQChunk, &tm_q64, kLatent + 32 * rank, q_row, bar_addr(bars.q_full));
      }
      // page ids, 32 per coalesced load, one chunk ahead
      int ids = lane < n_pages ? pt[lane] : 0;
      bool ok = true;
      for (int base = 0; base < n_pages && ok; base += 32) {
        const int next_i = base + 32 + lane;
        const int ids_next = next_i < n_pages ? pt[next_i] : 0;
        const int cnt = min(32, n_pages - base);
        for (int k = 0; k < cnt && ok; ++k) {
          const int i = base + k;
          int page = __shfl_sync(0xffffffffu, ids, k);
          if (lane == 0) {
            const int s = i % kStages;
            ok = mbar_wait(bar_addr(bars.empty[s]), ((i / kStages) & 1) ^ 1, p.status, abort);
            if (ok) {
              if (page < 0 || page >= p.num_pages) {
                record_status(p.status, MLA_ERR_BOUNDS);
                page = 0;  // stay in bounds; the result of this unit is not meaningful
              }
              const uint32_t sb = smem_u32(smem + kOffStage + s * kStageBytes);
              const uint32_t fb = bar_addr(bars.full[s]);
              mbar_arrive_expect_tx(fb, kStageBytes);
              for (int c = 0; c < 4; ++c)
                tma_load_2d(sb + c * kPChunk, &tm_c128, 64 * (4 * rank + c), page * kPage, fb);
              tma_load_2d(sb + 4 * kPChunk, &tm_c64, kLatent + 32 * rank, page * kPage, fb);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        ids = ids_next;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    if (n_pages > 0) {
      const uint32_t idesc_qk = idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
      const uint32_t idesc_pv = idesc_bf16(128, 256, /*a_mn=*/0, /*b_mn=*/1);
      const uint32_t qb = smem_u32(smem + kOffQ);
      const int last_rows = t_end - (page_begin + n_pages - 1) * kPage;  // valid rows of the last page
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.q_full), 0, p.status, abort));

      auto issue_pv = [&](int i) -> bool {
        const bool w = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.p_full[i & 1]), (i >> 1) & 1, p.status, abort));
        if (!w) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sb = smem_u32(smem + kOffStage + (i % kStages) * kStageBytes);
          const uint32_t a = tmem + kTmemS + (i & 1) * 64;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + kTmemO, a + 8 * k, smem_desc(sb + 2048 * k, kPChunk, 1024, kSw128), idesc_pv,
                   (i > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar_addr(bars.empty[i % kStages]));
          mma_commit(bar_addr(bars.pv_done));
        }
        __syncwarp();
        return true;
      };

      for (int i = 0; i < n_pages && ok; ++i) {
        const int s = i % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.full[s]), (i / kStages) & 1, p.status, abort));
        if (!ok) break;
        uint8_t* stage = smem + kOffStage + s * kStageBytes;
        if (i == n_pages - 1 && last_rows < kPage) {
          // Rows past the last visible token may hold anything (NaN in unwritten
          // slots); zero their latent columns so P = 0 there cannot make 0 * NaN.
          const int nrow = kPage - last_rows;
          for (int v = lane; v < 4 * nrow * 8; v += 32) {
            const int c = v / (nrow * 8), r = last_rows + (v / 8) % nrow, u = v & 7;
            *reinterpret_cast<uint4*>(stage + c * kPChunk + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sb = smem_u32(stage);
          const uint32_t d = tmem + kTmemS + (i & 1) * 64;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(d, smem_desc(qb + c * kQChunk + 32 * k, 16, 1024, kSw128),
                     smem_desc(sb + c * kPChunk + 32 * k, 16, 1024, kSw128), idesc_qk, (c | k) ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ss(d, smem_desc(qb + 4 * kQChunk + 32 * k, 16, 512, kSw64),
                   smem_desc(sb + 4 * kPChunk + 32 * k, 16, 512, kSw64), idesc_qk, 1u);
          mma_commit(bar_addr(bars.s_full[i & 1]));
        }
        __syncwarp();
        if (i >= 1) ok = issue_pv(i - 1);
      }
      if (ok) issue_pv(n_pages - 1);
      // no tcgen05 operation may still be running when TMEM is released
      if (lane == 0) mma_commit(bar_addr(bars.drain));
      __syncwarp();
      mbar_wait(bar_addr(bars.drain), 0, p.status, nullptr);
    }
  } else if (warp >= kExchangeWarp0) {
    // ------------------------------------------------------------ score exchange
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // head
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float* xrow = reinterpret_cast<float*>(smem + kOffX) + row * kXStride;
    const uint32_t x_remote = mapa(smem_u32(xrow), peer);
    const uint32_t xfull_remote = mapa(bar_addr(bars.x_full), peer);
    const uint32_t xfree_remote = mapa(bar_addr(bars.x_free), peer);
    bool ok = true;
    for (int i = 0; i < n_pages && ok; ++i) {
      const int buf = i & 1;
      const uint32_t s_addr = tmem + lane_off + kTmemS + buf * 64;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.s_full[buf]), (i >> 1) & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv0[32], sv1[32];
      tmem_ld32(s_addr, sv0);
      tmem_ld32(s_addr + 32, sv1);
      tmem_wait_ld();
      // send this CTA's partial scores to the peer
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_free), (i & 1) ^ 1, p.status, abort));
      if (!ok) break;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        st_async_v4(x_remote + 16 * q, sv0[4 * q], sv0[4 * q + 1], sv0[4 * q + 2], sv0[4 * q + 3], xfull_remote);
        st_async_v4(x_remote + 128 + 16 * q, sv1[4 * q], sv1[4 * q + 1], sv1[4 * q + 2], sv1[4 * q + 3],
                    xfull_remote);
      }
      // receive the peer's partial scores and add them
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_full), i & 1, p.status, abort));
      if (!ok) break;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = reinterpret_cast<const float4*>(xrow)[q];
        const float4 y = reinterpret_cast<const float4*>(xrow)[q + 8];
        sv0[4 * q + 0] = __float_as_uint(__uint_as_float(sv0[4 * q + 0]) + x.x);
        sv0[4 * q + 1] = __float_as_uint(__uint_as_float(sv0[4 * q + 1]) + x.y);
        sv0[4 * q + 2] = __float_as_uint(__uint_as_float(sv0[4 * q + 2]) + x.z);
        sv0[4 * q + 3] = __float_as_uint(__uint_as_float(sv0[4 * q + 3]) + x.w);
        sv1[4 * q + 0] = __float_as_uint(__uint_as_float(sv1[4 * q + 0]) + y.x);
        sv1[4 * q + 1] = __float_as_uint(__uint_as_float(sv1[4 * q + 1]) + y.y);
        sv1[4 * q + 2] = __float_as_uint(__uint_as_float(sv1[4 * q + 2]) + y.z);
        sv1[4 * q + 3] = __float_as_uint(__uint_as_float(sv1[4 * q + 3]) + y.w);
      }
      // once every row has read the exchange buffer, one thread re-arms it and
      // tells the peer it may send the next page's partial scores
      mbar_arrive(bar_addr(bars.x_read));
      if (row == 0) {
        ok = mbar_wait(bar_addr(bars.x_read), i & 1, p.status, abort);
        if (ok) {
          mbar_arrive_expect_tx(bar_addr(bars.x_full), kXTxBytes);
          mbar_arrive_remote(xfree_remote);
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // full scores back into the same TMEM buffer for the softmax warpgroup
      tmem_st32(s_addr, sv0);
      tmem_st32(s_addr + 32, sv1);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(bars.s_ready[buf]));
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // head
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t out_row = (static_cast<int64_t>(bj) * p.num_splits + split) * kHeads + row;
    float* orow = p.o_out + out_row * kLatent + rank * 256;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = n_pages > 0;

    if (ok) {
      for (int i = 0; i < n_pages && ok; ++i) {
        const int buf = i & 1;
        const uint32_t s_addr = tmem + lane_off + kTmemS + buf * 64;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.s_ready[buf]), (i >> 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
        // raw-score row max over the visible tokens (the scale is positive)
        const int n_valid = min(kPage, t_end - (page_begin + i) * kPage);
        float mx = -INFINITY;
        if (n_valid == kPage) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mx = fmaxf(mx, __uint_as_float(sv[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < n_valid) mx = fmaxf(mx, __uint_as_float(sv[c]));
        }
        mx *= kScaleLog2;
        float factor = 1.f;
        bool rescale = false;
        if (i == 0) {
          m_ref = mx;
        } else if (mx > m_ref + kRescaleLog2) {
          factor = ex2_approx(m_ref - mx);
          m_ref = mx;
          rescale = true;
        }
        const float neg_m = -m_ref;
        uint32_t pk[32];
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * c]), kScaleLog2, neg_m));
          float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * c + 1]), kScaleLog2, neg_m));
          if (2 * c >= n_valid) p0 = 0.f;
          if (2 * c + 1 >= n_valid) p1 = 0.f;
          pk[c] = pack_bf16x2(p0, p1);
          sum += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
        }
        l = l * factor + sum;
        // O' may only be touched once the previous P V has finished
        if (i >= 1) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done), (i - 1) & 1, p.status, abort));
          if (!ok) break;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale)) {
          for (int c0 = 0; c0 < 256; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + kTmemO + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * factor);
            tmem_st32(tmem + lane_off + kTmemO + c0, r);
          }
        }
        tmem_st32(s_addr, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_addr(bars.p_full[buf]));
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done), (n_pages - 1) & 1, p.status, abort));
      tc_fence_after();
    }
    // epilogue: this CTA's 256 columns of O' (normalised) and the row's log-sum-exp
    if (ok) {
      const float inv = 1.f / l;
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kTmemO + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(orow + c0 + 4 * q) =
              make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                          __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
      }
      if (rank == 0 && p.lse_out != nullptr) p.lse_out[out_row] = (m_ref + log2f(l)) * kLn2;
    } else {
      for (int c0 = 0; c0 < 256; c0 += 4) *reinterpret_cast<float4*>(orow + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rank == 0 && p.lse_out != nullptr) p.lse_out[out_row] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // no CTA leaves while its peer may still address its shared memory
}

int g_cluster_slots[64];
bool g_configured[64];

bool configure(int dev) {
  if (dev < 0 || dev >= 64) return false;
  if (!g_configured[dev]) {
    if (cudaFuncSetAttribute(decode_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return false;
    g_configured[dev] = true;
  }
  return true;
}

}  // namespace

int decode_cluster_slots() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 74;
  if (g_cluster_slots[dev] > 0) return g_cluster_slots[dev];
  int n = 0;
  if (configure(dev)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, decode_attn_tc_kernel, &cfg) != cudaSuccess) n = 0;
  }
  if (n <= 0) {
    cudaGetLastError();
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms / 2;
  }
  g_cluster_slots[dev] = n;
  return n;
}

cudaError_t launch_decode_partial(const uint16_t* q_abs, const uint16_t* cache,
                                  int64_t num_pages, const int32_t* page_table, int pt_stride,
                                  const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                  const SplitPlan& plan, float* o_out, float* lse_out,
                                  int* status, cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(B) * n_q * plan.num_splits;
  if (units == 0) return cudaSuccess;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || !configure(dev)) return cudaErrorInvalidDevice;
  CUtensorMap tq128, tq64, tc128, tc64;
  const uint64_t q_rows = static_cast<uint64_t>(B) * n_q * kHeads;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  if (!make_tmap_bf16_2d(&tq128, q_abs, q_rows, kRow, kRow, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&tq64, q_abs, q_rows, kRow, kRow, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_bf16_2d(&tc128, cache, c_rows, kRow, kRow, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&tc64, cache, c_rows, kRow, kRow, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.o_out = o_out;
  prm.lse_out = lse_out;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.n_q = n_q;
  prm.max_kv_len = max_kv_len;
  prm.split_pages = plan.split_pages;
  prm.num_splits = plan.num_splits;
  decode_attn_tc_kernel<<<static_cast<unsigned>(2 * units), kThreads, kSmemBytes, stream>>>(tq128, tq64, tc128, tc64,
                                                                                           prm);
  return cudaGetLastError();
}

}  // namespace mla
