// Split-KV absorbed attention over an FP8 (E4M3) paged latent cache.
//
// The cache of this variant stores, per token t, the 512 latent values as E4M3
// codes of c_t / s_t with one float32 scale s_t, and the rotated key as float16
// of k^R_t / s_t (the pages name FP8, one byte per value, among the cache
// precisions together with a scaling strategy: "DeepSeek-MLA-Principle" section
// 7, "DeepSeek MLA 架构详解" on the KV-cache memory formula).  The attention is
// the one of the bf16 kernel on the dequantised values c_t = s_t E4M3(code) and
// k^R_t = s_t f16(stored):
//   score_t = (q_abs[h,0:512] . c_t + q_abs[h,512:576] . k^R_t) / sqrt(192)
//   O'_s[h] = sum_t softmax(score)_t c_t,   lse_s[h] = log sum_t exp(score_t)
//
// Both parts of the score carry the same factor 1 / s_t, so the MMAs run on
// the codes themselves: E4M3 values are exactly representable in float16, so
// a dequantisation warpgroup widens each page's codes to float16 (exact) into
// the stage the MMAs read, and the query goes in as float16 (kind::f16 with f16
// operands).  The row warps multiply the column's partial score by s_t (before
// the fp16 exchange, which then carries the same units as the bf16 kernel's),
// and give P V the operand P_t s_t, so that O' = sum_t p_t s_t E4M3(code_t).
//
// Pipeline per CTA (cluster of two, CTA r owns latent columns [256r, 256r+256)
// as in the bf16 kernel): warps 12-15 read each page's 16 KB of codes and 64
// scales straight from global memory into registers (issued before they wait
// for the stage; they run up to three pages ahead of the MMAs) and widen the
// codes into a 4-slot ring of float16 stages; warp 0
// loads the page's 4 KB of key by TMA into the stage (its layout is the
// stage's) and pulls the next page's codes into L2; warp 1 issues QK^T, warp 2
// P V, warp 3 recycles the exchange buffers, and warps 4-11 are the two row
// warpgroups.  Without a landing ring for the codes, four float16 stages fit.
// Score exchange, lazy reference max, packed softmax arithmetic, TMEM layout
// and epilogue follow the bf16 kernel.
#include <cuda_fp16.h>

#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 4;          // float16 stages the MMAs read
constexpr int kThreads = 512;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kPvWarp = 2;
constexpr int kSignalWarp = 3;
constexpr int kRowWarp0 = 4;        // warps 4-7: row warpgroup 0, warps 8-11: row warpgroup 1
constexpr int kDqWarp0 = 12;        // warps 12-15: dequantisation warpgroup
constexpr int kRowThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O' half: [0, 256)
constexpr uint32_t kTmemS = 256;    // score buffer of warpgroup g: [256 + 64g, 320 + 64g)
constexpr uint32_t kTmemQ = 384;    // the CTA's 256 latent query columns as f16 pairs: [384, 512)

constexpr int kQRope = 128 * 64;      // 32 RoPE query columns x 128 heads, 64-byte rows (SW64)
constexpr int kPChunk = 64 * 128;     // 64 latent columns x 64 tokens, f16 (SW128)
constexpr int kPRope = 64 * 64;       // 32 RoPE columns x 64 tokens, f16 (SW64)
constexpr int kStageBytes = 4 * kPChunk + kPRope;
constexpr int kXBufBytes = kRowThreads * 128;
constexpr uint32_t kXTxBytes = kXBufBytes;
constexpr float kSumScaleLog2 = kScaleLog2 * 256.f;
constexpr int kPBytes = kHeads * 128;

constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kQRope;
constexpr int kOffX = kOffStage + kStages * kStageBytes;
constexpr int kOffP = kOffX + 2 * kXBufBytes;
constexpr int kOffSc = kOffP + 2 * kPBytes;     // per stage: 64 x s_t / 256, then 64 x s_t
constexpr int kOffBar = kOffSc + kStages * 512;
constexpr int kOffMax = kOffBar + 256;          // per-row reference max handed between warpgroups
constexpr int kSmemBytes = kOffMax + 4 * kHeads + 1024;  // + 1 KB alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0 && kOffX % 1024 == 0 && kOffP % 1024 == 0,
              "swizzled tiles start on 1 KB");

constexpr float kRescaleLog2 = 8.f;
constexpr int kOBoxBytes = 128 * 128;
constexpr int kOTileBytes = 4 * kOBoxBytes;
static_assert(2 * kOTileBytes <= kOffX - kOffStage, "output staging fits in the stages");

struct Bars {
  uint64_t full[kStages];       // float16 stage written (128 dequantisation threads) and its key landed
  uint64_t empty[kStages];      // P V of the stage's page has finished
  uint64_t q_full;
  uint64_t q_tmem;
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t x_full[2];
  uint64_t x_free[2];
  uint64_t x_read[2];
  uint64_t hand[2];
  uint64_t fin;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int wg_bad[2];
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  const uint16_t* q_abs;
  const float* scale;          // [num_pages * 64]
  const uint8_t* c8;           // [num_pages * 64, 512] E4M3 codes
  void* o_out;   // fp32 O' (one split), or the splits' bf16 partials (out_bf16)
  int out_bf16;
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

// bf16 pair -> f16 pair (exact for |x| in [2^-14, 65504]; nearest even otherwise)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  const __half2 h = __floats2half2_rn(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// two E4M3 codes (low byte first) -> f16 pair, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_attn_fp8_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_c8,
                       const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_o,
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

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_addr(bars.full[s]), kRowThreads + 1);  // the 128 dequantisation threads + the key's load
      mbar_init(bar_addr(bars.empty[s]), 1);
    }
    mbar_init(bar_addr(bars.q_full), 1);
    mbar_init(bar_addr(bars.q_tmem), 2 * kRowThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr(bars.s_full[s]), 1);
      mbar_init(bar_addr(bars.s_free[s]), kRowThreads);
      mbar_init(bar_addr(bars.p_full[s]), kRowThreads);
      mbar_init(bar_addr(bars.pv_done[s]), 1);
      mbar_init(bar_addr(bars.x_full[s]), 1);
      mbar_init(bar_addr(bars.x_free[s]), 1);
      mbar_init(bar_addr(bars.x_read[s]), kRowThreads);
      mbar_init(bar_addr(bars.hand[s]), kRowThreads);
    }
    mbar_init(bar_addr(bars.fin), 2 * kRowThreads);
    mbar_init(bar_addr(bars.drain), 2);
    bars.abort = 0;
    bars.wg_bad[0] = bars.wg_bad[1] = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_addr(bars.x_full[0]), kXTxBytes);
    mbar_arrive_expect_tx(bar_addr(bars.x_full[1]), kXTxBytes);
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
  grid_dep_wait();
  grid_dep_launch();

  const int kv = p.kv_lens[b];
  const bool bad = kv > p.max_kv_len || kv < p.n_q || (kv + kPage - 1) / kPage > p.pt_stride;
  const int t_begin = split * p.split_pages * kPage;
  const int t_end = bad ? t_begin : min(t_begin + p.split_pages * kPage, kv - p.n_q + j + 1);
  const int page_begin = t_begin / kPage;
  const int n_pages = t_end > t_begin ? (t_end + kPage - 1) / kPage - page_begin : 0;
  if (tid == 0 && bad && rank == 0) record_status(p.status, MLA_ERR_BOUNDS);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ keys into the stages, codes into L2
    if (n_pages > 0) {
      const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride + page_begin;
      int ids = lane < n_pages ? pt[lane] : 0;
      int ids_next = 32 + lane < n_pages ? pt[32 + lane] : 0;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q64);
        tma_prefetch_desc(&tm_c8);
        tma_prefetch_desc(&tm_kr);
        mbar_arrive_expect_tx(bar_addr(bars.q_full), kQRope);
        tma_load_2d(smem_u32(smem + kOffQ), &tm_q64, kLatent + 32 * rank, bj * kHeads, bar_addr(bars.q_full));
      }
      bool ok = true;
      for (int base = 0; base < n_pages && ok; base += 32) {
        const int cnt = min(32, n_pages - base);
        for (int k = 0; k < cnt && ok; ++k) {
          const int i = base + k;
          int page = __shfl_sync(0xffffffffu, ids, k);
          const int ahead_a = __shfl_sync(0xffffffffu, ids, (k + 1) & 31);
          const int ahead_b = __shfl_sync(0xffffffffu, ids_next, (k + 1) & 31);
          if (lane == 0) {
            // the codes of the page after this one into L2, for the dequantisation warps' loads
            const int ahead = k + 1 < 32 ? ahead_a : ahead_b;
            if (i + 1 < n_pages && ahead >= 0 && ahead < p.num_pages)
              for (int c = 0; c < 4; ++c) tma_prefetch_l2_2d(&tm_c8, 64 * (4 * rank + c), ahead * kPage);
            const int s = i % kStages;
            ok = mbar_wait(bar_addr(bars.empty[s]), ((i / kStages) & 1) ^ 1, p.status, abort);
            if (ok) {
              if (page < 0 || page >= p.num_pages) {
                record_status(p.status, MLA_ERR_BOUNDS);
                page = 0;
              }
              uint8_t* stage = smem + kOffStage + s * kStageBytes;
              const uint32_t fb = bar_addr(bars.full[s]);
              mbar_arrive_expect_tx(fb, kPRope);
              tma_load_2d(smem_u32(stage + 4 * kPChunk), &tm_kr, 32 * rank, page * kPage, fb);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        ids = ids_next;
        ids_next = base + 64 + lane < n_pages ? pt[base + 64 + lane] : 0;
      }
    }
  } else if (warp >= kDqWarp0) {
    // ------------------------------------------------------------ codes -> float16 stages
    // Thread dt reads the 16-code pieces q = dt + 128 r (r < 8) of the CTA's 16 KB of
    // the page: token t = q / 16, codes [16 (q % 16), +16) of its 256 columns, i.e.
    // float16 chunk c = (q % 16) / 4, units 2 ((q % 16) % 4) and + 1 of row t (128-byte
    // swizzle: unit u of row t at t * 128 + (u ^ (t & 7)) * 16).  A warp's loads cover
    // two tokens' 256 contiguous bytes each.
    const int dt = tid - kDqWarp0 * 32;  // 0..127
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride + page_begin;
    int ids = lane < n_pages ? pt[lane] : 0;
    int ids_next = 32 + lane < n_pages ? pt[32 + lane] : 0;
    uint4 cur[8];
    float sc_cur = 0.f;
    int base = 0;  // the first page of the ids / ids_next window
    for (int i = 0; i < n_pages; ++i) {
      if (i - base == 32) {  // slide the page-id window
        base += 32;
        ids = ids_next;
        ids_next = base + 32 + lane < n_pages ? pt[base + 32 + lane] : 0;
      }
      int pg = __shfl_sync(0xffffffffu, ids, i - base);
      if (pg < 0 || pg >= p.num_pages) pg = 0;  // out of range: reported by the producer
      {
        const uint8_t* src = p.c8 + static_cast<int64_t>(pg) * kPage * kLatent + 256 * rank;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int q = dt + 128 * r;
          cur[r] = *reinterpret_cast<const uint4*>(src + (q >> 4) * kLatent + (q & 15) * 16);
        }
        sc_cur = dt < 64 ? p.scale[static_cast<int64_t>(pg) * kPage + dt] : 0.f;
      }
      const int s = i % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(bars.empty[s]), ((i / kStages) & 1) ^ 1, p.status, abort)))
        break;
      uint8_t* stage = smem + kOffStage + s * kStageBytes;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int q = dt + 128 * r;
        const int t = q >> 4, c = (q & 15) >> 2, u = q & 3;
        const uint32_t w[4] = {cur[r].x, cur[r].y, cur[r].z, cur[r].w};
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          h[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu));
          h[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
        }
        uint8_t* row = stage + c * kPChunk + t * 128;
        *reinterpret_cast<uint4*>(row + (((2 * u) ^ (t & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(row + (((2 * u + 1) ^ (t & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      if (dt < 64) {
        float* sc = reinterpret_cast<float*>(smem + kOffSc + s * 512);
        sc[dt] = sc_cur * (1.f / 256.f);  // exact
        sc[64 + dt] = sc_cur;
      }
      fence_proxy_async_smem();  // the stage is read by the MMAs
      mbar_arrive(bar_addr(bars.full[s]));
    }
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ tcgen05 issuers
    const uint32_t st0 = smem_u32(smem + kOffStage);
    if (n_pages > 0 && lane == 0 && warp == kMmaWarp) {
      const uint32_t idesc_qk = idesc_f16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
      const uint64_t d_k128 = smem_desc(st0, 16, 1024, kSw128);
      const uint64_t d_k64 = smem_desc(st0 + 4 * kPChunk, 16, 512, kSw64);
      const uint64_t d_qr = smem_desc(smem_u32(smem + kOffQ), 16, 512, kSw64);
      bool ok = mbar_wait(bar_addr(bars.q_full), 0, p.status, abort) &&
                mbar_wait(bar_addr(bars.q_tmem), 0, p.status, abort);
      for (int i = 0; i < n_pages && ok; ++i) {
        ok = mbar_wait(bar_addr(bars.full[i % kStages]), (i / kStages) & 1, p.status, abort);
        if (ok && i > 1) ok = mbar_wait(bar_addr(bars.s_free[i & 1]), ((i - 2) >> 1) & 1, p.status, abort);
        if (!ok) break;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
        const uint32_t d = tmem + kTmemS + 64 * (i & 1);
        mma_ts(d, tmem + kTmemQ, d_k128 + so, idesc_qk, 0u);
#pragma unroll
        for (int k = 1; k < 16; ++k)
          mma_ts(d, tmem + kTmemQ + 8 * k, d_k128 + so + (k >> 2) * (kPChunk >> 4) + (k & 3) * 2, idesc_qk, 1u);
        mma_ss(d, d_qr, d_k64 + so, idesc_qk, 1u);
        mma_ss(d, d_qr + 2, d_k64 + so + 2, idesc_qk, 1u);
        mma_commit(bar_addr(bars.s_full[i & 1]));
      }
    }
    if (n_pages > 0 && lane == 0 && warp == kPvWarp) {
      const uint32_t idesc_pv = idesc_f16(128, 256, /*a_mn=*/0, /*b_mn=*/1);
      const uint64_t d_v = smem_desc(st0, kPChunk, 1024, kSw128);
      const uint64_t d_p = smem_desc(smem_u32(smem + kOffP), 16, 1024, kSw128);
      for (int i = 0; i < n_pages; ++i) {
        if (!mbar_wait(bar_addr(bars.p_full[i & 1]), (i >> 1) & 1, p.status, abort)) break;
        tc_fence_after();
        const uint64_t vb = d_v + static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
        const uint64_t a = d_p + static_cast<uint64_t>(((i & 1) * kPBytes) >> 4);
        mma_ss(tmem + kTmemO, a, vb, idesc_pv, i > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < 4; ++k) mma_ss(tmem + kTmemO, a + 2 * k, vb + 128 * k, idesc_pv, 1u);
        mma_commit(bar_addr(bars.empty[i % kStages]));
        mma_commit(bar_addr(bars.pv_done[i & 1]));
      }
    }
    if (n_pages > 0 && lane == 0) {
      mma_commit(bar_addr(bars.drain));
      mbar_wait(bar_addr(bars.drain), 0, p.status, nullptr);
    }
    __syncwarp();
  } else if (warp == kSignalWarp) {
    // ------------------------------------------------------------ exchange buffer recycling
    if (lane == 0) {
      for (int i = 0; i < n_pages; ++i) {
        const int buf = i & 1;
        if (!mbar_wait(bar_addr(bars.x_read[buf]), (i >> 1) & 1, p.status, abort)) break;
        mbar_arrive_expect_tx(bar_addr(bars.x_full[buf]), kXTxBytes);
        mbar_arrive_remote(mapa(bar_addr(bars.x_free[buf]), peer));
      }
    }
  } else {
    // ------------------------------------------------------------ row warpgroups
    const int g = (warp - kRowWarp0) >> 2;  // warpgroup: pages i = g (mod 2)
    const int quad = warp & 3;               // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;        // head
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float* m_slot = reinterpret_cast<float*>(smem + kOffMax) + row;
    // (max, sum) of each row at the end go into the warpgroup's exchange buffer, read out by then
    float2* fin_mine = reinterpret_cast<float2*>(smem + kOffX + g * kXBufBytes);
    const float2* fin_other = reinterpret_cast<const float2*>(smem + kOffX + (g ^ 1) * kXBufBytes);
    bool ok = n_pages > 0;
    if (ok) {
      // The query goes into the MMAs as float16 (the codes' type).
      // Latent query columns [256r + 128g, 256r + 128g + 128) of the row into TMEM as f16 pairs.
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q_abs + (static_cast<int64_t>(bj) * kHeads + row) * kRow +
                                                         256 * rank + 128 * g);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = qsrc[8 * h + q];
          w[4 * q] = bf16x2_to_f16x2(v.x);
          w[4 * q + 1] = bf16x2_to_f16x2(v.y);
          w[4 * q + 2] = bf16x2_to_f16x2(v.z);
          w[4 * q + 3] = bf16x2_to_f16x2(v.w);
        }
        tmem_st32(tmem + lane_off + kTmemQ + 64 * g + 32 * h, w);
      }
      tmem_wait_st();
      if (g == 0) {
        // the RoPE query columns (landed by TMA): this thread converts the 64 bytes of its row
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.q_full), 0, p.status, abort));
        if (ok) {
          uint4* qr = reinterpret_cast<uint4*>(smem + kOffQ + row * 64);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v = qr[u];
            v.x = bf16x2_to_f16x2(v.x);
            v.y = bf16x2_to_f16x2(v.y);
            v.z = bf16x2_to_f16x2(v.z);
            v.w = bf16x2_to_f16x2(v.w);
            qr[u] = v;
          }
          fence_proxy_async_smem();  // visible to the MMAs that read it
        }
      }
      tc_fence_before();
      mbar_arrive(bar_addr(bars.q_tmem));
    }
    // exchange buffer g, this row: 16-byte unit q at q * 2048 + row * 16
    uint8_t* xrow = smem + kOffX + g * kXBufBytes + row * 16;
    const uint32_t x_remote = mapa(smem_u32(xrow), peer);
    const uint32_t xfull_remote = mapa(bar_addr(bars.x_full[g]), peer);
    const uint32_t s_addr = tmem + lane_off + kTmemS + 64 * g;
    uint8_t* prow = smem + kOffP + g * kPBytes + row * 128;  // this row of P
    const uint64_t scale2 = f32x2(kSumScaleLog2, kSumScaleLog2);
    float m_mine = -INFINITY, l = 0.f;  // reference max this warpgroup last used, and its partial sum
    for (int i = g; i < n_pages && ok; i += 2) {
      const uint32_t use = (i >> 1) & 1;
      const int n_valid = min(kPage, t_end - (page_begin + i) * kPage);  // visible tokens of the page
      // the page's token scales: s_t / 256 (exchange units) and s_t (P V operand), as f32 pairs
      const uint64_t* sc2 = reinterpret_cast<const uint64_t*>(smem + kOffSc + (i % kStages) * 512);
      const uint64_t* sp2 = sc2 + 32;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.s_full[g]), use, p.status, abort));
      // the stage's scales were written by the dequantisation warpgroup: acquire them
      // from its arrival (that phase has completed: the stage cannot move on before P V(i))
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.full[i % kStages]), (i / kStages) & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      // this CTA's partial scores times s_t / 256 (that is S_r / 256) as fp16 pairs:
      // word w holds columns 2w, 2w + 1
      uint32_t mine[32];
      {
        uint32_t a[32], c[32];
        tmem_ld32(s_addr, a);
        tmem_ld32(s_addr + 32, c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_addr(bars.s_free[g]));  // QK^T of page i + 2 may overwrite the buffer
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float2 x = f32x2_split(mul_f32x2(f32x2(__uint_as_float(a[2 * q]), __uint_as_float(a[2 * q + 1])), sc2[q]));
          const float2 y = f32x2_split(mul_f32x2(f32x2(__uint_as_float(c[2 * q]), __uint_as_float(c[2 * q + 1])), sc2[16 + q]));
          mine[q] = pack_f16x2(x.x, x.y);
          mine[16 + q] = pack_f16x2(y.x, y.y);
        }
      }
      // send: wait until the peer has read what this warpgroup sent two pages ago
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_free[g]), use ^ 1u, p.status, abort));
      if (!ok) break;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_async_v4(x_remote + q * (kRowThreads * 16), mine[4 * q], mine[4 * q + 1], mine[4 * q + 2], mine[4 * q + 3],
                    xfull_remote);
      // receive the peer's partial scores; both CTAs add fp16(S_0) + fp16(S_1)
      // in fp16, in the same order, so they hold the same S * 2^-8
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_full[g]), use, p.status, abort));
      if (!ok) break;
      uint32_t sh[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(xrow + q * (kRowThreads * 16));
        sh[4 * q] = hadd2(mine[4 * q], v.x);
        sh[4 * q + 1] = hadd2(mine[4 * q + 1], v.y);
        sh[4 * q + 2] = hadd2(mine[4 * q + 2], v.z);
        sh[4 * q + 3] = hadd2(mine[4 * q + 3], v.w);
      }
      mbar_arrive(bar_addr(bars.x_read[g]));  // warp 10 recycles the exchange buffer
      if (n_valid < kPage) {
        // columns past the last visible token (they may hold anything) become
        // -inf: out of the max, and exp gives 0 for them
#pragma unroll
        for (int w = 0; w < 32; ++w) {
          const uint32_t lo = 2 * w < n_valid ? (sh[w] & 0x0000ffffu) : 0x0000fc00u;
          const uint32_t hi = 2 * w + 1 < n_valid ? (sh[w] & 0xffff0000u) : 0xfc000000u;
          sh[w] = lo | hi;
        }
      }
      // row max (eight independent chains, then a tree: the same in any order), log2 domain
      uint32_t m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = sh[k];
#pragma unroll
      for (int w = 8; w < 32; ++w) m8[w & 7] = hmax2(m8[w & 7], sh[w]);
      const uint32_t mm = hmax2(hmax2(hmax2(m8[0], m8[1]), hmax2(m8[2], m8[3])), hmax2(hmax2(m8[4], m8[5]), hmax2(m8[6], m8[7])));
      const float2 mf = unpack_f16x2(mm);
      const float mx = fmaxf(mf.x, mf.y) * kSumScaleLog2;
      // the reference max after page i - 1 (from the other warpgroup)
      bool rescale = false;
      float factor = 1.f;
      if (i == 0) {
        m_mine = mx;
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.hand[g ^ 1]), ((i - 1) >> 1) & 1, p.status, abort));
        if (!ok) break;
        const float m_prev = *m_slot;
        if (m_prev != m_mine) {  // raised since this warpgroup's last page
          l *= ex2_approx(m_mine - m_prev);
          m_mine = m_prev;
        }
        if (mx > m_mine + kRescaleLog2) {
          factor = ex2_approx(m_mine - mx);
          m_mine = mx;
          l *= factor;
          rescale = true;
        }
      }
      *m_slot = m_mine;
      mbar_arrive(bar_addr(bars.hand[g]));  // page i + 1 may start its softmax
      // p = 2^(S * scale - m) in packed fp32 pairs; the row sum adds p, the MMA
      // gets p s_t in float16 (columns past the last token: 0)
      const uint64_t neg_m2 = f32x2(-m_mine, -m_mine);
      uint32_t pk[32];
      uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int w = 0; w < 32; ++w) {
        const float2 sf = unpack_f16x2(sh[w]);
        const float2 e = f32x2_split(fma_f32x2(f32x2(sf.x, sf.y), scale2, neg_m2));
        const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
        const float2 ps = f32x2_split(mul_f32x2(f32x2(p0, p1), sp2[w]));
        pk[w] = pack_f16x2_rn(2 * w < n_valid ? ps.x : 0.f, 2 * w + 1 < n_valid ? ps.y : 0.f);
        s4[w & 3] = add_f32x2(s4[w & 3], f32x2(p0, p1));
      }
      {
        const float2 a = f32x2_split(add_f32x2(add_f32x2(s4[0], s4[1]), add_f32x2(s4[2], s4[3])));
        l += a.x + a.y;
      }
      if (n_valid < kPage) {
        // Value rows past the last visible token may hold anything (NaN in
        // unwritten slots): zero them so that P = 0 there cannot make 0 * NaN.
        uint8_t* stage = smem + kOffStage + (i % kStages) * kStageBytes;
        const int nrow = kPage - n_valid;
        for (int v = row; v < 4 * nrow * 8; v += kRowThreads) {
          const int c = v / (nrow * 8), r = n_valid + (v / 8) % nrow, u = v & 7;
          *reinterpret_cast<uint4*>(stage + c * kPChunk + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      // The P buffer is free once P V(i - 2) has finished; O' may only be
      // rescaled once P V(i - 1) has.
      if (i >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[g]), use ^ 1u, p.status, abort));
        if (!ok) break;
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();  // visible to the P V MMAs
      if (__any_sync(0xffffffffu, rescale)) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[g ^ 1]), ((i - 1) >> 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + kTmemO + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * factor);
          tmem_st32(tmem + lane_off + kTmemO + c0, r);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      mbar_arrive(bar_addr(bars.p_full[g]));
    }
    // Exchanged partials are fp16(S_r / 256): one beyond |S_r| = 65520 * 256
    // (or a NaN) becomes infinite or NaN and leaves the row's max or sum non-finite.
    if (ok && g < n_pages && !(isfinite(l) && isfinite(m_mine))) record_status(p.status, MLA_ERR_RANGE);

    // epilogue: combine the two warpgroups' sums, then warpgroup g writes
    // columns [128g, 128g + 128) of this CTA's half of O' (normalised)
    fin_mine[row] = make_float2(m_mine, l);
    mbar_arrive(bar_addr(bars.fin));
    ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.fin), 0, p.status, abort));
    const int last = n_pages - 1;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[last & 1]), (last >> 1) & 1, p.status, abort));
    tc_fence_after();
    const int64_t out_row = (static_cast<int64_t>(bj) * p.num_splits + split) * kHeads + row;
    // One decision per warpgroup: its 128 x 128 tile of O' is staged in the
    // (now idle) ring and stored by TMA, or, if any of its rows has no valid
    // result, the warpgroup writes zeros directly.
    if (!ok && lane == 0) bars.wg_bad[g] = 1;
    named_barrier_sync(1 + g, kRowThreads);
    if (*reinterpret_cast<volatile int*>(&bars.wg_bad[g]) == 0) {
      const float2 f0 = g == 0 ? fin_mine[row] : fin_other[row], f1 = g == 0 ? fin_other[row] : fin_mine[row];
      const float m = fmaxf(f0.x, f1.x);
      const float lt = (f0.y > 0.f ? f0.y * ex2_approx(f0.x - m) : 0.f) + (f1.y > 0.f ? f1.y * ex2_approx(f1.x - m) : 0.f);
      const float inv = 1.f / lt;
      // four boxes of 32 fp32 columns x 128 rows, 128-byte swizzle: row r at
      // r * 128, 16-byte chunk c at (c ^ (r & 7)) * 16
      uint8_t* tile = smem + kOffStage + g * kOTileBytes;
      const int32_t y0 = static_cast<int32_t>(out_row) - row;  // row 0 of the unit
      if (p.out_bf16) {
        // a split's partial: two boxes of 64 bf16 columns x 128 rows (same swizzle)
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
          uint8_t* brow = tile + k * kOBoxBytes + row * 128;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {  // 32 columns (four 16-byte chunks) at a time
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + kTmemO + 128 * g + 64 * k + 32 * hh, r);
            tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const uint32_t* q = r + 8 * c4;
              const int c = 4 * hh + c4;
              *reinterpret_cast<uint4*>(brow + ((c ^ (row & 7)) << 4)) =
                  make_uint4(pack_bf16x2(__uint_as_float(q[0]) * inv, __uint_as_float(q[1]) * inv),
                             pack_bf16x2(__uint_as_float(q[2]) * inv, __uint_as_float(q[3]) * inv),
                             pack_bf16x2(__uint_as_float(q[4]) * inv, __uint_as_float(q[5]) * inv),
                             pack_bf16x2(__uint_as_float(q[6]) * inv, __uint_as_float(q[7]) * inv));
            }
          }
          fence_proxy_async_smem();  // visible to the TMA store
          named_barrier_sync(1 + g, kRowThreads);
          if (row == 0) {
            tma_store_2d(&tm_o, smem_u32(tile + k * kOBoxBytes), static_cast<int32_t>(rank * 256 + 128 * g + 64 * k),
                         y0);
            bulk_commit_group();
          }
        }
      }
#pragma unroll 1
      for (int k = 0; k < (p.out_bf16 ? 0 : 4); ++k) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kTmemO + 128 * g + 32 * k, r);
        tmem_wait_ld();
        uint8_t* brow = tile + k * kOBoxBytes + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(brow + ((c ^ (row & 7)) << 4)) =
              make_float4(__uint_as_float(r[4 * c]) * inv, __uint_as_float(r[4 * c + 1]) * inv,
                          __uint_as_float(r[4 * c + 2]) * inv, __uint_as_float(r[4 * c + 3]) * inv);
        fence_proxy_async_smem();  // visible to the TMA store
        named_barrier_sync(1 + g, kRowThreads);
        if (row == 0) {  // each box goes out as soon as it is staged
          tma_store_2d(&tm_o, smem_u32(tile + k * kOBoxBytes), static_cast<int32_t>(rank * 256 + 128 * g + 32 * k), y0);
          bulk_commit_group();
        }
      }
      if (rank == 0 && g == 0 && p.lse_out != nullptr) p.lse_out[out_row] = (m + log2f(lt)) * kLn2;
      if (row == 0) bulk_wait_read<0>();  // the staging area has been read (the writes complete with the grid)
    } else {
      const int64_t o0 = out_row * kLatent + rank * 256 + 128 * g;
      if (p.out_bf16) {
        uint16_t* orow = static_cast<uint16_t*>(p.o_out) + o0;
        for (int c0 = 0; c0 < 128; c0 += 8) *reinterpret_cast<uint4*>(orow + c0) = make_uint4(0u, 0u, 0u, 0u);
      } else {
        float* orow = static_cast<float*>(p.o_out) + o0;
        for (int c0 = 0; c0 < 128; c0 += 4) *reinterpret_cast<float4*>(orow + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (rank == 0 && g == 0 && p.lse_out != nullptr) p.lse_out[out_row] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // no CTA leaves while its peer may still address its shared memory
}


bool g_configured[64];

bool configure(int dev) {
  if (dev < 0 || dev >= 64) return false;
  if (!g_configured[dev]) {
    if (cudaFuncSetAttribute(decode_attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return false;
    g_configured[dev] = true;
  }
  return true;
}

}  // namespace

cudaError_t launch_decode_partial_fp8(const uint16_t* q_abs, const uint8_t* cache_c8, const float* cache_scale,
                                      const uint16_t* cache_kr, int64_t num_pages, const int32_t* page_table,
                                      int pt_stride, const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                      const SplitPlan& plan, void* o_out, float* lse_out, int* status,
                                      cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(B) * n_q * plan.num_splits;
  if (units == 0) return cudaSuccess;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || !configure(dev)) return cudaErrorInvalidDevice;
  CUtensorMap tq64, tc8, tkr, to;
  const uint64_t q_rows = static_cast<uint64_t>(B) * n_q * kHeads;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  if (!make_tmap_bf16_2d(&tq64, q_abs, q_rows, kRow, kRow, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_u8_2d(&tc8, cache_c8, c_rows, kLatent, kLatent, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_bf16_2d(&tkr, cache_kr, c_rows, kRope, kRope, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const bool out_bf16 = plan.num_splits > 1;  // partials for the merge
  const uint64_t o_rows = static_cast<uint64_t>(units) * kHeads;
  if (out_bf16 ? !make_tmap_bf16_2d(&to, o_out, o_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)
               : !make_tmap_f32_2d(&to, o_out, o_rows, kLatent, kLatent, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.q_abs = q_abs;
  prm.scale = cache_scale;
  prm.c8 = cache_c8;
  prm.o_out = o_out;
  prm.out_bf16 = out_bf16;
  prm.lse_out = lse_out;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.n_q = n_q;
  prm.max_kv_len = max_kv_len;
  prm.split_pages = plan.split_pages;
  prm.num_splits = plan.num_splits;
  return launch_kernel(decode_attn_fp8_kernel, dim3(static_cast<unsigned>(2 * units)), dim3(kThreads), kSmemBytes,
                       stream, tq64, tc8, tkr, to, prm);
}

}  // namespace mla
