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
//   * computes the partial score over those 288 columns and swaps it with its
//     peer through distributed shared memory; both CTAs round both partials to
//     fp16 (scaled by 2^-8 for range) and add them in the same order, so they
//     hold bitwise-equal scores S = S_0 + S_1;
//   * runs the same online softmax as its peer on that S, so both use identical
//     P, running max and sum, and accumulates its half of O' = P c.
// Half of the CTA's 256 latent query columns sit in TMEM (QK^T MMAs with A read
// from TMEM), the other half and the RoPE columns in shared memory, which leaves
// room for a 4-stage ring of half-pages.  P has TMEM buffers of its own, so a
// score buffer is free as soon as the softmax has read it: QK^T of page i+1 is
// issued while the softmax of page i is still running.
//
// Warp roles: warp 0 issues TMA loads (page ids are read 32 at a time), warp 1 allocates TMEM and issues tcgen05.mma (QK^T into one of two
// TMEM score buffers; P V with P read from TMEM), warps 6-9 are the exchange
// warpgroup (query into TMEM at start; per page: read the partial scores, swap
// them with the peer, write the full scores back into TMEM), warps 2-5 are the
// softmax/epilogue warpgroup, and warp 10 re-arms each exchange buffer once it
// has been read and tells the peer (a cluster-scope release that would
// otherwise stall the exchange warpgroup).  Both warpgroups have one thread per head row, and
// the exchange for page i+1 overlaps the softmax of page i.  The softmax keeps a
// lazily updated reference max: O' in TMEM is rescaled only when a page raises a
// row's max by more than 2^8.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 4;
constexpr int kThreads = 352;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kExchangeWarp0 = 6;
constexpr int kSignalWarp = 10;
constexpr int kRowThreads = 128;    // threads of each row warpgroup
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O' half: [0, 256)
constexpr uint32_t kTmemS = 256;    // two score buffers: [256, 320), [320, 384)
constexpr uint32_t kTmemP = 384;    // two P buffers (64 bf16 per row = 32 columns): [384, 416), [416, 448)
constexpr uint32_t kTmemQ = 448;    // the CTA's first 128 latent query columns as bf16 pairs: [448, 512)

constexpr int kQChunk = 128 * 128;    // 64 latent query columns x 128 heads, 128-byte rows (SW128)
constexpr int kQRope = 128 * 64;      // 32 RoPE columns x 128 heads, 64-byte rows (SW64)
constexpr int kQBytes = 2 * kQChunk + kQRope;  // query columns kept in shared memory
constexpr int kPChunk = 64 * 128;     // 64 latent columns x 64 tokens (SW128)
constexpr int kPRope = 64 * 64;       // 32 RoPE columns x 64 tokens (SW64)
constexpr int kStageBytes = 4 * kPChunk + kPRope;
constexpr int kXRowBytes = 144;       // 64 fp16 scores + 16 B pad: conflict-free 16-byte accesses
constexpr int kXBufBytes = kRowThreads * kXRowBytes;
constexpr uint32_t kXTxBytes = kRowThreads * 128;
constexpr float kXScale = 1.f / 256.f;  // exchanged partial scores are fp16(S_r * 2^-8)
constexpr float kXUnscale = 256.f;

constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kQBytes;
constexpr int kOffX = kOffStage + kStages * kStageBytes;
constexpr int kOffBar = kOffX + 2 * kXBufBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers + 1 KB alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr float kRescaleLog2 = 8.f;

struct Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full;      // query columns in shared memory
  uint64_t q_tmem;      // latent query columns in TMEM
  uint64_t s_full[2];   // partial scores of this CTA are in TMEM
  uint64_t s_ready[2];  // full scores are in TMEM
  uint64_t s_free[2];   // the softmax has read the full scores of this buffer
  uint64_t p_full[2];
  uint64_t pv_done;
  uint64_t x_full[2];   // peer's partial scores landed in exchange buffer k
  uint64_t x_free[2];   // peer has read our partial scores from its buffer k
  uint64_t x_read[2];   // all rows have read exchange buffer k
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  const uint16_t* q_abs;
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

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_addr(bars.full[s]), 1);
      mbar_init(bar_addr(bars.empty[s]), 1);
    }
    mbar_init(bar_addr(bars.q_full), 1);
    mbar_init(bar_addr(bars.q_tmem), kRowThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr(bars.s_full[s]), 1);
      mbar_init(bar_addr(bars.s_ready[s]), kRowThreads);
      mbar_init(bar_addr(bars.s_free[s]), kRowThreads);
      mbar_init(bar_addr(bars.p_full[s]), kRowThreads);
      mbar_init(bar_addr(bars.x_full[s]), 1);
      mbar_init(bar_addr(bars.x_free[s]), 1);
      mbar_init(bar_addr(bars.x_read[s]), kRowThreads);
    }
    mbar_init(bar_addr(bars.pv_done), 1);
    mbar_init(bar_addr(bars.drain), 1);
    bars.abort = 0;
    fence_mbar_init();
    // arm the first use of both exchange buffers: 16 KB of the peer's partial scores each
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
  // global memory only from here on: the previous kernel of the stream has finished
  grid_dep_wait();
  grid_dep_launch();

  // The unit's token range [t_begin, t_end): identical in both CTAs of the cluster.
  const int kv = p.kv_lens[b];
  const bool bad = kv > p.max_kv_len || kv < p.n_q || (kv + kPage - 1) / kPage > p.pt_stride;
  const int t_begin = split * p.split_pages * kPage;
  const int t_end = bad ? t_begin : min(t_begin + p.split_pages * kPage, kv - p.n_q + j + 1);
  const int page_begin = t_begin / kPage;
  const int n_pages = t_end > t_begin ? (t_end + kPage - 1) / kPage - page_begin : 0;
  if (tid == 0 && bad && rank == 0) record_status(p.status, MLA_ERR_BOUNDS);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (n_pages > 0) {
      const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride + page_begin;
      int ids = lane < n_pages ? pt[lane] : 0;
      int ids_next = 32 + lane < n_pages ? pt[32 + lane] : 0;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q128);
        tma_prefetch_desc(&tm_q64);
        tma_prefetch_desc(&tm_c128);
        tma_prefetch_desc(&tm_c64);
        // query columns [256r + 128, 256r + 256) and the RoPE half r into shared memory
        const uint32_t qb = smem_u32(smem + kOffQ);
        const int q_row = bj * kHeads;
        mbar_arrive_expect_tx(bar_addr(bars.q_full), kQBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_2d(qb + c * kQChunk, &tm_q128, 256 * rank + 128 + 64 * c, q_row, bar_addr(bars.q_full));
        tma_load_2d(qb + 2 * kQChunk, &tm_q64, kLatent + 32 * rank, q_row, bar_addr(bars.q_full));
      }
      bool ok = true;
      for (int base = 0; base < n_pages && ok; base += 32) {
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
        ids_next = base + 64 + lane < n_pages ? pt[base + 64 + lane] : 0;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    if (n_pages > 0) {
      const uint32_t idesc_qk = idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
      const uint32_t idesc_pv = idesc_bf16(128, 256, /*a_mn=*/0, /*b_mn=*/1);
      // Descriptors of stage 0 and of the query in shared memory; a stage, chunk
      // or K step is a byte offset added to the start-address field (16-byte units).
      const uint32_t st0 = smem_u32(smem + kOffStage);
      const uint64_t d_k128 = smem_desc(st0, 16, 1024, kSw128);             // keys, latent chunk 0
      const uint64_t d_k64 = smem_desc(st0 + 4 * kPChunk, 16, 512, kSw64);  // keys, RoPE half
      const uint64_t d_v = smem_desc(st0, kPChunk, 1024, kSw128);           // values (MN-major)
      const uint64_t d_ql = smem_desc(smem_u32(smem + kOffQ), 16, 1024, kSw128);               // query chunks 2, 3
      const uint64_t d_qr = smem_desc(smem_u32(smem + kOffQ + 2 * kQChunk), 16, 512, kSw64);   // query RoPE half
      const int last_rows = t_end - (page_begin + n_pages - 1) * kPage;  // valid rows of the last page
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.q_full), 0, p.status, abort) &&
                                            mbar_wait(bar_addr(bars.q_tmem), 0, p.status, abort));

      // S(i) = Q K(i)^T into score buffer i & 1, once page i has landed and the
      // softmax has read the scores of page i - 2 from that buffer.
      auto issue_qk = [&](int i) -> bool {
        const int s = i % kStages, buf = i & 1;
        bool w = mbar_wait(bar_addr(bars.full[s]), (i / kStages) & 1, p.status, abort);
        w = w && mbar_wait(bar_addr(bars.s_free[buf]), ((i >> 1) & 1) ^ 1, p.status, abort);
        if (!__all_sync(0xffffffffu, w)) return false;
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
          const uint64_t so = static_cast<uint64_t>((s * kStageBytes) >> 4);
          const uint32_t d = tmem + kTmemS + buf * 64;
          // latent chunks 0, 1: A = query columns in TMEM (8 columns per K step of 16)
          mma_ts(d, tmem + kTmemQ, d_k128 + so, idesc_qk, 0u);
#pragma unroll
          for (int k = 1; k < 8; ++k)
            mma_ts(d, tmem + kTmemQ + 8 * k, d_k128 + so + (k >> 2) * (kPChunk >> 4) + (k & 3) * 2, idesc_qk, 1u);
          // latent chunks 2, 3: A = query columns in shared memory
#pragma unroll
          for (int k = 8; k < 16; ++k)
            mma_ss(d, d_ql + ((k - 8) >> 2) * (kQChunk >> 4) + (k & 3) * 2,
                   d_k128 + so + (k >> 2) * (kPChunk >> 4) + (k & 3) * 2, idesc_qk, 1u);
          // RoPE part
          mma_ss(d, d_qr, d_k64 + so, idesc_qk, 1u);
          mma_ss(d, d_qr + 2, d_k64 + so + 2, idesc_qk, 1u);
          mma_commit(bar_addr(bars.s_full[buf]));
        }
        __syncwarp();
        return true;
      };
      // O' += P(i) V(i), then page i's stage goes back to the producer.
      auto issue_pv = [&](int i) -> bool {
        const bool w = mbar_wait(bar_addr(bars.p_full[i & 1]), (i >> 1) & 1, p.status, abort);
        if (!__all_sync(0xffffffffu, w)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t vb = d_v + static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
          const uint32_t a = tmem + kTmemP + (i & 1) * 32;
          mma_ts(tmem + kTmemO, a, vb, idesc_pv, i > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < 4; ++k) mma_ts(tmem + kTmemO, a + 8 * k, vb + 128 * k, idesc_pv, 1u);
          mma_commit(bar_addr(bars.empty[i % kStages]));
          mma_commit(bar_addr(bars.pv_done));
        }
        __syncwarp();
        return true;
      };

      // QK^T runs two pages ahead of P V: S(i + 2) only needs the softmax to have
      // read S(i), while P V(i) needs the whole softmax of page i.
      if (ok) ok = issue_qk(0);
      if (ok && n_pages > 1) ok = issue_qk(1);
      for (int i = 0; i < n_pages && ok; ++i) {
        if (i + 2 < n_pages) ok = issue_qk(i + 2);
        if (ok) ok = issue_pv(i);
      }
      // no tcgen05 operation may still be running when TMEM is released
      if (lane == 0) mma_commit(bar_addr(bars.drain));
      __syncwarp();
      mbar_wait(bar_addr(bars.drain), 0, p.status, nullptr);
    }
  } else if (warp == kSignalWarp) {
    // ------------------------------------------------------------ exchange buffer recycling
    if (lane == 0) {
      for (int i = 0; i < n_pages; ++i) {
        const int buf = i & 1;
        if (!mbar_wait(bar_addr(bars.x_read[buf]), (i >> 1) & 1, p.status, abort)) break;
        mbar_arrive_expect_tx(bar_addr(bars.x_full[buf]), kXTxBytes);   // armed for the buffer's next use
        mbar_arrive_remote(mapa(bar_addr(bars.x_free[buf]), peer));      // the peer may refill it
      }
    }
  } else if (warp >= kExchangeWarp0) {
    // ------------------------------------------------------------ score exchange
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // head
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = n_pages > 0;
    if (ok) {
      // this CTA's first 128 latent query columns of the row into TMEM as bf16 pairs
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q_abs + (static_cast<int64_t>(bj) * kHeads + row) * kRow +
                                                         256 * rank);
#pragma unroll 1
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = qsrc[c0 / 4 + q];
          w[4 * q] = v.x;
          w[4 * q + 1] = v.y;
          w[4 * q + 2] = v.z;
          w[4 * q + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kTmemQ + c0, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(bars.q_tmem));
    }
    uint8_t* xrow0 = smem + kOffX + row * kXRowBytes;
    const uint32_t x_remote0 = mapa(smem_u32(xrow0), peer);
    float range_max = 0.f;
    for (int i = 0; i < n_pages && ok; ++i) {
      const int buf = i & 1;        // TMEM score buffer and exchange buffer
      const uint32_t use = (i >> 1) & 1;
      const uint32_t s_addr = tmem + lane_off + kTmemS + buf * 64;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.s_full[buf]), use, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      uint32_t mine[32];
      {
        uint32_t a[32], c[32];
        tmem_ld32(s_addr, a);
        tmem_ld32(s_addr + 32, c);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float x0 = __uint_as_float(a[2 * q]), x1 = __uint_as_float(a[2 * q + 1]);
          const float y0 = __uint_as_float(c[2 * q]), y1 = __uint_as_float(c[2 * q + 1]);
          range_max = fmaxf(range_max, fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(y0), fabsf(y1))));
          mine[q] = pack_f16x2(x0 * kXScale, x1 * kXScale);
          mine[16 + q] = pack_f16x2(y0 * kXScale, y1 * kXScale);
        }
      }
      // send: wait until the peer has read what we sent into this buffer two pages ago
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_free[buf]), use ^ 1u, p.status, abort));
      if (!ok) break;
      const uint32_t x_remote = x_remote0 + buf * kXBufBytes;
      const uint32_t xfull_remote = mapa(bar_addr(bars.x_full[buf]), peer);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_async_v4(x_remote + 16 * q, mine[4 * q], mine[4 * q + 1], mine[4 * q + 2], mine[4 * q + 3], xfull_remote);
      // receive the peer's partial scores; both CTAs add fp16(S_0) + fp16(S_1) in fp32
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_full[buf]), use, p.status, abort));
      if (!ok) break;
      uint32_t full0[32], full1[32];
      {
        const uint4* xr = reinterpret_cast<const uint4*>(xrow0 + buf * kXBufBytes);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = xr[q];
          const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int w = 4 * q + e;  // packed word index: columns 2w, 2w+1
            const float2 a = unpack_f16x2(mine[w]);
            const float2 c = unpack_f16x2(pw[e]);
            const uint32_t lo = __float_as_uint((a.x + c.x) * kXUnscale);
            const uint32_t hi = __float_as_uint((a.y + c.y) * kXUnscale);
            if (w < 16) {
              full0[2 * w] = lo;
              full0[2 * w + 1] = hi;
            } else {
              full1[2 * (w - 16)] = lo;
              full1[2 * (w - 16) + 1] = hi;
            }
          }
        }
      }
      tmem_st32(s_addr, full0);
      tmem_st32(s_addr + 32, full1);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(bars.s_ready[buf]));
      // this row is done with the exchange buffer (warp 10 recycles it)
      mbar_arrive(bar_addr(bars.x_read[buf]));
    }
    // exchanged partials are fp16(S_r / 256): beyond this magnitude they overflow
    if (range_max > 1.6e7f) record_status(p.status, MLA_ERR_RANGE);
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
        tc_fence_before();
        mbar_arrive(bar_addr(bars.s_free[buf]));  // the MMA issuer may overwrite this buffer
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
        tmem_st32(tmem + lane_off + kTmemP + buf * 32, pk);
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
  prm.q_abs = q_abs;
  prm.o_out = o_out;
  prm.lse_out = lse_out;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.n_q = n_q;
  prm.max_kv_len = max_kv_len;
  prm.split_pages = plan.split_pages;
  prm.num_splits = plan.num_splits;
  return launch_kernel(decode_attn_tc_kernel, dim3(static_cast<unsigned>(2 * units)), dim3(kThreads), kSmemBytes, stream,
                       tq128, tq64, tc128, tc64, prm);
}

}  // namespace mla
