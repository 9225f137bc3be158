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
//     fp16 (scaled by 2^-8 for range: the query enters the MMAs pre-scaled) and
//     add them in fp16 in the same order, so they hold bitwise-equal scores
//     S = S_0 + S_1;
//   * runs the same online softmax as its peer on that S, so both use identical
//     P, running max and sum, and accumulates its half of O' = P c.
// The CTA's 256 latent query columns sit in TMEM, so the latent QK^T MMAs read A
// from TMEM and only their B operand (the page's keys) from shared memory: at
// N = 64 that is a quarter of the shared-memory bandwidth, which leaves room
// for the TMA writes and the score exchange (SS MMAs, which also read A from
// shared memory, slowed down severalfold next to them).  Only the 32 RoPE query
// columns stay in shared memory.  TMEM then holds O' (256 columns), the query
// (128) and two 64-column score buffers (page i uses buffer i & 1), so QK^T of
// the next page never waits for the scores of the last one to be read (with a
// single score buffer that hand-over, some 700 cycles per page, bounded the
// page rate); P goes to shared memory (the A operand of P V), with a 4-slot ring
// of half-pages beside it.
//
// The per-page work of the row threads is a chain of waits (the peer's partial
// scores arrive some 1,300 cycles after a CTA sends its own, and the two CTAs
// of a cluster drift apart by up to a page), about 3,900 cycles in all, so
// three row warpgroups take the pages in turn (page i goes to warpgroup i mod 3)
// and the chain of one page overlaps those of the next two.  Exchange buffers
// and P buffers are used by page parity: a warpgroup waits on a buffer only
// until the page two before its own has released it.  The mbarriers that signal
// those buffers (P V finished, partial scores landed, partial scores read by the
// peer, scores in TMEM, scores read) are kept per page mod 4, not per page
// parity: a parity wait is only
// sound when the waiter cannot be two phases ahead, and a warpgroup's own
// history (its page three back, and the max handed down to it) guarantees the
// events of page i - 4 but not those of page i - 2.
//
// Warp roles: warp 0 issues TMA loads (the query first, then the pages; page
// ids are read 32 at a time); warp 1 allocates TMEM and one of its threads
// issues the QK^T MMAs, while one thread of warp 15 issues the P V MMAs: an MMA
// issue blocks until the tensor pipe takes it, so with a single issuer a ready
// P V waited behind a whole QK^T batch (and the reverse); warps 2-13 are the
// three row warpgroups, one thread per head row: warpgroup g reads the partial
// scores of its page from its TMEM score buffer (which frees it for QK^T two
// pages on), swaps them with the peer CTA, adds them, runs the softmax step
// and writes P into shared memory.  The warpgroups pass only the running reference max
// on to the next page's warpgroup.  Warp 14 re-arms each exchange buffer once it
// has been read and tells the peer (a cluster-scope release that would
// otherwise stall a row warpgroup).  The reference max is updated lazily: O' in
// TMEM is rescaled only when a page raises a row's max by more than 2^8; each
// warpgroup keeps its own partial row sum relative to the max it last used.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 4;
// When the producer turns to page i it first pulls page i + kL2Ahead into L2:
// that page's TMA load, issued about one slot period later, then pays the L2
// latency instead of the DRAM one, which shortens the life of a ring slot.
// Measured at B = 32, L = 4096: 1 or 2 ahead 53.3-53.6 us, 4 ahead 55.0,
// 8 ahead 60.1, 12 ahead 64.8, none 60.4.
constexpr int kL2Ahead = 1;
constexpr int kRowWGs = 3;
constexpr int kThreads = 128 * kRowWGs + 128;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kRowWarp0 = 2;        // warps 2-13: row warpgroups 0, 1, 2
constexpr int kSignalWarp = kRowWarp0 + 4 * kRowWGs;
constexpr int kPvWarp = kSignalWarp + 1;
constexpr int kRowThreads = 128;    // threads of each row warpgroup
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O' half: [0, 256)
constexpr uint32_t kTmemQ = 256;    // the CTA's 256 latent query columns as bf16 pairs: [256, 384)
constexpr uint32_t kTmemS = 384;    // partial scores of page i: [384 + 64 (i & 1), 448 + 64 (i & 1))

constexpr int kQRope = 128 * 64;      // 32 RoPE query columns x 128 heads, 64-byte rows (SW64)
constexpr int kPChunk = 64 * 128;     // 64 latent columns x 64 tokens (SW128)
constexpr int kPRope = 64 * 64;       // 32 RoPE columns x 64 tokens (SW64)
constexpr int kStageBytes = 4 * kPChunk + kPRope;
// Exchange buffer: 64 fp16 partial scores per row, stored unit-major (16-byte unit
// q of row r at q * 2048 + r * 16), so that each warp's stores and loads of one
// unit cover 512 contiguous bytes: whole 128-byte lines.
constexpr int kXBufBytes = kRowThreads * 128;
constexpr uint32_t kXTxBytes = kXBufBytes;
// Exchanged partial scores are fp16(S_r * 2^-8); their sum times 2^8 kScale is
// the scaled score, so the softmax folds 2^8 into its log2-domain scale.  The
// row work is done on fp16 pairs (add, max) and packed fp32 pairs (exponent
// argument, row sum), half the instructions of scalar fp32.
constexpr float kSumScaleLog2 = kScaleLog2 * 256.f;

constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kQRope;
constexpr int kOffX = kOffStage + kStages * kStageBytes;
// P of page i in buffer i & 1: 128 rows x 64 bf16, K-major with the 128-byte
// swizzle (the A operand of P V), row r at r * 128 with 16-byte chunk c at
// (c ^ (r & 7)) * 16.
constexpr int kPBytes = kHeads * 128;
constexpr int kOffP = kOffX + 2 * kXBufBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
// At the start the CTA's 256 latent query columns (128 rows) land by TMA in ring
// slots 2 and 3 as four 64-column boxes with the 128-byte swizzle (row r of box b
// at b * 16 KB + r * 128, its 16-byte chunk c at (c ^ (r & 7)) * 16); row
// warpgroups 0 and 1 move them into TMEM, and only then do pages 2 and 3 load there.
constexpr int kQBoxBytes = kHeads * 128;
constexpr int kQStageSlot = 2;
constexpr int kOffQStage = kOffStage + kQStageSlot * kStageBytes;
static_assert(kQStageSlot + 2 == kStages && 4 * kQBoxBytes <= 2 * kStageBytes, "query staging fits in the last two slots");
constexpr int kOffMax = kOffBar + 512;            // per-row reference max handed between warpgroups
constexpr int kOffFin = kOffMax + 4 * kHeads;     // per-warpgroup (max, sum) per row at the end
constexpr int kSmemBytes = kOffFin + 8 * kRowWGs * kHeads + 1024;  // + 1 KB alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles start on 1 KB");

constexpr float kRescaleLog2 = 8.f;
// Output staging at the end: row warpgroup g < 2 stages its 128 x 128 tile of O'
// in the ring (idle by then): four 32-column fp32 boxes for the final O' of a
// single split, two 64-column bf16 boxes for a split's partial.
constexpr int kOBoxBytes = 128 * 128;
constexpr int kOTileBytes = 4 * kOBoxBytes;
static_assert(2 * kOTileBytes <= kStages * kStageBytes, "output staging fits in the ring");

struct Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full;            // RoPE query columns in shared memory
  uint64_t q_lat;             // latent query columns staged in ring slots 3-4
  uint64_t q_tmem;            // latent query columns in TMEM
  uint64_t s_full[4];         // partial scores of the last page i = k (mod 4) are in score buffer i & 1
  uint64_t s_free[4];         // ... and have been read (QK^T of page i + 2 may overwrite them)
  uint64_t hand[kRowWGs];     // warpgroup g has published the reference max of its page
  uint64_t p_full[2];         // P of the current page of parity k is in P buffer k (and O' rescaled)
  uint64_t pv_done[4];        // P V of the last page i = k (mod 4) has finished
  uint64_t x_full[4];         // peer's partial scores of page i = k (mod 4) landed (buffer i & 1)
  uint64_t x_free[4];         // peer has read our partial scores of page i = k (mod 4)
  uint64_t x_read[2];         // all rows have read exchange buffer k
  uint64_t fin;               // every warpgroup has published its final (max, sum)
  uint64_t drain;             // both issuers' MMAs have finished
  uint32_t tmem_base;
  int abort;
  int wg_bad[kRowWGs];        // a row of warpgroup g has no valid result: the outputs are zeros
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  void* o_out;         // fp32 O' (one split), or the splits' bf16 partials (out_bf16)
  float* lse_out;
  int out_bf16;
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
decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_qlat, const __grid_constant__ CUtensorMap tm_q64,
                      const __grid_constant__ CUtensorMap tm_c128,
                      const __grid_constant__ CUtensorMap tm_c64, const __grid_constant__ CUtensorMap tm_o,
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
    mbar_init(bar_addr(bars.q_lat), 1);
    mbar_init(bar_addr(bars.q_tmem), 2 * kRowThreads);
    for (int g = 0; g < kRowWGs; ++g) {
      mbar_init(bar_addr(bars.hand[g]), kRowThreads);
      bars.wg_bad[g] = 0;
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_addr(bars.p_full[k]), kRowThreads);
      mbar_init(bar_addr(bars.x_read[k]), kRowThreads);
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(bar_addr(bars.s_full[k]), 1);
      mbar_init(bar_addr(bars.s_free[k]), kRowThreads);
      mbar_init(bar_addr(bars.pv_done[k]), 1);
      mbar_init(bar_addr(bars.x_full[k]), 1);
      mbar_init(bar_addr(bars.x_free[k]), 1);
    }
    mbar_init(bar_addr(bars.fin), kRowWGs * kRowThreads);
    mbar_init(bar_addr(bars.drain), 2);
    bars.abort = 0;
    fence_mbar_init();
    // armed for pages 0-3: 16 KB of the peer's partial scores each
    for (int k = 0; k < 4; ++k) mbar_arrive_expect_tx(bar_addr(bars.x_full[k]), kXTxBytes);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  // global memory only from here on: the previous kernel of the stream has finished
  grid_dep_wait();
  grid_dep_launch();

  // The query (its latent half r and RoPE half r) does not depend on the unit's
  // token range: it is requested first, and the page ids of the split are read
  // while the sequence length is still on its way.
  int ids = 0, ids_next = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_qlat);
      tma_prefetch_desc(&tm_q64);
      mbar_arrive_expect_tx(bar_addr(bars.q_lat), 4 * kQBoxBytes);
      tma_load_3d(smem_u32(smem + kOffQStage), &tm_qlat, 0, bj * kHeads, 4 * rank, bar_addr(bars.q_lat));
      mbar_arrive_expect_tx(bar_addr(bars.q_full), kQRope);
      tma_load_2d(smem_u32(smem + kOffQ), &tm_q64, kLatent + 32 * rank, bj * kHeads, bar_addr(bars.q_full));
      tma_prefetch_desc(&tm_c128);
      tma_prefetch_desc(&tm_c64);
    }
    const int pb = split * p.split_pages;
    const int32_t* pt0 = p.page_table + static_cast<int64_t>(b) * p.pt_stride + pb;
    ids = pb + lane < p.pt_stride ? pt0[lane] : 0;
    ids_next = pb + 32 + lane < p.pt_stride ? pt0[32 + lane] : 0;
  }

  // The unit's token range [t_begin, t_end): identical in both CTAs of the cluster.
  const int kv = p.kv_lens[b];
  const bool bad = kv > p.max_kv_len || kv < p.n_q || (kv + kPage - 1) / kPage > p.pt_stride;
  const int t_begin = split * p.split_pages * kPage;
  const int t_end = bad ? t_begin : min(t_begin + p.split_pages * kPage, kv - p.n_q + j + 1);
  const int page_begin = t_begin / kPage;
  const int n_pages = t_end > t_begin ? (t_end + kPage - 1) / kPage - page_begin : 0;
  if (tid == 0 && bad && rank == 0) record_status(p.status, MLA_ERR_BOUNDS);
  // the peer's barriers exist before any remote traffic (the first partial
  // scores, long after the loads above are on their way)
  cluster_sync();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (n_pages > 0) {
      const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride + page_begin;
      // this CTA's 288 columns of a page into L2
      auto prefetch = [&](int page) {
        if (page < 0 || page >= p.num_pages) return;
        tma_prefetch_l2_3d(&tm_c128, 0, page * kPage, 4 * rank);
        tma_prefetch_l2_2d(&tm_c64, kLatent + 32 * rank, page * kPage);
      };
      bool ok = true;
      for (int base = 0; base < n_pages && ok; base += 32) {
        const int cnt = min(32, n_pages - base);
        for (int k = 0; k < cnt && ok; ++k) {
          const int i = base + k;
          int page = __shfl_sync(0xffffffffu, ids, k);
          const int ahead_a = __shfl_sync(0xffffffffu, ids, (k + kL2Ahead) & 31);
          const int ahead_b = __shfl_sync(0xffffffffu, ids_next, (k + kL2Ahead) & 31);
          if (lane == 0 && i + kL2Ahead < n_pages) prefetch(k + kL2Ahead < 32 ? ahead_a : ahead_b);
          if (lane == 0) {
            const int s = i % kStages;
            // slots 3-4 hold the staged query until the row threads have moved it to TMEM
            if (i == kQStageSlot) ok = mbar_wait(bar_addr(bars.q_tmem), 0, p.status, abort);
            ok = ok && mbar_wait(bar_addr(bars.empty[s]), ((i / kStages) & 1) ^ 1, p.status, abort);
            if (ok) {
              if (page < 0 || page >= p.num_pages) {
                record_status(p.status, MLA_ERR_BOUNDS);
                page = 0;  // stay in bounds; the result of this unit is not meaningful
              }
              const uint32_t sb = smem_u32(smem + kOffStage + s * kStageBytes);
              const uint32_t fb = bar_addr(bars.full[s]);
              mbar_arrive_expect_tx(fb, kStageBytes);
              // the CTA's four 64-column chunks of the page in one box: (64 columns, 64 tokens, 4 chunks)
              tma_load_3d(sb, &tm_c128, 0, page * kPage, 4 * rank, fb);
              tma_load_2d(sb + 4 * kPChunk, &tm_c64, kLatent + 32 * rank, page * kPage, fb);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        ids = ids_next;
        ids_next = base + 64 + lane < n_pages ? pt[base + 64 + lane] : 0;
      }
    } else if (lane == 0) {
      // nothing to do, but no copy into this CTA's shared memory may still be in
      // flight when it exits
      mbar_wait(bar_addr(bars.q_lat), 0, p.status, abort);
      mbar_wait(bar_addr(bars.q_full), 0, p.status, abort);
    }
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ tcgen05 issuers
    // One thread of warp 1 issues QK^T and one thread of warp 15 issues P V,
    // each blocking on its own barriers, so that neither kind waits behind the
    // other's issue (an MMA issue returns only once the tensor pipe accepts it).
    // They touch disjoint TMEM (scores / O' and P) and a stage is released by
    // P V of its page, which follows QK^T of that page through the softmax.
    const uint32_t st0 = smem_u32(smem + kOffStage);
    if (n_pages > 0 && lane == 0 && warp == kMmaWarp) {
      const uint32_t idesc_qk = idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
      // Descriptors of stage 0 and of the RoPE query columns; a stage, chunk or
      // K step is a byte offset added to the start-address field (16-byte units).
      const uint64_t d_k128 = smem_desc(st0, 16, 1024, kSw128);             // keys, latent chunk 0
      const uint64_t d_k64 = smem_desc(st0 + 4 * kPChunk, 16, 512, kSw64);  // keys, RoPE half
      const uint64_t d_qr = smem_desc(smem_u32(smem + kOffQ), 16, 512, kSw64);  // RoPE query half
      bool ok = mbar_wait(bar_addr(bars.q_full), 0, p.status, abort) &&
                mbar_wait(bar_addr(bars.q_tmem), 0, p.status, abort);
      // S(i) = Q K(i)^T into score buffer i & 1, once page i has landed and the
      // scores of page i - 2 have been read out of that buffer.
      for (int i = 0; i < n_pages && ok; ++i) {
        ok = mbar_wait(bar_addr(bars.full[i % kStages]), (i / kStages) & 1, p.status, abort);
        if (ok && i > 1) ok = mbar_wait(bar_addr(bars.s_free[(i - 2) & 3]), ((i - 2) >> 2) & 1, p.status, abort);
        if (!ok) break;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
        const uint32_t d = tmem + kTmemS + 64 * (i & 1);
        // latent part: A = query columns in TMEM (8 columns per K step of 16)
        mma_ts(d, tmem + kTmemQ, d_k128 + so, idesc_qk, 0u);
#pragma unroll
        for (int k = 1; k < 16; ++k)
          mma_ts(d, tmem + kTmemQ + 8 * k, d_k128 + so + (k >> 2) * (kPChunk >> 4) + (k & 3) * 2, idesc_qk, 1u);
        // RoPE part: A = query columns in shared memory
        mma_ss(d, d_qr, d_k64 + so, idesc_qk, 1u);
        mma_ss(d, d_qr + 2, d_k64 + so + 2, idesc_qk, 1u);
        mma_commit(bar_addr(bars.s_full[i & 3]));
      }
    }
    if (n_pages > 0 && lane == 0 && warp == kPvWarp) {
      const uint32_t idesc_pv = idesc_bf16(128, 256, /*a_mn=*/0, /*b_mn=*/1);
      const uint64_t d_v = smem_desc(st0, kPChunk, 1024, kSw128);  // values (MN-major)
      const uint64_t d_p = smem_desc(smem_u32(smem + kOffP), 16, 1024, kSw128);  // P buffer 0 (K-major)
      // O' += P(i) V(i) once P(i) is written; then page i's stage goes back to
      // the producer and page i + 2 may reuse the P buffer.
      for (int i = 0; i < n_pages; ++i) {
        if (!mbar_wait(bar_addr(bars.p_full[i & 1]), (i >> 1) & 1, p.status, abort)) break;
        tc_fence_after();
        const uint64_t vb = d_v + static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
        const uint64_t a = d_p + static_cast<uint64_t>(((i & 1) * kPBytes) >> 4);
        mma_ss(tmem + kTmemO, a, vb, idesc_pv, i > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < 4; ++k) mma_ss(tmem + kTmemO, a + 2 * k, vb + 128 * k, idesc_pv, 1u);
        mma_commit(bar_addr(bars.empty[i % kStages]));
        mma_commit(bar_addr(bars.pv_done[i & 3]));
      }
    }
    if (n_pages > 0 && lane == 0) {
      // no tcgen05 operation may still be running when TMEM is released
      mma_commit(bar_addr(bars.drain));
      mbar_wait(bar_addr(bars.drain), 0, p.status, nullptr);
    }
    __syncwarp();
  } else if (warp == kSignalWarp) {
    // ------------------------------------------------------------ exchange buffer recycling
    if (lane == 0) {
      for (int i = 0; i < n_pages; ++i) {
        if (!mbar_wait(bar_addr(bars.x_read[i & 1]), (i >> 1) & 1, p.status, abort)) break;
        mbar_arrive_expect_tx(bar_addr(bars.x_full[i & 3]), kXTxBytes);  // armed for page i + 4
        mbar_arrive_remote(mapa(bar_addr(bars.x_free[i & 3]), peer));     // the peer may refill buffer i & 1
      }
    }
  } else {
    // ------------------------------------------------------------ row warpgroups
    const int g = (warp - kRowWarp0) >> 2;  // warpgroup: pages i = g (mod 3)
    const int quad = warp & 3;               // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;        // head
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float* m_slot = reinterpret_cast<float*>(smem + kOffMax) + row;
    float2* fin = reinterpret_cast<float2*>(smem + kOffFin);
    bool ok = n_pages > 0;
    if (ok && g < 2) {
      // The query goes into the MMAs times 2^-8 (exact in bf16), so that the
      // partial scores come out as S_r * 2^-8, the form they are exchanged in.
      // Latent query columns [256r + 128g, 256r + 128g + 128) of the row into TMEM
      // as bf16 pairs, from the two 64-column boxes the producer staged by TMA
      // (one bulk request per CTA instead of 16 scattered loads per thread, which
      // the L1's outstanding-miss limit had spread over several microseconds).
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.q_lat), 0, p.status, abort));
      if (ok) {
        const uint8_t* qst = smem + kOffQStage + (2 * g) * kQBoxBytes + row * 128;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t w[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(qst + h * kQBoxBytes + ((q ^ (row & 7)) << 4));
            w[4 * q] = bf16x2_times_2m8(v.x);
            w[4 * q + 1] = bf16x2_times_2m8(v.y);
            w[4 * q + 2] = bf16x2_times_2m8(v.z);
            w[4 * q + 3] = bf16x2_times_2m8(v.w);
          }
          tmem_st32(tmem + lane_off + kTmemQ + 64 * g + 32 * h, w);
        }
      }
      tmem_wait_st();
      if (g == 0 && ok) {
        // the RoPE query columns (landed by TMA): this thread scales the 64 bytes of its row
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.q_full), 0, p.status, abort));
        if (ok) {
          uint4* qr = reinterpret_cast<uint4*>(smem + kOffQ + row * 64);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v = qr[u];
            v.x = bf16x2_times_2m8(v.x);
            v.y = bf16x2_times_2m8(v.y);
            v.z = bf16x2_times_2m8(v.z);
            v.w = bf16x2_times_2m8(v.w);
            qr[u] = v;
          }
          fence_proxy_async_smem();  // visible to the MMAs that read it
        }
      }
      tc_fence_before();
      mbar_arrive(bar_addr(bars.q_tmem));
    }
    // exchange buffer k, this row: 16-byte unit q at q * 2048 + row * 16
    uint8_t* xrow0 = smem + kOffX + row * 16;
    const uint32_t x_remote0 = mapa(smem_u32(xrow0), peer);
    const uint32_t xfull_remote0 = mapa(bar_addr(bars.x_full[0]), peer);  // the peer's x_full[k] is 8k bytes on
    const uint32_t s_addr0 = tmem + lane_off + kTmemS;
    const uint64_t scale2 = f32x2(kSumScaleLog2, kSumScaleLog2);
    float m_mine = -INFINITY, l = 0.f;  // reference max this warpgroup last used, and its partial sum
    for (int i = g; i < n_pages && ok; i += kRowWGs) {
      const int xb = i & 1;                      // score, exchange and P buffer of the page
      const int n_valid = min(kPage, t_end - (page_begin + i) * kPage);  // visible tokens of the page
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.s_full[i & 3]), (i >> 2) & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = s_addr0 + 64 * xb;
      // this CTA's partial scores S_r * 2^-8 as fp16 pairs: word w holds columns 2w, 2w + 1
      uint32_t mine[32];
      {
        uint32_t a[32], c[32];
        tmem_ld32(s_addr, a);
        tmem_ld32(s_addr + 32, c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_addr(bars.s_free[i & 3]));  // QK^T of page i + 2 may overwrite the buffer
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          mine[q] = pack_f16x2(__uint_as_float(a[2 * q]), __uint_as_float(a[2 * q + 1]));
          mine[16 + q] = pack_f16x2(__uint_as_float(c[2 * q]), __uint_as_float(c[2 * q + 1]));
        }
      }
      // send: wait until the peer has read what was sent for page i - 2 (same buffer)
      if (i >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_free[(i - 2) & 3]), ((i - 2) >> 2) & 1,
                                                       p.status, abort));
        if (!ok) break;
      }
      const uint32_t x_remote = x_remote0 + xb * kXBufBytes;
      const uint32_t xfull_remote = xfull_remote0 + 8 * (i & 3);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_async_v4(x_remote + q * (kRowThreads * 16), mine[4 * q], mine[4 * q + 1], mine[4 * q + 2], mine[4 * q + 3],
                    xfull_remote);
      // receive the peer's partial scores; both CTAs add fp16(S_0) + fp16(S_1)
      // in fp16, in the same order, so they hold the same S * 2^-8
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(bars.x_full[i & 3]), (i >> 2) & 1, p.status, abort));
      if (!ok) break;
      const uint8_t* xrow = xrow0 + xb * kXBufBytes;
      uint32_t sh[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(xrow + q * (kRowThreads * 16));
        sh[4 * q] = hadd2(mine[4 * q], v.x);
        sh[4 * q + 1] = hadd2(mine[4 * q + 1], v.y);
        sh[4 * q + 2] = hadd2(mine[4 * q + 2], v.z);
        sh[4 * q + 3] = hadd2(mine[4 * q + 3], v.w);
      }
      mbar_arrive(bar_addr(bars.x_read[xb]));  // warp 14 recycles the exchange buffer
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
      // the reference max after page i - 1 (from the warpgroup of page i - 1)
      bool rescale = false;
      float factor = 1.f;
      if (i == 0) {
        m_mine = mx;
      } else {
        const int gp = (i - 1) % kRowWGs;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.hand[gp]), ((i - 1) / kRowWGs) & 1, p.status, abort));
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
      // P = 2^(S * scale - m) in packed fp32 pairs; P goes to the MMA in bf16,
      // the row sum adds the fp32 values
      const uint64_t neg_m2 = f32x2(-m_mine, -m_mine);
      uint32_t pk[32];
      uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int w = 0; w < 32; ++w) {
        const float2 sf = unpack_f16x2(sh[w]);
        const float2 e = f32x2_split(fma_f32x2(f32x2(sf.x, sf.y), scale2, neg_m2));
        const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
        pk[w] = pack_bf16x2(p0, p1);
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
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[(i - 2) & 3]), ((i - 2) >> 2) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
      }
      uint8_t* prow = smem + kOffP + xb * kPBytes + row * 128;  // this row of P(i)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();  // visible to the P V MMAs
      if (__any_sync(0xffffffffu, rescale)) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[(i - 1) & 3]), ((i - 1) >> 2) & 1, p.status, abort));
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
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(bars.p_full[xb]));
    }
    // Exchanged partials are fp16(S_r / 256): one beyond |S_r| = 65520 * 256
    // (or a NaN) becomes infinite or NaN and leaves the row's max or sum non-finite.
    if (ok && g < n_pages && !(isfinite(l) && isfinite(m_mine))) record_status(p.status, MLA_ERR_RANGE);

    // epilogue: combine the warpgroups' sums, then warpgroup g < 2 writes
    // columns [128g, 128g + 128) of this CTA's half of O' (normalised)
    fin[g * kHeads + row] = make_float2(m_mine, l);
    if (!ok) bars.wg_bad[g] = 1;
    mbar_arrive(bar_addr(bars.fin));
    if (g < 2) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.fin), 0, p.status, abort));
      const int last = n_pages - 1;
      if (ok && last >= 0)
        ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(bars.pv_done[last & 3]), (last >> 2) & 1, p.status, abort));
      tc_fence_after();
      const int64_t out_row = (static_cast<int64_t>(bj) * p.num_splits + split) * kHeads + row;
      // One decision per warpgroup: its 128 x 128 tile of O' is staged in the
      // (now idle) ring and stored by TMA, or, if any row of the CTA has no
      // valid result, the warpgroup writes zeros directly.
      if (!ok && lane == 0) bars.wg_bad[g] = 1;
      named_barrier_sync(1 + g, kRowThreads);
      volatile int* wb = bars.wg_bad;
      bool any_bad = false;
#pragma unroll
      for (int k = 0; k < kRowWGs; ++k) any_bad = any_bad || wb[k] != 0;
      if (!any_bad && n_pages > 0) {
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < kRowWGs; ++k) m = fmaxf(m, fin[k * kHeads + row].x);
        float lt = 0.f;
#pragma unroll
        for (int k = 0; k < kRowWGs; ++k) {
          const float2 f = fin[k * kHeads + row];
          lt += f.y > 0.f ? f.y * ex2_approx(f.x - m) : 0.f;
        }
        const float inv = 1.f / lt;
        // four boxes of 32 fp32 columns x 128 rows, 128-byte swizzle: row r at
        // r * 128, 16-byte chunk c at (c ^ (r & 7)) * 16
        uint8_t* tile = smem + kOffStage + g * kOTileBytes;
        const int32_t y0 = static_cast<int32_t>(out_row) - row;  // row 0 of the unit
        if (p.out_bf16) {
          // a split's partial: two boxes of 64 bf16 columns x 128 rows, 128-byte
          // swizzle: row r at r * 128, 16-byte chunk c at (c ^ (r & 7)) * 16
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
                                  const SplitPlan& plan, void* o_out, float* lse_out,
                                  int* status, cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(B) * n_q * plan.num_splits;
  if (units == 0) return cudaSuccess;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || !configure(dev)) return cudaErrorInvalidDevice;
  CUtensorMap tqlat, tq64, tc128, tc64, to;
  const uint64_t q_rows = static_cast<uint64_t>(B) * n_q * kHeads;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  if (!make_tmap_bf16_chunks(&tqlat, q_abs, q_rows, kRow, 128, 4) ||
      !make_tmap_bf16_2d(&tq64, q_abs, q_rows, kRow, kRow, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_bf16_chunks(&tc128, cache, c_rows, kRow, 64, 4) ||
      !make_tmap_bf16_2d(&tc64, cache, c_rows, kRow, kRow, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const bool out_bf16 = plan.num_splits > 1;  // partials for the merge
  const uint64_t o_rows = static_cast<uint64_t>(units) * kHeads;
  if (out_bf16 ? !make_tmap_bf16_2d(&to, o_out, o_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)
               : !make_tmap_f32_2d(&to, o_out, o_rows, kLatent, kLatent, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.o_out = o_out;
  prm.lse_out = lse_out;
  prm.out_bf16 = out_bf16;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.n_q = n_q;
  prm.max_kv_len = max_kv_len;
  prm.split_pages = plan.split_pages;
  prm.num_splits = plan.num_splits;
  return launch_kernel(decode_attn_tc_kernel, dim3(static_cast<unsigned>(2 * units)), dim3(kThreads), kSmemBytes, stream,
                       tqlat, tq64, tc128, tc64, to, prm);
}

}  // namespace mla
