// Non-absorbed path, step 2: causal multi-head attention of a chunk of new
// tokens over the decompressed keys and values (the prefill / chunked-prefill form).
//
// "MLA 矩阵吸收 …" section 2.2 (Non-Absorbed: score = Q K^T on the decompressed
// K, standard MHA, O = softmax(score) V) and section 6 (FlashAttention-style
// kernel for the chunk); "DeepSeek-MLA-Principle" section 2: score =
// [q^C ; RoPE(q^R)] . [k^C ; k^R] / sqrt(d_h + d_h^R), eqs. (2)-(10), and
// section 6 (prefill is compute bound, the non-absorbed L^2 terms are ~3x smaller).
//
// Persistent: one CTA per SM walks a list of query tiles (sequence b, head h, 128
// new tokens).  The tiles are taken in units of two, tiles p and n_qt - 1 - p of
// one (b, h), so that under the causal mask every unit holds about the same
// number of key tiles; CTA c takes units c, c + G, c + 2G, ... in (b, h) order, so
// the heads in flight at once keep their keys and values in L2.  Every role walks
// the same tile list with running counters, so the rings and barrier phases run
// on across tiles without draining.
//
// Per tile: the query [q^C ; RoPE(q^R, pos)] (192 columns) goes to shared memory,
// q^C by two TMA boxes (128 tokens of one head) from the QK^T thread and the
// rotated q^R from the softmax warps; per 128-key tile one producer warp loads, by
// TMA, the head's decompressed keys (128 columns) and the shared RoPE key of the
// cache (64 columns, through the page table, whose entries it reads 32 at a time)
// into a 2-stage key ring, and another the values into a 2-stage value ring: a key
// stage is free again as soon as its S = Q K^T has been computed, so the next keys
// load while the softmax runs.  S (M = 128 queries, N = 128 keys, K = 192) goes to
// one of two TMEM buffers; the softmax warps (two threads per query, one per
// 64-key half of the tile) apply the causal mask and an online softmax with a
// lazily updated reference max (O is rescaled only when a row's max grows by more
// than 2^8), write P as bf16 into one of two TMEM buffers (so P of the next tile
// never waits for P V of this one), and O += P V (N = 128, K = 128 keys)
// accumulates in TMEM.  Query j of sequence b sits at position seq_lens_before[b]
// + j and sees the keys 0 .. seq_lens_before[b] + j.
//
// Between two query tiles: the next tile's query rows are pulled into L2 while
// the current tile runs; once the current tile's last QK^T has finished, the QK^T
// thread requests the next q^C and the softmax warps (having read the last scores)
// build the next RoPE chunk, before the current tile's epilogue; QK^T of the next
// tile then runs during that epilogue, and its first P V waits only until the
// epilogue has read O out of TMEM.  The epilogue transposes 16-byte units across
// lanes so that each warp store writes whole 128-byte lines of O.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kQTile = 128;
constexpr int kKTile = 128;
constexpr int kStages = 2;
// warp 0 key TMA, warp 1 QK^T issuer, warps 2-9 softmax (two per query row),
// warp 10 value TMA, warp 11 P V issuer
constexpr int kThreads = 384;
constexpr int kSoftWarp0 = 2;
constexpr int kVWarp = 10;
constexpr int kPvWarp = 11;
constexpr int kSoftThreads = 256;
constexpr int kChunk = 128 * 128;   // 128 rows x 64 bf16 columns (SW128)
constexpr int kOffQ = 0;            // query: 3 chunks (q^C 0-63, q^C 64-127, RoPE(q^R))
constexpr int kKStageBytes = 3 * kChunk;  // keys 2 chunks, RoPE keys 1
constexpr int kVStageBytes = 2 * kChunk;  // values 2 chunks
constexpr int kOffK = kOffQ + 3 * kChunk;
constexpr int kOffV = kOffK + kStages * kKStageBytes;
constexpr int kOffBar = kOffV + kStages * kVStageBytes;
constexpr int kOffHx = kOffBar + 256;           // half-row maxima [4][2][128], then row sums [2][128]
constexpr int kOffMeta = kOffHx + 4 * (4 * 2 * 128 + 2 * 128);  // per sequence: L and kv (up to kMetaCap)
constexpr int kMetaCap = 512;
constexpr int kSmemBytes = kOffMeta + 2 * 4 * kMetaCap + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemO = 0;      // O: [0, 128)
constexpr uint32_t kTmemS = 128;    // two score buffers: [128, 256), [256, 384)
constexpr uint32_t kTmemP = 384;    // two P buffers (128 keys as bf16 pairs): [384, 448), [448, 512)
constexpr float kRescaleLog2 = 8.f;

struct Bars {
  uint64_t kfull[kStages];
  uint64_t kempty[kStages];
  uint64_t vfull[kStages];
  uint64_t vempty[kStages];
  uint64_t q_ready;    // the RoPE query chunk of the next tile is in shared memory (one phase per tile)
  uint64_t q_full;     // its q^C chunks have landed (TMA; one phase per tile)
  uint64_t o_free;     // the epilogue has read O out of TMEM (one phase per tile)
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t hx[2];      // both halves of every row have published their half-row max
  uint64_t fin;        // both halves have published their row sums (one phase per tile)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  const int32_t* seq_lens_before;
  const float* rope;
  const int32_t* page_table;
  const int32_t* kv_lens;
  uint16_t* out;
  float* lse;
  int* status;
  int64_t num_pages;
  int pt_stride;
  int rope_max_pos;
  int max_kv_len;
  int n_q;
  int B;
  int n_qt;      // query tiles per (sequence, head)
  int n_pair;    // units per (sequence, head): tiles p and n_qt - 1 - p
  int n_units;   // B * heads * n_pair
};

// One query tile of this CTA's list and what it needs to know about its sequence.
struct Tile {
  int b, h, qt, L, kv, j0, n_kt;
  bool bad;
};

// The k-th tile of this CTA's list (k advanced past it); false once the list is done.
// Every role calls this in the same order, so all of them see the same tiles.  `meta`
// is the shared-memory copy of the sequences' L and kv (nullptr: read them globally).
__device__ __forceinline__ bool next_tile(const Params& p, const int* meta, int& k, Tile& t) {
  for (;;) {
    const int w = static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * (k >> 1);
    if (w >= p.n_units) return false;
    const int second = k & 1;
    ++k;
    const int pr = w % p.n_pair, bh = w / p.n_pair;
    const int q_hi = p.n_qt - 1 - pr;
    if (second && pr == q_hi) continue;  // the middle tile of an odd count is a unit alone
    t.b = bh / kHeads;
    t.h = bh % kHeads;
    t.qt = second ? pr : q_hi;
    t.L = meta != nullptr ? meta[t.b] : p.seq_lens_before[t.b];
    t.kv = meta != nullptr ? meta[kMetaCap + t.b] : p.kv_lens[t.b];
    t.bad = t.L < 0 || t.kv != t.L + p.n_q || t.kv > p.max_kv_len || (t.kv + kPage - 1) / kPage > p.pt_stride ||
            t.L + p.n_q > p.rope_max_pos;
    t.j0 = t.qt * kQTile;
    const int j_last = min(p.n_q, t.j0 + kQTile) - 1;  // last query of the tile
    t.n_kt = t.bad ? 0 : (t.L + j_last + 1 + kKTile - 1) / kKTile;
    return true;
  }
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_q,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.kfull[s]), 1);
      mbar_init(smem_u32(&bars.kempty[s]), 1);
      mbar_init(smem_u32(&bars.vfull[s]), 1);
      mbar_init(smem_u32(&bars.vempty[s]), 1);
    }
    mbar_init(smem_u32(&bars.q_ready), kSoftThreads);
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.o_free), kSoftThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.s_full[s]), 1);
      mbar_init(smem_u32(&bars.s_free[s]), kSoftThreads);
      mbar_init(smem_u32(&bars.p_full[s]), kSoftThreads);
      mbar_init(smem_u32(&bars.hx[s]), kSoftThreads);
      mbar_init(smem_u32(&bars.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&bars.drain), 2);  // both issuers
    mbar_init(smem_u32(&bars.fin), kSoftThreads);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  grid_dep_wait();
  grid_dep_launch();
  // every role walks the tile list, which needs each tile's sequence lengths
  int* meta = p.B <= kMetaCap ? reinterpret_cast<int*>(smem + kOffMeta) : nullptr;
  if (meta != nullptr) {
    for (int i = tid; i < p.B; i += kThreads) {
      meta[i] = p.seq_lens_before[i];
      meta[kMetaCap + i] = p.kv_lens[i];
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ key TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_kr);
    }
    bool ok = true;
    int k = 0, g = 0;  // tile list position, key tiles loaded so far
    Tile t;
    while (ok && next_tile(p, meta, k, t)) {
      if (t.n_kt == 0) {
        if (lane == 0 && t.bad && t.qt == 0 && t.h == 0) record_status(p.status, MLA_ERR_BOUNDS);
        continue;
      }
      const int row0 = (t.b * kHeads + t.h) * p.max_kv_len;  // this head's rows in K
      const int32_t* pt = p.page_table + static_cast<int64_t>(t.b) * p.pt_stride;
      const int n_pg = (t.kv + kPage - 1) / kPage;            // pages holding the sequence (<= pt_stride)
      int ids = 0;
      for (int kt = 0; kt < t.n_kt && ok; ++kt, ++g) {
        if ((kt & 15) == 0) {  // the page ids of key tiles kt .. kt + 15, one per lane
          const int q = 2 * kt + lane;
          ids = q < n_pg ? pt[q] : 0;
        }
        const int pg0 = __shfl_sync(0xffffffffu, ids, (2 * kt) & 31);
        const int pg1 = __shfl_sync(0xffffffffu, ids, (2 * kt + 1) & 31);
        if (lane == 0) {
          const int s = g % kStages;
          ok = mbar_wait(smem_u32(&bars.kempty[s]), ((g / kStages) & 1) ^ 1, p.status, abort);
          if (ok) {
            const uint32_t st = smem_u32(smem + kOffK + s * kKStageBytes);
            const uint32_t fb = smem_u32(&bars.kfull[s]);
            mbar_arrive_expect_tx(fb, kKStageBytes);
            for (int c = 0; c < 2; ++c) tma_load_2d(st + c * kChunk, &tm_k, 64 * c, row0 + kt * kKTile, fb);
            for (int pg = 0; pg < 2; ++pg) {
              const int tok = kt * kKTile + pg * kPage;
              int page = pg == 0 ? pg0 : pg1;
              if (tok >= t.kv) {
                page = 0;  // past the sequence: masked, any page will do
              } else if (page < 0 || page >= p.num_pages) {
                record_status(p.status, MLA_ERR_BOUNDS);
                page = 0;  // stay in bounds; the result of this tile is not meaningful
              }
              tma_load_2d(st + 2 * kChunk + pg * (kChunk / 2), &tm_kr, kLatent, page * kPage, fb);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ value TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      bool ok = true;
      int k = 0, g = 0;
      Tile t;
      while (ok && next_tile(p, meta, k, t)) {
        const int row0 = (t.b * kHeads + t.h) * p.max_kv_len;  // this head's rows in V
        for (int kt = 0; kt < t.n_kt; ++kt, ++g) {
          const int s = g % kStages;
          ok = mbar_wait(smem_u32(&bars.vempty[s]), ((g / kStages) & 1) ^ 1, p.status, abort);
          if (!ok) break;
          const uint32_t st = smem_u32(smem + kOffV + s * kVStageBytes);
          const uint32_t fb = smem_u32(&bars.vfull[s]);
          mbar_arrive_expect_tx(fb, kVStageBytes);
          for (int c = 0; c < 2; ++c) tma_load_2d(st + c * kChunk, &tm_v, 64 * c, row0 + kt * kKTile, fb);
        }
      }
    }
  } else if (warp == 1 || warp == kPvWarp) {
    // ------------------------------------------------------------ tcgen05 issuers
    // One thread issues QK^T and another P V: an MMA issue returns only once the
    // tensor pipe takes it, so with one issuer QK^T of the next key tile waited
    // behind P V of the previous one (and that behind its P).
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, 128, /*a_mn=*/0, /*b_mn=*/0);
      const uint32_t idesc_pv = idesc_bf16(128, 128, /*a_mn=*/0, /*b_mn=*/1);
      const uint64_t d_q = smem_desc(smem_u32(smem + kOffQ), 16, 1024, kSw128);
      const uint64_t d_k = smem_desc(smem_u32(smem + kOffK), 16, 1024, kSw128);           // keys (K-major)
      const uint64_t d_v = smem_desc(smem_u32(smem + kOffV), kChunk, 1024, kSw128);       // values (MN-major)
      bool ok = true;
      int k = 0, g = 0, n = 0;  // tile list position, key tiles issued, query tiles with keys
      Tile t;
      // q^C of a tile (128 tokens of one head, 32 KB apart in memory) by two TMA boxes
      auto load_qc = [&](const Tile& tt) {
        const uint32_t fb = smem_u32(&bars.q_full);
        mbar_arrive_expect_tx(fb, 2 * kChunk);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(smem_u32(smem + kOffQ + c * kChunk), &tm_q, 64 * c, tt.h, tt.b * p.n_q + tt.j0, fb);
      };
      if (warp == 1) tma_prefetch_desc(&tm_q);
      while (ok && next_tile(p, meta, k, t)) {
        if (t.n_kt == 0) continue;
        if (warp == 1) {
          if (n == 0) load_qc(t);
          ok = mbar_wait(smem_u32(&bars.q_full), n & 1, p.status, abort) &&
               mbar_wait(smem_u32(&bars.q_ready), n & 1, p.status, abort);
          for (int kt = 0; kt < t.n_kt && ok; ++kt, ++g) {
            const int s = g % kStages, buf = g & 1;
            ok = mbar_wait(smem_u32(&bars.kfull[s]), (g / kStages) & 1, p.status, abort) &&
                 mbar_wait(smem_u32(&bars.s_free[buf]), ((g >> 1) & 1) ^ 1, p.status, abort);
            if (!ok) break;
            tc_fence_after();
            const uint64_t so = static_cast<uint64_t>((s * kKStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 12; ++kk)  // K = 192: three 64-column chunks of four K steps
              mma_ss(tmem + kTmemS + 128 * buf, d_q + (kk >> 2) * (kChunk >> 4) + (kk & 3) * 2,
                     d_k + so + (kk >> 2) * (kChunk >> 4) + (kk & 3) * 2, idesc_qk, kk > 0 ? 1u : 0u);
            mma_commit(smem_u32(&bars.kempty[s]));   // the key stage may be refilled
            mma_commit(smem_u32(&bars.s_full[buf]));
          }
          // the next tile's q^C, as soon as this tile's last QK^T has finished reading
          // the query buffer (its completion is the last score buffer's barrier)
          Tile t2;
          int k2 = k;
          bool more = false;
          while (!more && next_tile(p, meta, k2, t2)) more = t2.n_kt > 0;
          if (ok && more) {
            ok = mbar_wait(smem_u32(&bars.s_full[(g - 1) & 1]), ((g - 1) >> 1) & 1, p.status, abort);
            if (ok) load_qc(t2);
          }
        } else {
          // the first P V of a tile overwrites O: only once the last tile's epilogue has read it
          if (n > 0) ok = mbar_wait(smem_u32(&bars.o_free), (n - 1) & 1, p.status, abort);
          for (int kt = 0; kt < t.n_kt && ok; ++kt, ++g) {
            const int s = g % kStages, buf = g & 1;
            ok = mbar_wait(smem_u32(&bars.p_full[buf]), (g >> 1) & 1, p.status, abort) &&
                 mbar_wait(smem_u32(&bars.vfull[s]), (g / kStages) & 1, p.status, abort);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vb = d_v + static_cast<uint64_t>((s * kVStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // K = 128 keys
              mma_ts(tmem + kTmemO, tmem + kTmemP + 64 * buf + 8 * kk, vb + 128 * kk, idesc_pv,
                     (kt > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&bars.vempty[s]));
            mma_commit(smem_u32(&bars.pv_done[buf]));
          }
        }
        ++n;
      }
      if (!ok) {
        record_status(p.status, MLA_ERR_TIMEOUT);
        *abort = 1;
      }
      // no tcgen05 operation may still be running when TMEM is released
      mma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax: two threads per query
    // Thread (row r, half hf) owns the key columns [64 hf, 64 hf + 64) of every key
    // tile and the output columns [64 hf, 64 hf + 64): the two halves of a row sit
    // in warps w and w + 4 (same TMEM lanes, same SM sub-partition), so one's
    // exponentials overlap the other's loads and waits.  They swap their half-row
    // maxima through shared memory and take identical decisions from them.
    const int quad = warp & 3;
    const int hf = (warp - kSoftWarp0) >> 2;
    const int r = quad * 32 + lane;       // query row of the tile (TMEM lane)
    const int st = tid - 32 * kSoftWarp0;  // 0 .. 255
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float* hmax = reinterpret_cast<float*>(smem + kOffHx);  // [4 tiles][2 halves][128 rows]
    float* fin = hmax + 4 * 2 * kQTile;                      // [2 halves][128 rows]
    uint8_t* qs = smem + kOffQ;

    // The RoPE chunk of a query tile, RoPE(q^R, pos) (the q^C chunks come by TMA), by
    // all 256 softmax threads in 16-byte units: consecutive lanes take consecutive
    // units of a row (the next token's row of the same head is 16 KB further on), so a
    // warp's load covers four rows instead of 32 separate lines.  Every load is issued
    // before the first shared-memory store (a store through a byte pointer may alias
    // any load).
    auto build_rope = [&](const Tile& t) {
      uint4 qr[4];       // q^R: unit u = st + 256 i, row u / 8, elements 8 (u % 8) .. + 7
      float4 cs[4][4];   // cos and sin of those elements' frequencies (two float4 each)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int u = st + 256 * i, rr = u >> 3, f0 = 8 * (u & 3);  // frequencies f0 .. f0 + 7
        if (!t.bad && t.j0 + rr < p.n_q) {
          const int64_t qrow = (static_cast<int64_t>(t.b) * p.n_q + t.j0 + rr) * kHeads + t.h;
          qr[i] = __ldg(reinterpret_cast<const uint4*>(p.q_rope + qrow * kRope) + (u & 7));
          const float4* tab = reinterpret_cast<const float4*>(p.rope + static_cast<int64_t>(t.L + t.j0 + rr) * kRope);
          cs[i][0] = __ldg(tab + f0 / 4);
          cs[i][1] = __ldg(tab + f0 / 4 + 1);
          cs[i][2] = __ldg(tab + (kHalfRope + f0) / 4);
          cs[i][3] = __ldg(tab + (kHalfRope + f0) / 4 + 1);
        } else {
          qr[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) cs[i][kk] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // rotate-half: element f < 32 pairs with f + 32, four units (lane ^ 4) away
        const int u = st + 256 * i;
        const bool second = (u & 4) != 0;   // this unit holds elements 32 + f
        const uint32_t mine[4] = {qr[i].x, qr[i].y, qr[i].z, qr[i].w};
        uint32_t other[4], w[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) other[kk] = __shfl_xor_sync(0xffffffffu, mine[kk], 4);
        const float c8[8] = {cs[i][0].x, cs[i][0].y, cs[i][0].z, cs[i][0].w,
                             cs[i][1].x, cs[i][1].y, cs[i][1].z, cs[i][1].w};
        const float s8[8] = {cs[i][2].x, cs[i][2].y, cs[i][2].z, cs[i][2].w,
                             cs[i][3].x, cs[i][3].y, cs[i][3].z, cs[i][3].w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          float o[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float a = __uint_as_float(e ? mine[kk] & 0xffff0000u : mine[kk] << 16);
            const float bb = __uint_as_float(e ? other[kk] & 0xffff0000u : other[kk] << 16);
            const float x1 = second ? bb : a, x2 = second ? a : bb;
            const float c = c8[2 * kk + e], sn = s8[2 * kk + e];
            o[e] = second ? __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn))
                          : __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn));
          }
          w[kk] = pack_bf16x2(o[0], o[1]);
        }
        *reinterpret_cast<uint4*>(qs + 2 * kChunk + sw128((u >> 3) * 128 + (u & 7) * 16)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.q_ready));
    };
    // The query rows of a tile (and their cos / sin rows) pulled into L2: 128 rows of
    // 2 + 1 lines, and 128 contiguous table rows of 256 bytes.
    auto prefetch_query = [&](const Tile& t) {
      if (t.bad) return;
      const int rr = st >> 1;
      if (t.j0 + rr < p.n_q) {
        const int64_t qrow = (static_cast<int64_t>(t.b) * p.n_q + t.j0 + rr) * kHeads + t.h;
        prefetch_l2(p.q_nope + qrow * kNope + (st & 1) * 64);
        if ((st & 1) == 0) prefetch_l2(p.q_rope + qrow * kRope);
        prefetch_l2(p.rope + static_cast<int64_t>(t.L + t.j0 + rr) * kRope + (st & 1) * 32);
      }
    };
    // The next tile of the list that has keys (tiles of an invalid sequence have none:
    // their live rows get O = 0 and lse = -inf here).
    int k = 0;
    auto next_active = [&](Tile& t) -> bool {
      while (next_tile(p, meta, k, t)) {
        if (t.n_kt > 0) return true;
        const int j = t.j0 + r;
        if (j < p.n_q) {
          const int64_t orow = (static_cast<int64_t>(t.b) * p.n_q + j) * kHeads + t.h;
          uint16_t* dst = p.out + orow * kNope + 64 * hf;
          for (int c0 = 0; c0 < 64; c0 += 8) *reinterpret_cast<uint4*>(dst + c0) = make_uint4(0, 0, 0, 0);
          if (hf == 0 && p.lse != nullptr) p.lse[orow] = -INFINITY;
        }
      }
      return false;
    };

    constexpr float kScaleL2 = kScaleLog2;
    const int c_off = 64 * hf;            // this thread's first key column of a tile
    bool ok = true;
    int g = 0, n = 0;                     // key tiles so far, query tiles so far
    Tile cur, nxt;
    bool have = next_active(cur);
    if (have) build_rope(cur);
    while (have && ok) {
      bool have_next = next_active(nxt);
      if (have_next) prefetch_query(nxt);
      const int j = cur.j0 + r;           // query index in the chunk
      const bool live = j < p.n_q;
      const int pos = cur.L + j;          // its position: sees keys 0 .. pos
      float m_ref = -INFINITY, l = 0.f;
      for (int kt = 0; kt < cur.n_kt && ok; ++kt, ++g) {
        const int buf = g & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[buf]), (g >> 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
        // keys kt*128 + c visible to this query: c < n_vis; this thread's columns c_off + c, c < n_mine
        const int n_vis = live ? max(0, min(kKTile, pos + 1 - kt * kKTile)) : (kt == 0 ? 1 : 0);
        const int n_mine = max(0, min(64, n_vis - c_off));
        float sv[64];
        {
          uint32_t v[2][32];  // both loads in flight, one wait
#pragma unroll
          for (int q = 0; q < 2; ++q) tmem_ld32(tmem + lane_off + kTmemS + 128 * buf + c_off + 32 * q, v[q]);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[32 * q + c] = __uint_as_float(v[q][c]);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.s_free[buf]));  // QK^T two key tiles on may overwrite the buffer
        // half-row max in eight independent chains, then the row max from both halves
        float m8[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) m8[kk] = -INFINITY;
        if (n_mine >= 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < n_mine) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
        }
        const float mh = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        // the slot of key tile g is written again at g + 4, after P V(g) (which needs
        // the partner's P of tile g, written after it read this value) has finished:
        // the wait for P V(g) comes before the P store of g + 2
        float* hx = hmax + (g & 3) * 2 * kQTile;
        hx[hf * kQTile + r] = mh;
        mbar_arrive(smem_u32(&bars.hx[buf]));
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.hx[buf]), (g >> 1) & 1, p.status, abort));
        if (!ok) break;
        float mx = fmaxf(mh, hx[(hf ^ 1) * kQTile + r]);
        mx *= kScaleL2;
        float factor = 1.f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = mx;  // first key tile with a visible key (or still -inf)
        } else if (mx > m_ref + kRescaleLog2) {
          factor = ex2_approx(m_ref - mx);
          m_ref = mx;
          rescale = true;
        }
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        // P = 2^(S scale - m): exponent arguments on packed fp32 pairs; the row sum
        // adds the float32 weights before their rounding to bf16 (round-to-nearest-even
        // is unbiased), in four independent pair chains.  Only a row's diagonal key
        // tile has masked columns, so the other tiles skip the compare and select.
        uint32_t pk[32];
        const uint64_t scale2 = f32x2(kScaleL2, kScaleL2), negm2 = f32x2(neg_m, neg_m);
        uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
        if (n_mine >= 64) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 e = f32x2_split(fma_f32x2(f32x2(sv[2 * c], sv[2 * c + 1]), scale2, negm2));
            const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
            pk[c] = pack_bf16x2(p0, p1);
            s4[c & 3] = add_f32x2(s4[c & 3], f32x2(p0, p1));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 e = f32x2_split(fma_f32x2(f32x2(sv[2 * c], sv[2 * c + 1]), scale2, negm2));
            float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
            if (2 * c >= n_mine) p0 = 0.f;
            if (2 * c + 1 >= n_mine) p1 = 0.f;
            pk[c] = pack_bf16x2(p0, p1);
            s4[c & 3] = add_f32x2(s4[c & 3], f32x2(p0, p1));
          }
        }
        const float2 s2 = f32x2_split(add_f32x2(add_f32x2(s4[0], s4[1]), add_f32x2(s4[2], s4[3])));
        l = l * factor + (s2.x + s2.y);
        // P buffer g & 1 is free once P V(g - 2) has finished (of this tile or the
        // last); O may only be rescaled once P V(g - 1) of this tile has
        if (g >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[buf]), ((g - 2) >> 1) & 1, p.status, abort));
          if (!ok) break;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale)) {
          if (kt >= 1) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&bars.pv_done[buf ^ 1]), ((g - 1) >> 1) & 1, p.status, abort));
            if (!ok) break;
            tc_fence_after();
          }
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kTmemO + c_off + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * factor);
            tmem_st32(tmem + lane_off + kTmemO + c_off + c0, v);
          }
        }
        tmem_st32(tmem + lane_off + kTmemP + 64 * buf + 32 * hf, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[buf]));
      }
      if (!ok) break;
      // this tile's last scores have been read, so its QK^T is done with the query
      // buffer: the next tile's RoPE query goes in now (its q^C by TMA from the QK^T
      // thread) and its QK^T runs during the epilogue
      if (have_next) build_rope(nxt);
      const int g_last = g - 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars.pv_done[g_last & 1]), (g_last >> 1) & 1, p.status, abort));
      // the row sum from both halves (both rescaled against the same reference max)
      fin[hf * kQTile + r] = l;
      mbar_arrive(smem_u32(&bars.fin));
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.fin), n & 1, p.status, abort)) && ok;
      if (!ok) break;
      const float lt = fin[r] + fin[kQTile + r];
      tc_fence_after();
      // epilogue: O / l as bf16 (this thread's 64 columns), and the natural log-sum-exp.
      // tcgen05.ld is a warp-wide instruction, so every lane loads and only live rows store.
      uint32_t v[2][32];
#pragma unroll
      for (int q = 0; q < 2; ++q) tmem_ld32(tmem + lane_off + kTmemO + c_off + 32 * q, v[q]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free));  // the next tile's first P V may overwrite O
      // this row's 64 columns as eight 16-byte units, then an 8 x 8 transpose of the
      // units across each aligned group of 8 lanes (butterfly over lane bits 4, 2, 1):
      // lane a then holds unit a of the group's 8 rows, so a warp's store covers 4 rows
      // x 128 contiguous bytes instead of 32 rows 32 KB apart
      const float inv = live ? 1.f / lt : 0.f;
      uint4 x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t* y = &v[q >> 2][8 * (q & 3)];
        x[q] = make_uint4(pack_bf16x2(__uint_as_float(y[0]) * inv, __uint_as_float(y[1]) * inv),
                          pack_bf16x2(__uint_as_float(y[2]) * inv, __uint_as_float(y[3]) * inv),
                          pack_bf16x2(__uint_as_float(y[4]) * inv, __uint_as_float(y[5]) * inv),
                          pack_bf16x2(__uint_as_float(y[6]) * inv, __uint_as_float(y[7]) * inv));
      }
      const int a8 = lane & 7;
#pragma unroll
      for (int sh = 2; sh >= 0; --sh) {
        const int m = 1 << sh;
        const bool hi = (a8 & m) != 0;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (jj & m) continue;
          const uint4 snd = hi ? x[jj] : x[jj | m];
          uint4 rcv;
          rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
          rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
          rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, m);
          rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, m);
          if (hi) x[jj] = rcv;
          else x[jj | m] = rcv;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int jr = cur.j0 + quad * 32 + (lane & ~7) + i;  // the row whose unit a8 is x[i]
        if (jr < p.n_q) {
          const int64_t orow = (static_cast<int64_t>(cur.b) * p.n_q + jr) * kHeads + cur.h;
          *reinterpret_cast<uint4*>(p.out + orow * kNope + c_off + 8 * a8) = x[i];
        }
      }
      if (live && hf == 0 && p.lse != nullptr)
        p.lse[(static_cast<int64_t>(cur.b) * p.n_q + j) * kHeads + cur.h] = (m_ref + log2f(lt)) * kLn2;
      ++n;
      cur = nxt;
      have = have_next;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool g_configured[64];
int g_sms[64];

}  // namespace

cudaError_t launch_prefill_attn(const uint16_t* q_nope, const uint16_t* q_rope, const int32_t* seq_lens_before,
                                const float* rope_table, int rope_max_pos, const uint16_t* k_nope,
                                const uint16_t* v, int max_kv_len, const uint16_t* cache, int64_t num_pages,
                                const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                uint16_t* out, float* lse, int* status, cudaStream_t stream) {
  if (B == 0 || n_q == 0) return cudaSuccess;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_configured[dev] = true;
  }
  CUtensorMap tk, tv, tkr, tq;
  const uint64_t kv_rows = static_cast<uint64_t>(B) * kHeads * max_kv_len;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  if (!make_tmap_bf16_2d(&tk, k_nope, kv_rows, kNope, kNope, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&tv, v, kv_rows, kNope, kNope, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&tkr, cache, c_rows, kRow, kRow, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      // q^C [B n_q tokens][heads][128]: box of 64 columns x 1 head x 128 tokens
      !make_tmap_bf16_3d(&tq, q_nope, kNope, kHeads, static_cast<uint64_t>(B) * n_q, kNope * 2,
                         static_cast<uint64_t>(kHeads) * kNope * 2, 64, 1, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.q_nope = q_nope;
  prm.q_rope = q_rope;
  prm.seq_lens_before = seq_lens_before;
  prm.rope = rope_table;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.out = out;
  prm.lse = lse;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.rope_max_pos = rope_max_pos;
  prm.max_kv_len = max_kv_len;
  prm.n_q = n_q;
  prm.B = B;
  prm.n_qt = (n_q + kQTile - 1) / kQTile;
  prm.n_pair = (prm.n_qt + 1) / 2;
  prm.n_units = B * kHeads * prm.n_pair;
  const int grid = prm.n_units < g_sms[dev] ? prm.n_units : g_sms[dev];
  return launch_kernel(prefill_attn_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, tk, tv, tkr, tq, prm);
}

}  // namespace mla
