// Non-absorbed path, step 1: per-head keys and values decompressed from the
// latent cache, K[b, h, t, :] = W_UK[h] c_t and V[b, h, t, :] = W_UV[h] c_t.
//
// "MLA 矩阵吸收 …" section 2.2 (Non-Absorbed, the prefill form: K = c_t W_UK,
// V = c_t W_UV decompressed first, then standard MHA) and section 6 (the switch
// to this path for chunks of about 64 new tokens or more); "DeepSeek-MLA-
// Principle" section 6 (prefill vs decode, the L^2 terms favour decompression).
//
// A dense contraction per 128-token tile of a sequence: the tile's latent rows
// C (128 x 512) against the 128 per-head weight pairs [W_UK[h]; W_UV[h]]
// (256 x 512).  The two CTAs of a cluster take two consecutive tiles through the
// same heads: the work is a list of units (tile pair, head), tile-major, and
// each persistent cluster (one CTA per SM) takes a contiguous range of it, so the
// ranges differ by at most one unit and a cluster changes tile pairs about
// twice.  Of every weight slot, CTA 0 loads the W_UK chunk and CTA 1 the W_UV
// chunk, each multicast to both: the weights stream from L2, and L2's bandwidth
// into the SMs bounded a CTA that fetched all of them itself.
//
// The latent rows are the A operand of all 128 units of their tile, so they sit
// in TMEM (256 columns of bf16 pairs) for the whole tile and the MMAs read only
// the weights from shared memory.  One MMA (M = 128 tokens, N = 256, K = 16)
// makes the head's keys and values together: an MMA holds its issuing thread
// ~113 cycles at N = 128 and ~138 at N = 256 (A in TMEM), so N = 256 does twice
// the work for 1.2 times the issue time.  That leaves a single 256-column
// accumulator beside the latent rows.  Two epilogue warpgroups, one for the
// keys' 128 columns and one for the values', move it to registers together (the
// MMAs of the next head wait for that), hand it back, and then convert their
// half to bf16 and store it by TMA, one 64-column box at a time from a staging
// box of their own.  Weights stream from L2 in 32 KB slots (64 K-columns of
// W_UK[h] and of W_UV[h]) through a 6-slot ring; a tile's latent rows come
// through the same ring, two 64-column chunks per slot, issued after the last
// weight slot of the tile before, and the epilogue warps move them into TMEM
// once the MMAs of that tile are done, then release their slots.  A slot is
// refilled once both CTAs have consumed it.  Rows of a tile past the sequence's
// length are written as zeros (an attention kernel that reads whole 128-token
// tiles multiplies finite values there); tiles past it are not touched.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTile = 128;                  // tokens per tile
constexpr int kUnitsPerTile = kHeads;       // unit w of a tile: head w, keys and values
constexpr int kChunkBytes = 128 * 128;      // 128 rows x 64 bf16 columns (SW128)
constexpr int kSlotBytes = 2 * kChunkBytes;  // a ring slot: two such chunks
constexpr int kStages = 6;                  // ring slots
constexpr int kASlots = 4;                  // latent rows of a tile: 8 chunks of 64 columns, 2 per slot
// With each weight slot the producer pulls the one kL2Ahead slots later into L2,
// so that the ring's loads do not wait for DRAM: the weights' lines compete in L2
// with the keys and values streaming out.
constexpr int kL2Ahead = 12;
constexpr uint16_t kBoth = 0x3;             // both CTAs of the cluster
constexpr int kThreads = 320;               // warp 0 TMA, warp 1 MMA, warps 2-5 keys, warps 6-9 values
constexpr int kTmaWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiThreads = 256;            // both epilogue warpgroups
constexpr int kGroupThreads = 128;          // one of them
constexpr int kOffRing = 0;
constexpr int kOffO = kOffRing + kStages * kSlotBytes;  // output boxes (keys, values): 64 columns each
constexpr int kOffBar = kOffO + 2 * kChunkBytes;
constexpr int kSmemBytes = kOffBar + 512 + 1024;       // + 1 KB alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kASlots < kStages, "a tile's latent chunks fit the ring beside a weight slot");
constexpr uint32_t kTmemD = 0;    // accumulator: keys in columns [0, 128), values in [128, 256)
constexpr uint32_t kTmemA = 256;  // latent rows of the current tile, bf16 pairs: columns [256, 512)

struct Bars {
  uint64_t full[kStages];   // the slot's chunks have landed
  uint64_t empty[kStages];  // both CTAs have consumed the slot's chunks (MMAs finished, or moved to TMEM)
  uint64_t a_moved;         // the CTA's k-th tile's latent rows are in TMEM
  uint64_t a_free;          // the MMAs of the k-th tile have finished: TMEM A may be overwritten
  uint64_t d_full;          // the accumulator holds the current unit
  uint64_t d_empty;         // the epilogue has read it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  int* status;
  int64_t num_pages;
  int64_t units;        // tile pairs * kUnitsPerTile
  int64_t total_tiles;  // B * tiles
  int pt_stride;
  int max_kv_len;
  int tiles;      // tiles per sequence, ceil(max_kv_len / 128)
};

// Global tile g: its sequence, first token, tokens of the sequence in it (0 for
// none, for a sequence whose length is inconsistent, or for g past the last tile).
struct TileInfo {
  int b, t0, valid;
  bool bad;
};
__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t g) {
  TileInfo ti;
  if (g >= p.total_tiles) {
    ti.b = 0;
    ti.t0 = 0;
    ti.valid = 0;
    ti.bad = false;
    return ti;
  }
  ti.b = static_cast<int>(g / p.tiles);
  ti.t0 = static_cast<int>(g % p.tiles) * kTile;
  const int kv = p.kv_lens[ti.b];
  ti.bad = kv < 0 || kv > p.max_kv_len || (kv + kPage - 1) / kPage > p.pt_stride;
  ti.valid = ti.bad ? 0 : max(0, min(kTile, kv - ti.t0));
  return ti;
}

// Tile pair q is live if either of its tiles holds tokens: both CTAs then run it.
__device__ __forceinline__ bool pair_live(const Params& p, int64_t q) {
  return tile_info(p, 2 * q).valid > 0 || tile_info(p, 2 * q + 1).valid > 0;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decompress_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_wk,
                        const __grid_constant__ CUtensorMap tm_wv, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  // this cluster's units [u_begin, u_end); the CTA works on tile 2 q + rank of pair q
  const int64_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int64_t u_begin = p.units * cluster / clusters;
  const int64_t u_end = p.units * (cluster + 1) / clusters;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);
      mbar_init(smem_u32(&bars.empty[s]), 2);  // one consumer in each CTA
    }
    mbar_init(smem_u32(&bars.a_moved), kEpiThreads);
    mbar_init(smem_u32(&bars.a_free), 1);
    mbar_init(smem_u32(&bars.d_full), 1);
    mbar_init(smem_u32(&bars.d_empty), kEpiThreads);
    mbar_init(smem_u32(&bars.drain), 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  cluster_sync();  // the peer's barriers exist before any chunk is multicast or slot released
  grid_dep_wait();
  grid_dep_launch();

  // Every role walks the same tiles of [u_begin, u_end) in the same order and
  // skips the same empty ones, so they agree on the k-th tile, the i-th unit and
  // the n-th ring slot: per tile, 4 latent slots, then 8 weight slots per unit.
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_c);
      tma_prefetch_desc(&tm_wk);
      tma_prefetch_desc(&tm_wv);
      bool ok = true;
      int n = 0;  // slots issued
      auto slot = [&](int& s) {
        s = n % kStages;
        ok = mbar_wait(smem_u32(&bars.empty[s]), ((n / kStages) & 1) ^ 1, p.status, abort);
        if (ok) mbar_arrive_expect_tx(smem_u32(&bars.full[s]), kSlotBytes);
        return ok;
      };
      for (int64_t u = u_begin; u < u_end && ok;) {
        const int64_t q = u / kUnitsPerTile;
        const int64_t u_hi = min(u_end, (q + 1) * kUnitsPerTile);
        const TileInfo ti = tile_info(p, 2 * q + rank);
        if (ti.bad) record_status(p.status, MLA_ERR_BOUNDS);
        if (pair_live(p, q)) {
          // the tile's latent rows: two 64-token pages per chunk; a page past the
          // sequence's end (or of a tile with no tokens) is read from page 0 (its
          // rows are not stored)
          int page[2] = {0, 0};
          for (int pg = 0; pg < 2; ++pg) {
            if (pg * kPage < ti.valid) {
              page[pg] = p.page_table[static_cast<int64_t>(ti.b) * p.pt_stride + ti.t0 / kPage + pg];
              if (page[pg] < 0 || page[pg] >= p.num_pages) {
                record_status(p.status, MLA_ERR_BOUNDS);
                page[pg] = 0;  // stay in bounds; the result of this tile is not meaningful
              }
            }
          }
          for (int j = 0; j < kASlots && ok; ++j, ++n) {
            int s;
            if (!slot(s)) break;
            for (int cc = 0; cc < 2; ++cc)
              for (int pg = 0; pg < 2; ++pg)
                tma_load_2d(smem_u32(smem + kOffRing + s * kSlotBytes + cc * kChunkBytes + pg * (kChunkBytes / 2)),
                            &tm_c, 64 * (2 * j + cc), page[pg] * kPage, smem_u32(&bars.full[s]));
          }
          for (int64_t w = u; w < u_hi && ok; ++w) {
            const int h = static_cast<int>(w % kUnitsPerTile);
            for (int kc = 0; kc < 8 && ok; ++kc, ++n) {
              const CUtensorMap* tm = rank ? &tm_wv : &tm_wk;  // this CTA's half of the slot
              const int64_t wa = w + (kc + kL2Ahead) / 8;  // unit of the slot kL2Ahead on
              if (wa < u_end)
                tma_prefetch_l2_2d(tm, 64 * ((kc + kL2Ahead) % 8), static_cast<int>(wa % kUnitsPerTile) * kNope);
              int s;
              if (!slot(s)) break;
              // rows 0-127 of the B operand: W_UK[h] (from CTA 0); rows 128-255:
              // W_UV[h] (from CTA 1); each lands in both CTAs' slot s
              tma_load_2d_mc(smem_u32(smem + kOffRing + s * kSlotBytes + rank * kChunkBytes), tm, 64 * kc, h * kNope,
                             smem_u32(&bars.full[s]), kBoth);
            }
          }
        }
        u = u_hi;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 256, /*a_mn=*/0, /*b_mn=*/0);
      const uint64_t d_w = smem_desc(smem_u32(smem + kOffRing), 16, 1024, kSw128);
      bool ok = true;
      int k = 0, i = 0, n = 0;  // tiles, units, ring slots
      for (int64_t u = u_begin; u < u_end && ok;) {
        const int64_t q = u / kUnitsPerTile;
        const int64_t u_hi = min(u_end, (q + 1) * kUnitsPerTile);
        if (pair_live(p, q)) {
          n += kASlots;  // the latent slots are the epilogue warps'
          ok = mbar_wait(smem_u32(&bars.a_moved), k & 1, p.status, abort);
          for (int64_t w = u; w < u_hi && ok; ++w, ++i) {
            ok = mbar_wait(smem_u32(&bars.d_empty), (i & 1) ^ 1, p.status, abort);
            tc_fence_after();
            for (int kc = 0; kc < 8 && ok; ++kc, ++n) {
              const int s = n % kStages;
              ok = mbar_wait(smem_u32(&bars.full[s]), (n / kStages) & 1, p.status, abort);
              if (!ok) break;
              tc_fence_after();
              // A: latent columns [64 kc + 16 k4, +16) = TMEM columns kTmemA + 32 kc + 8 k4
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                mma_ts(tmem + kTmemD, tmem + kTmemA + 32 * kc + 8 * k4, d_w + ((s * kSlotBytes) >> 4) + 2 * k4,
                       idesc, (kc > 0 || k4 > 0) ? 1u : 0u);
              mma_commit_mc(smem_u32(&bars.empty[s]), kBoth);  // the slot is free here and in the peer
            }
            if (ok) mma_commit(smem_u32(&bars.d_full));
          }
          if (ok) mma_commit(smem_u32(&bars.a_free));
          ++k;
        }
        u = u_hi;
      }
      // no tcgen05 operation may still be running when TMEM is released
      mma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue: token rows
    // Warpgroup x (warps 2-5: x = 0, keys; warps 6-9: x = 1, values); thread r
    // owns token row r of the tile (TMEM lane r) and the accumulator's columns
    // [128 x, 128 x + 128).  The four warps of a warpgroup leave their loop
    // together: each wait's outcome is ANDed over them.
    const int x = (warp - kEpiWarp0) >> 2;
    const uint32_t bar_id = 1 + x;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = warp == kEpiWarp0 + 4 * x && lane == 0;
    uint8_t* stage = smem + kOffO + x * kChunkBytes;
    bool ok = true;
    int k = 0, i = 0, n = 0;
    for (int64_t u = u_begin; u < u_end && ok;) {
      const int64_t q = u / kUnitsPerTile;
      const int64_t u_hi = min(u_end, (q + 1) * kUnitsPerTile);
      const TileInfo ti = tile_info(p, 2 * q + rank);
      if (pair_live(p, q)) {
        // latent chunks 4x .. 4x + 3 (ring slots n + 2x, n + 2x + 1) into TMEM,
        // once the last tile's MMAs are done
        bool okl = k == 0 || mbar_wait(smem_u32(&bars.a_free), (k - 1) & 1, p.status, abort);
        for (int j = 0; j < 2; ++j)
          okl = okl && mbar_wait(smem_u32(&bars.full[(n + 2 * x + j) % kStages]), ((n + 2 * x + j) / kStages) & 1,
                                 p.status, abort);
        ok = named_barrier_and(bar_id, kGroupThreads, okl);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 4 * x; c < 4 * x + 4; ++c) {
          // row r of latent chunk c: page 0's rows, then page 1's, 128 bytes each
          const uint8_t* src =
              smem + kOffRing + ((n + c / 2) % kStages) * kSlotBytes + (c & 1) * kChunkBytes + r * 128;
          uint32_t wv[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + ((e ^ (r & 7)) << 4));
            wv[4 * e] = v.x;
            wv[4 * e + 1] = v.y;
            wv[4 * e + 2] = v.z;
            wv[4 * e + 3] = v.w;
          }
          tmem_st32(tmem + lane_off + kTmemA + 32 * c, wv);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.a_moved));
        // every thread of the warpgroup has read its two slots: they are free
        // here (and in the peer)
        named_barrier_sync(bar_id, kGroupThreads);
        if (leader)
          for (int j = 0; j < 2; ++j) {
            const uint32_t e = smem_u32(&bars.empty[(n + 2 * x + j) % kStages]);
            mbar_arrive(e);
            mbar_arrive_remote(mapa(e, peer));
          }
        n += kASlots;
        ++k;
        const bool live = r < ti.valid;
        for (int64_t w = u; w < u_hi; ++w, ++i) {
          n += 8;  // the unit's weight slots are the MMAs'
          const int h = static_cast<int>(w % kUnitsPerTile);
          // the last unit's TMA stores have read this warpgroup's output box
          if (leader) bulk_wait_read<0>();
          ok = named_barrier_and(bar_id, kGroupThreads, mbar_wait(smem_u32(&bars.d_full), i & 1, p.status, abort));
          if (!ok) break;
          tc_fence_after();
          // this warpgroup's 128 columns into registers as bf16 pairs: word j
          // holds columns 128 x + 2j, 128 x + 2j + 1
          uint32_t kv[64];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t va[32], vb[32];
            tmem_ld32(tmem + lane_off + kTmemD + 128 * x + 64 * c2, va);
            tmem_ld32(tmem + lane_off + kTmemD + 128 * x + 64 * c2 + 32, vb);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              kv[32 * c2 + e] = live ? pack_bf16x2(__uint_as_float(va[2 * e]), __uint_as_float(va[2 * e + 1])) : 0u;
              kv[32 * c2 + 16 + e] =
                  live ? pack_bf16x2(__uint_as_float(vb[2 * e]), __uint_as_float(vb[2 * e + 1])) : 0u;
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.d_empty));  // with the other warpgroup's: the next head may start
          // the two 64-column boxes in turn: row r into the staging box (128-byte
          // rows, 16-byte unit e at (e ^ (r & 7)) * 16), then one TMA store
          uint8_t* orow = stage + r * 128;
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            if (bx == 1) {
              if (leader) bulk_wait_read<0>();  // the first box's store has read the staging box
              named_barrier_sync(bar_id, kGroupThreads);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *reinterpret_cast<uint4*>(orow + ((e ^ (r & 7)) << 4)) =
                  make_uint4(kv[32 * bx + 4 * e], kv[32 * bx + 4 * e + 1], kv[32 * bx + 4 * e + 2],
                             kv[32 * bx + 4 * e + 3]);
            fence_proxy_async_smem();  // the box is visible to the TMA store
            named_barrier_sync(bar_id, kGroupThreads);
            if (leader && ti.valid > 0) {  // a tile with no tokens is not stored
              const CUtensorMap* tm = x ? &tm_v : &tm_k;
              tma_store_3d(tm, smem_u32(stage), 64 * bx, ti.t0, ti.b * kHeads + h);
              bulk_commit_group();
            }
          }
        }
      }
      u = u_hi;
    }
    if (leader) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  cluster_sync();  // no CTA leaves while its peer may still address its shared memory
}

bool g_configured[64];
int g_cluster_slots[64];

// Clusters of this kernel that can be resident at once (the persistent grid is
// sized to one wave of them).
int cluster_slots(int dev, int sms) {
  if (g_cluster_slots[dev] > 0) return g_cluster_slots[dev];
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
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decompress_kv_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  g_cluster_slots[dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_decompress_kv(const uint16_t* cache, int64_t num_pages, const int32_t* page_table, int pt_stride,
                                 const int32_t* kv_lens, int B, int max_kv_len, const uint16_t* w_uk,
                                 const uint16_t* w_uv, uint16_t* k_out, uint16_t* v_out, int* status,
                                 cudaStream_t stream) {
  if (B == 0 || max_kv_len == 0) return cudaSuccess;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decompress_kv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    g_configured[dev] = true;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return cudaErrorInvalidDevice;
  CUtensorMap tc, twk, twv, tk, tv;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  const uint64_t w_rows = static_cast<uint64_t>(kHeads) * kNope;
  const uint64_t bh = static_cast<uint64_t>(B) * kHeads;
  const uint64_t row_bytes = kNope * 2;
  // K and V as [B * 128 heads][max_kv_len tokens][128]: a 128-token box that runs
  // past max_kv_len is clipped there instead of spilling into the next head
  if (!make_tmap_bf16_2d(&tc, cache, c_rows, kRow, kRow, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&twk, w_uk, w_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&twv, w_uv, w_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_3d(&tk, k_out, kNope, max_kv_len, bh, row_bytes, row_bytes * max_kv_len, 64, kTile, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_3d(&tv, v_out, kNope, max_kv_len, bh, row_bytes, row_bytes * max_kv_len, 64, kTile, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.max_kv_len = max_kv_len;
  prm.tiles = (max_kv_len + kTile - 1) / kTile;
  prm.total_tiles = static_cast<int64_t>(B) * prm.tiles;
  prm.units = (prm.total_tiles + 1) / 2 * kUnitsPerTile;
  const int slots = cluster_slots(dev, sms);
  const int64_t clusters = prm.units < slots ? prm.units : slots;
  const int64_t grid = 2 * (clusters > 0 ? clusters : 1);
  return launch_kernel(decompress_kv_tc_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes,
                       stream, tc, twk, twv, tk, tv, prm);
}

}  // namespace mla
