// Non-absorbed path, step 1: per-head keys and values decompressed from the
// latent cache, K[b, h, t, :] = W_UK[h] c_t and V[b, h, t, :] = W_UV[h] c_t.
//
// "MLA 矩阵吸收 …" section 2.2 (Non-Absorbed, the prefill form: K = c_t W_UK,
// V = c_t W_UV decompressed first, then standard MHA) and section 6 (the switch
// to this path for chunks of about 64 new tokens or more); "DeepSeek-MLA-
// Principle" section 6 (prefill vs decode, the L^2 terms favour decompression).
//
// One CTA per (sequence, 128-token tile, group of 8 heads).  The tile's latent
// rows (128 x 512 bf16, 128 KB) are read once by TMA from the paged cache into
// shared memory and stay there; for each of the 8 heads and for W_UK and W_UV
// the 128 x 512 weight matrix streams through a 4-slot ring in 64-column chunks,
// one chain of 32 tcgen05 MMAs (M = 128 tokens, N = 128, K = 512) accumulates in
// one of four 128-column TMEM buffers, and four epilogue warps convert and store
// the buffer while the next head's MMAs run.  Rows of the tile past the
// sequence's length are written as zeros, so an attention kernel that reads whole
// 128-token tiles multiplies finite values there.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTile = 128;          // tokens per CTA
constexpr int kHeadsPerCta = 8;
constexpr int kUnits = 2 * kHeadsPerCta;  // (head, K or V)
constexpr int kWStages = 4;
constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16 columns (SW128)
constexpr int kOffA = 0;                 // 8 latent chunks of the tile
constexpr int kOffW = kOffA + 8 * kChunkBytes;
constexpr int kOffBar = kOffW + kWStages * kChunkBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
  uint64_t a_full;
  uint64_t w_full[kWStages];
  uint64_t w_empty[kWStages];
  uint64_t d_full[4];
  uint64_t d_empty[4];
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const int32_t* page_table;
  const int32_t* kv_lens;
  uint16_t* k_out;
  uint16_t* v_out;
  int* status;
  int64_t num_pages;
  int pt_stride;
  int max_kv_len;
};

__global__ void __launch_bounds__(kThreads, 1)
decompress_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_wk,
                        const __grid_constant__ CUtensorMap tm_wv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;

  grid_dep_wait();
  grid_dep_launch();
  const int kv = p.kv_lens[b];
  if (kv < 0 || kv > p.max_kv_len || (kv + kPage - 1) / kPage > p.pt_stride) {
    if (tid == 0 && tile == 0 && hg == 0) record_status(p.status, MLA_ERR_BOUNDS);
    return;
  }
  const int t0 = tile * kTile;
  if (t0 >= kv) return;  // nothing of this sequence in the tile
  const int valid = min(kTile, kv - t0);

  if (tid == 0) {
    mbar_init(smem_u32(&bars.a_full), 1);
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(smem_u32(&bars.w_full[s]), 1);
      mbar_init(smem_u32(&bars.w_empty[s]), 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(smem_u32(&bars.d_full[s]), 1);
      mbar_init(smem_u32(&bars.d_empty[s]), 128);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_c);
      tma_prefetch_desc(&tm_wk);
      tma_prefetch_desc(&tm_wv);
      // the tile's latent rows: two 64-token pages x eight 64-column chunks
      mbar_arrive_expect_tx(smem_u32(&bars.a_full), 8 * kChunkBytes);
      for (int pg = 0; pg < 2; ++pg) {
        int page = 0;
        if (pg * kPage < valid) {
          page = p.page_table[static_cast<int64_t>(b) * p.pt_stride + (t0 / kPage) + pg];
          if (page < 0 || page >= p.num_pages) {
            record_status(p.status, MLA_ERR_BOUNDS);
            page = 0;  // stay in bounds; the result of this tile is not meaningful
          }
        }
        for (int c = 0; c < 8; ++c)
          tma_load_2d(smem_u32(smem + kOffA + c * kChunkBytes + pg * (kChunkBytes / 2)), &tm_c, 64 * c,
                      page * kPage, smem_u32(&bars.a_full));
      }
      // weight chunks: unit u = (head kHeadsPerCta*hg + u/2, u%2 ? W_UV : W_UK), 8 chunks each
      for (int i = 0; i < kUnits * 8; ++i) {
        const int u = i >> 3, kc = i & 7, s = i % kWStages;
        if (!mbar_wait(smem_u32(&bars.w_empty[s]), ((i / kWStages) & 1) ^ 1, p.status, abort)) break;
        const int h = kHeadsPerCta * hg + (u >> 1);
        mbar_arrive_expect_tx(smem_u32(&bars.w_full[s]), kChunkBytes);
        tma_load_2d(smem_u32(smem + kOffW + s * kChunkBytes), (u & 1) ? &tm_wv : &tm_wk, 64 * kc, h * kNope,
                    smem_u32(&bars.w_full[s]));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ tcgen05 issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 128, /*a_mn=*/0, /*b_mn=*/0);
      const uint64_t d_a = smem_desc(smem_u32(smem + kOffA), 16, 1024, kSw128);
      const uint64_t d_w = smem_desc(smem_u32(smem + kOffW), 16, 1024, kSw128);
      bool ok = mbar_wait(smem_u32(&bars.a_full), 0, p.status, abort);
      for (int u = 0; u < kUnits && ok; ++u) {
        const int buf = u & 3;
        ok = mbar_wait(smem_u32(&bars.d_empty[buf]), ((u >> 2) & 1) ^ 1, p.status, abort);
        tc_fence_after();
        for (int kc = 0; kc < 8 && ok; ++kc) {
          const int i = u * 8 + kc, s = i % kWStages;
          ok = mbar_wait(smem_u32(&bars.w_full[s]), (i / kWStages) & 1, p.status, abort);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + 128 * buf, d_a + ((kc * kChunkBytes) >> 4) + 2 * k,
                   d_w + ((s * kChunkBytes) >> 4) + 2 * k, idesc, (kc > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars.w_empty[s]));
        }
        if (ok) mma_commit(smem_u32(&bars.d_full[buf]));
      }
      // no tcgen05 operation may still be running when TMEM is released
      mma_commit(smem_u32(&bars.a_full));
      mbar_wait(smem_u32(&bars.a_full), 1, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue: token rows
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // token row of the tile (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t t = t0 + r;
    for (int u = 0; u < kUnits; ++u) {
      const int buf = u & 3;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.d_full[buf]), (u >> 2) & 1, p.status, abort))) break;
      tc_fence_after();
      const int h = kHeadsPerCta * hg + (u >> 1);
      uint16_t* dst = ((u & 1) ? p.v_out : p.k_out) +
                      ((static_cast<int64_t>(b) * kHeads + h) * p.max_kv_len + t) * kNope;
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + 128 * buf + c0, v);
        tmem_wait_ld();
        if (t < p.max_kv_len) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const bool live = r < valid;
            d4[q] = make_uint4(live ? pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])) : 0u,
                               live ? pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])) : 0u,
                               live ? pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])) : 0u,
                               live ? pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])) : 0u);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.d_empty[buf]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool g_configured[64];

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
  CUtensorMap tc, twk, twv;
  const uint64_t c_rows = static_cast<uint64_t>(num_pages) * kPage;
  const uint64_t w_rows = static_cast<uint64_t>(kHeads) * kNope;
  if (!make_tmap_bf16_2d(&tc, cache, c_rows, kRow, kRow, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&twk, w_uk, w_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&twv, w_uv, w_rows, kLatent, kLatent, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.k_out = k_out;
  prm.v_out = v_out;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.max_kv_len = max_kv_len;
  dim3 grid((max_kv_len + kTile - 1) / kTile, kHeads / kHeadsPerCta, B);
  return launch_kernel(decompress_kv_tc_kernel, grid, dim3(kThreads), kSmemBytes, stream, tc, twk, twv, prm);
}

}  // namespace mla
