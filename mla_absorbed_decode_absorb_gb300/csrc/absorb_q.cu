// Absorbed query: q_abs[t,h,0:512] = sum_d q_nope[t,h,d] W_UK[h,d,:] and
// q_abs[t,h,512:576] = RoPE(q_rope[t,h,:], pos_t).
//
// "MLA 矩阵吸收 …" section 2.1 (Q' = Q W_UK^T, W_UK absorbed into the query);
// "DeepSeek-MLA-Principle" key absorption q~ = (W_UK[h])^T q^C and eq. (8);
// "DeepSeek MLA 架构详解" step 3 (einsum 'bhd,hdm->bhm').
//
// tcgen05 version, operands swapped so the large side is M: per head h the CTA
// computes D[m, t] = sum_d W_UK[h][d][m] * q_nope[t][h][d] for 128 latent
// columns m (M = 128) and up to 64 query tokens t (N; more tokens take more CTAs,
// which also spreads the RoPE half and the append over more threads).  A = W_UK[h] is
// MN-major (m contiguous), B = q_nope rows are K-major (d contiguous); both are
// staged into shared memory in the 128-byte-swizzled canonical layouts (A by
// two TMA boxes of 64 m x 128 d, B by 16-byte asynchronous copies), one MMA
// chain of 8 x (K = 16) accumulates into TMEM, and four warps read their 32
// TMEM lanes back (lane = m, column = token) and store bf16.
//
// The same launch may also write the step's new cache rows (the append): the
// query side does not read them, so one launch replaces two and the attention
// waits for one grid instead of two.  Warp 0 of CTA k appends tokens k, k + grid, ...
#include "append_row.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kMTile = 128;   // latent columns per CTA
constexpr int kNMax = 64;     // query tokens per CTA
constexpr int kThreads = 128;
constexpr int kAChunk = 128 * 128;          // bytes of one 64-column MN chunk: 128 d rows x 128 B
constexpr int kSmemA = 2 * kAChunk;         // 32 KB
constexpr int kSmemB = 2 * kNMax * 128;     // two 64-wide K chunks of up to 64 rows: 16 KB
constexpr int kSmemBytes = kSmemA + kSmemB + 1024 /*align*/ + 64;

// Tokens of the widest tile (rounded up to the MMA's N granularity of 16), and
// the TMEM columns for its fp32 accumulator (a power of two, at least 32).
__host__ __device__ inline int tile_tokens(int T) { return (min(kNMax, T) + 15) & ~15; }
__host__ __device__ inline uint32_t tmem_cols_for(int nb) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(nb)) c <<= 1;
  return c;
}
__host__ __device__ inline int smem_bytes_for(int T) { return kSmemA + 2 * tile_tokens(T) * 128 + 1024 + 64; }
constexpr uint32_t kWaitBarOffset = 16;  // weight barrier after the MMA barrier and the TMEM slot

__global__ void __launch_bounds__(kThreads)
absorb_q_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_rope,
                   const int32_t* __restrict__ lens,
                   const float* __restrict__ rope, int rope_max_pos, uint16_t* __restrict__ q_abs,
                   int T, int n_q, int* status, bool weights_early, const AppendArgs ap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSmemA;
  // B and TMEM are sized for the widest token tile of this launch (<= 64)
  const int nb = tile_tokens(T);
  const uint32_t tmem_cols = tmem_cols_for(nb);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + 2 * nb * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  uint64_t* wbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(bar) + kWaitBarOffset);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * kMTile;
  const int h = blockIdx.y;
  const int t0 = blockIdx.z * kNMax;
  const int nt = min(kNMax, T - t0);
  const int npad = (nt + 15) & ~15;

  // A: W_UK[h][d][m0 .. m0+128) -> two MN-major chunks of 64 columns, rows d,
  // by TMA (the weights may be requested before the previous kernel of the
  // stream has finished); B: q_nope[t0 + t][h][0 .. 128) -> two K-major chunks
  // of 64, rows t (zero past nt), by 16-byte asynchronous copies.
  auto load_w = [&]() {
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(wbar), kSmemA);
      for (int c = 0; c < 2; ++c) tma_load_2d(smem_u32(sA + c * kAChunk), &tm_w, m0 + 64 * c, h * kNope, smem_u32(wbar));
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
  if ((ap.cache != nullptr || ap.c8 != nullptr) && warp == 0) {
    const int64_t ncta = static_cast<int64_t>(gridDim.x) * gridDim.y * gridDim.z;
    const int64_t tokens = static_cast<int64_t>(ap.B) * ap.n_new;
    for (int64_t tok = (static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x; tok < tokens;
         tok += ncta) {
      if (ap.cache != nullptr)
        append_token_bf16(ap, tok, lane, status);
      else
        append_token_fp8(ap, tok, lane, status);
    }
  }
  for (int v = tid; v < npad * 16; v += kThreads) {
    const int t = v >> 4, u = v & 15, c = u >> 3;
    uint8_t* dst = sB + c * npad * 128 + sw128(t * 128 + (u & 7) * 16);
    if (t < nt)
      cp_async16(smem_u32(dst), reinterpret_cast<const uint4*>(q_nope + (static_cast<int64_t>(t0 + t) * kHeads + h) * kNope) + u);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  // RoPE of the query's position branch while the copies are in flight; the
  // head's M tiles share the (token, frequency) pairs.  Four items per thread at a
  // time with all their loads in flight together: the lengths, then the query
  // pairs and the cos / sin pairs (two round trips per four items, not per item).
  constexpr int kRopeBatch = 4;
  const int rope_stride = gridDim.x * kThreads;
  for (int i0 = blockIdx.x * kThreads + tid; i0 < nt * kHalfRope; i0 += kRopeBatch * rope_stride) {
    int64_t pos[kRopeBatch];
    bool on[kRopeBatch];
#pragma unroll
    for (int k = 0; k < kRopeBatch; ++k) {
      const int i = i0 + k * rope_stride;
      on[k] = i < nt * kHalfRope;
      const int t = t0 + (on[k] ? i : 0) / kHalfRope;
      pos[k] = on[k] ? static_cast<int64_t>(lens[t / n_q]) + t % n_q : 0;
    }
    float x1[kRopeBatch], x2[kRopeBatch], c[kRopeBatch], sn[kRopeBatch];
#pragma unroll
    for (int k = 0; k < kRopeBatch; ++k) {
      const int i = i0 + k * rope_stride, t = t0 + i / kHalfRope, f = i % kHalfRope;
      const bool in = on[k] && pos[k] >= 0 && pos[k] < rope_max_pos;
      const uint16_t* x = q_rope + (static_cast<int64_t>(t) * kHeads + h) * kRope;
      x1[k] = in ? bf16_bits_to_f32(x[f]) : 0.f;
      x2[k] = in ? bf16_bits_to_f32(x[f + kHalfRope]) : 0.f;
      c[k] = in ? rope[pos[k] * kRope + f] : 0.f;
      sn[k] = in ? rope[pos[k] * kRope + kHalfRope + f] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kRopeBatch; ++k) {
      if (!on[k]) continue;
      const int i = i0 + k * rope_stride, t = t0 + i / kHalfRope, f = i % kHalfRope;
      uint16_t* row = q_abs + (static_cast<int64_t>(t) * kHeads + h) * kRow + kLatent;
      if (pos[k] < 0 || pos[k] >= rope_max_pos) {
        record_status(status, MLA_ERR_BOUNDS);
        row[f] = row[f + kHalfRope] = 0;
        continue;
      }
      row[f] = f32_to_bf16_bits(__fsub_rn(__fmul_rn(x1[k], c[k]), __fmul_rn(x2[k], sn[k])));
      row[f + kHalfRope] = f32_to_bf16_bits(__fadd_rn(__fmul_rn(x2[k], c[k]), __fmul_rn(x1[k], sn[k])));
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool wok = true;
  if (tid == 0) wok = mbar_wait(smem_u32(wbar), 0, status);  // the weight tile has landed
  if (tid == 0 && wok) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16(128, npad, /*a_mn=*/1, /*b_mn=*/0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
    for (int k = 0; k < kNope / 16; ++k) {
      const uint64_t ad = smem_desc(a0 + k * 16 * 128, kAChunk, 1024, kSw128);
      const uint64_t bd = smem_desc(b0 + (k >> 2) * npad * 128 + (k & 3) * 32, 16, 1024, kSw128);
      mma_ss(tmem, ad, bd, idesc, k > 0);
    }
    mma_commit(smem_u32(bar));
  }
  if (tid == 0 && !wok) mbar_arrive(smem_u32(bar));  // no MMA: release the waiters (the result is flagged)
  const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), 0, status));
  tc_fence_after();

  if (ok) {
    const int m = m0 + warp * 32 + lane;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c0 = 0; c0 < npad; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = c0 + i;
        if (t < nt) q_abs[(static_cast<int64_t>(t0 + t) * kHeads + h) * kRow + m] = f32_to_bf16_bits(__uint_as_float(r[i]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// The RoPE half of q_abs alone (q_abs[t, h, 512:576] = RoPE(q_rope[t, h], pos_t)),
// for callers that produce the latent half by other means (the query-side
// weight fold); the same float32 recipe as above, one thread per (t, h, f).
__global__ void __launch_bounds__(256)
rope_q_kernel(const uint16_t* __restrict__ q_rope, const int32_t* __restrict__ lens, const float* __restrict__ rope,
              int rope_max_pos, uint16_t* __restrict__ q_abs, int T, int n_q, int* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * kHeads * kHalfRope) return;
  const int f = static_cast<int>(i % kHalfRope);
  const int64_t th = i / kHalfRope;  // t * 128 + h
  const int t = static_cast<int>(th / kHeads);
  const int b = t / n_q, j = t % n_q;
  const int64_t pos = static_cast<int64_t>(lens[b]) + j;
  uint16_t* row = q_abs + th * kRow + kLatent;
  if (pos < 0 || pos >= rope_max_pos) {
    record_status(status, MLA_ERR_BOUNDS);
    row[f] = row[f + kHalfRope] = 0;
    return;
  }
  const uint16_t* x = q_rope + th * kRope;
  const float x1 = bf16_bits_to_f32(x[f]), x2 = bf16_bits_to_f32(x[f + kHalfRope]);
  const float c = rope[pos * kRope + f], sn = rope[pos * kRope + kHalfRope + f];
  row[f] = f32_to_bf16_bits(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn)));
  row[f + kHalfRope] = f32_to_bf16_bits(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn)));
}

}  // namespace

cudaError_t launch_rope_q(const uint16_t* q_rope, const int32_t* seq_lens_before, const float* rope_table,
                          int rope_max_pos, uint16_t* q_abs, int B, int n_q, int* status, cudaStream_t stream) {
  const int T = B * n_q;
  if (T == 0) return cudaSuccess;
  const int64_t n = static_cast<int64_t>(T) * kHeads * kHalfRope;
  return launch_kernel(rope_q_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, q_rope,
                       seq_lens_before, rope_table, rope_max_pos, q_abs, T, n_q, status);
}

namespace {

cudaError_t launch_absorb(const uint16_t* q_nope, const uint16_t* q_rope, const int32_t* seq_lens_before,
                          const uint16_t* w_uk, const float* rope_table, int rope_max_pos, uint16_t* q_abs, int B,
                          int n_q, const AppendArgs& ap, int* status, cudaStream_t stream) {
  const int T = B * n_q;
  static bool configured[kMaxDevicesLocal] = {};  // the attribute is per device
  const int dev_ = current_device_index();
  if (dev_ < 0) return cudaErrorInvalidDevice;
  if (!configured[dev_]) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev_] = true;
  }
  // W_UK as a [128 * 128, 512] matrix: box 64 columns x 128 rows, 128-byte swizzle
  CUtensorMap tw;
  if (!make_tmap_bf16_2d(&tw, w_uk, static_cast<uint64_t>(kHeads) * kNope, kLatent, kLatent, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  dim3 grid(kLatent / kMTile, kHeads, (T + kNMax - 1) / kNMax);
  return launch_kernel(absorb_q_tc_kernel, grid, dim3(kThreads), smem_bytes_for(T), stream, tw, q_nope, q_rope,
                       seq_lens_before, rope_table, rope_max_pos, q_abs, T, n_q, status, launch_overlap() >= 2, ap);
}

}  // namespace

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope,
                            const int32_t* seq_lens_before, const uint16_t* w_uk,
                            const float* rope_table, int rope_max_pos, uint16_t* q_abs,
                            int B, int n_q, int* status, cudaStream_t stream) {
  if (B * n_q == 0) return cudaSuccess;
  AppendArgs none{};
  return launch_absorb(q_nope, q_rope, seq_lens_before, w_uk, rope_table, rope_max_pos, q_abs, B, n_q, none, status,
                       stream);
}

cudaError_t launch_append_absorb_q(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const uint16_t* q_nope,
                                   const uint16_t* q_rope, const int32_t* seq_lens_before, const int32_t* page_table,
                                   int pt_stride, const uint16_t* w_uk, const float* rope_table, int rope_max_pos,
                                   uint16_t* cache, int64_t num_pages, uint16_t* q_abs, int B, int n_q, int* status,
                                   cudaStream_t stream) {
  if (B * n_q == 0) return cudaSuccess;
  const AppendArgs ap{c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
                      cache, num_pages, B, n_q};
  return launch_absorb(q_nope, q_rope, seq_lens_before, w_uk, rope_table, rope_max_pos, q_abs, B, n_q, ap, status,
                       stream);
}

cudaError_t launch_append_absorb_q_fp8(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const uint16_t* q_nope,
                                       const uint16_t* q_rope, const int32_t* seq_lens_before,
                                       const int32_t* page_table, int pt_stride, const uint16_t* w_uk,
                                       const float* rope_table, int rope_max_pos, uint8_t* c8, float* scale,
                                       uint16_t* kr, int64_t num_pages, uint16_t* q_abs, int B, int n_q, int* status,
                                       cudaStream_t stream) {
  if (B * n_q == 0) return cudaSuccess;
  const AppendArgs ap{c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
                      nullptr, num_pages, B, n_q, c8, scale, kr};
  return launch_absorb(q_nope, q_rope, seq_lens_before, w_uk, rope_table, rope_max_pos, q_abs, B, n_q, ap, status,
                       stream);
}

}  // namespace mla
