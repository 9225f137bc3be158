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
// (m contiguous).  All of W_UV[h] (128 KB) is requested at once with 16-byte
// asynchronous copies; while it is in flight the CTA builds O' (merging the
// splits in float32 with the same operations, in the same order, as the
// stand-alone merge kernel) and rounds it to bf16 into shared memory.  One
// chain of 32 MMAs (K = 16 each) accumulates in TMEM.
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kNMax = 64;                          // query tokens per CTA
constexpr int kThreads = 256;
constexpr int kChunk = 128 * 128;                  // 128 rows x 64 m (128 B), SW128
constexpr int kSmemA = (kLatent / 64) * kChunk;    // W_UV[h]: 8 chunks, 128 KB
constexpr int kSmemB = (kLatent / 64) * kNMax * 128;  // O' bf16: 8 chunks of up to 64 rows, 64 KB

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
  return kSmemA + (kLatent / 64) * nb * 128 + 16 + 4 * (2 * kNMax + table) + 1024;
}

// src: O' rows; with src_lse == nullptr, row (t, h) is src[(t * 128 + h) * 512]
// (one source); otherwise num_splits partial rows src[((t * S + s) * 128 + h) * 512]
// with log-sum-exps src_lse[(t * S + s) * 128 + h] are merged first, and the
// merged log-sum-exp goes to lse_out[t * 128 + h] (if non-null).
__global__ void __launch_bounds__(kThreads, 1)
out_absorb_tc_kernel(const float* __restrict__ src, const float* __restrict__ src_lse, int num_splits,
                     const uint16_t* __restrict__ w_uv, uint16_t* __restrict__ out, float* __restrict__ lse_out,
                     int T, int* status, bool weights_early) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nb = tile_tokens(T);  // B and TMEM are sized for the widest token tile of this launch
  const uint32_t tmem_cols = tmem_cols_for(nb);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSmemA;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + (kLatent / 64) * nb * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  float* s_max = reinterpret_cast<float*>(bar + 2);  // per token: max_s lse_s
  float* s_inv = s_max + kNMax;                      // per token: 1 / sum_s exp(lse_s - max)
  float* s_w = s_inv + kNMax;                        // [token][split] weights (table mode)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kNMax;
  const int nt = min(kNMax, T - t0);
  const int npad = (nt + 15) & ~15;
  const int64_t S = num_splits;

  // A: W_UV[h][d][0 .. 512) -> 8 K-major chunks of 64 m, rows d (all in flight
  // at once; possibly requested before the previous kernel has finished)
  auto load_w = [&]() {
    const uint4* wsrc = reinterpret_cast<const uint4*>(w_uv + static_cast<int64_t>(h) * kNope * kLatent);
#pragma unroll 4
    for (int v = tid; v < kNope * (kLatent / 8); v += kThreads) {
      const int d = v >> 6, u = v & 63;  // 16-byte unit u of row d: chunk u / 8
      cp_async16(smem_u32(sA + (u >> 3) * kChunk + sw128(d * 128 + (u & 7) * 16)), wsrc + v);
    }
  };
  if (weights_early) load_w();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
  }
  grid_dep_wait();
  grid_dep_launch();
  if (!weights_early) load_w();
  // Merge weights: w[t][s] = exp(lse_s - max_s lse_s) (-1 marks an empty split,
  // which is skipped), kept in shared memory for up to kTableSplits splits.
  const bool table = num_splits <= kTableSplits;
  if (src_lse != nullptr && tid < nt) {
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

  // B: O'[t0 + t][h][0 .. 512) rounded to bf16: 8 K-major chunks of 64, rows t
  // (zero past nt).  Thread (tq, u) = (tid / 64, tid % 64) builds 16-byte unit u
  // (8 consecutive m) of tokens t = tq + 4i, 8 tokens at a time, so that each
  // split's 16 loads are in flight together.
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
          const float4* p = reinterpret_cast<const float4*>(src + (static_cast<int64_t>(t0 + t) * kHeads + h) * kLatent) + 2 * u;
          a[k] = p[0];
          b[k] = p[1];
        }
      }
    } else {
      for (int s = 0; s < num_splits; ++s) {
        float4 x[8], y[8];
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = tq + 4 * (i0 + k);
          w[k] = -1.f;
          x[k] = y[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (t < nt && s_max[t] != -INFINITY) {
            const int64_t r = (static_cast<int64_t>(t0 + t) * S + s) * kHeads + h;
            if (table) {
              w[k] = s_w[t * num_splits + s];
            } else {
              const float l = src_lse[r];
              w[k] = l == -INFINITY ? -1.f : expf(l - s_max[t]);
            }
            const float4* p = reinterpret_cast<const float4*>(src + r * kLatent) + 2 * u;
            x[k] = p[0];
            y[k] = p[1];
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (w[k] >= 0.f) {
            a[k].x = fmaf(w[k], x[k].x, a[k].x); a[k].y = fmaf(w[k], x[k].y, a[k].y);
            a[k].z = fmaf(w[k], x[k].z, a[k].z); a[k].w = fmaf(w[k], x[k].w, a[k].w);
            b[k].x = fmaf(w[k], y[k].x, b[k].x); b[k].y = fmaf(w[k], y[k].y, b[k].y);
            b[k].z = fmaf(w[k], y[k].z, b[k].z); b[k].w = fmaf(w[k], y[k].w, b[k].w);
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
  cp_async_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
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

cudaError_t launch(const float* src, const float* src_lse, int num_splits, const uint16_t* w_uv, uint16_t* out,
                   float* lse_out, int T, int* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(out_absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes_for(kNMax, kTableSplits));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(kHeads, (T + kNMax - 1) / kNMax);
  return launch_kernel(out_absorb_tc_kernel, grid, dim3(kThreads), smem_bytes_for(T, num_splits), stream, src,
                       src_lse, num_splits, w_uv, out, lse_out, T, status, launch_overlap() >= 2);
}

}  // namespace

cudaError_t launch_out_absorb(const float* o_latent, const uint16_t* w_uv, uint16_t* out, int B, int n_q,
                              int* status, cudaStream_t stream) {
  return launch(o_latent, nullptr, 1, w_uv, out, nullptr, B * n_q, status, stream);
}

cudaError_t launch_combine_out_absorb(const float* o_part, const float* lse_part, int num_splits,
                                      const uint16_t* w_uv, uint16_t* out, float* lse, int B, int n_q,
                                      int* status, cudaStream_t stream) {
  return launch(o_part, lse_part, num_splits, w_uv, out, lse, B * n_q, status, stream);
}

}  // namespace mla
