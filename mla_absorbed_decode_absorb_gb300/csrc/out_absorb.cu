// Value up-projection applied once to the latent output: O[t,h,d] = sum_m O'[t,h,m] W_UV[h,d,m].
//
// "MLA 矩阵吸收 …" section 2.1, V side (O = (Attn c) W_UV, done once, independent
// of the history length); "DeepSeek-MLA-Principle" value absorption
// o = W_UV[h] m; "DeepSeek MLA 架构详解" step 5 (einsum 'bhm,hdm->bhd').
//
// tcgen05 version, operands swapped so the large side is M: per head h the CTA
// computes D[d, t] = sum_m W_UV[h][d][m] * O'[t][h][m] with the 128 output
// dimensions d as M and up to 256 query tokens as N.  Both operands are
// K-major (m contiguous).  The 512-long K axis is staged in four 128-wide
// steps; O' is rounded from float32 to bf16 as it is staged.
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kNMax = 256;
constexpr int kThreads = 128;
constexpr int kKStep = 128;                       // latent columns per stage
constexpr int kAChunk = 128 * 128;                // 128 d rows x 64 m (128 B)
constexpr int kSmemA = 2 * kAChunk;               // 32 KB
constexpr int kSmemB = 2 * kNMax * 128;           // 64 KB
constexpr int kSmemBytes = kSmemA + kSmemB + 1024 + 64;

// Tokens of the widest tile (rounded up to the MMA's N granularity of 16), and
// the TMEM columns for its fp32 accumulator (a power of two, at least 32).
__host__ __device__ inline int tile_tokens(int T) { return (min(kNMax, T) + 15) & ~15; }
__host__ __device__ inline uint32_t tmem_cols_for(int nb) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(nb)) c <<= 1;
  return c;
}
__host__ __device__ inline int smem_bytes_for(int T) { return kSmemA + 2 * tile_tokens(T) * 128 + 1024 + 64; }

__global__ void __launch_bounds__(kThreads)
out_absorb_tc_kernel(const float* __restrict__ o_lat, const uint16_t* __restrict__ w_uv,
                     uint16_t* __restrict__ out, int T, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSmemA;
  // B and TMEM are sized for the widest token tile of this launch (<= 256)
  const int nb = tile_tokens(T);
  const uint32_t tmem_cols = tmem_cols_for(nb);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + 2 * nb * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kNMax;
  const int nt = min(kNMax, T - t0);
  const int npad = (nt + 15) & ~15;

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc = idesc_bf16(128, npad, /*a_mn=*/0, /*b_mn=*/0);
  const uint16_t* wh = w_uv + static_cast<int64_t>(h) * kNope * kLatent;
  bool ok = true;

  for (int step = 0; step < kLatent / kKStep && ok; ++step) {
    const int mk = step * kKStep;
    // A: W_UV[h][d][mk .. mk+128): rows d, two K-major chunks of 64 (asynchronous
    // 16-byte copies, completed below before the MMAs read them).
#pragma unroll 4
    for (int v = tid; v < kNope * 16; v += kThreads) {
      const int d = v >> 4, u = v & 15, c = u >> 3;
      cp_async16(smem_u32(sA + c * kAChunk + sw128(d * 128 + (u & 7) * 16)),
                 reinterpret_cast<const uint4*>(wh + d * kLatent + mk) + u);
    }
    // B: O'[t0+t][h][mk .. mk+128) rounded to bf16: rows t, two K-major chunks of 64.
    for (int v0 = 0; v0 < npad * 16; v0 += 4 * kThreads) {
      float4 a[4], b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = v0 + tid + k * kThreads, t = v >> 4, u = v & 15;
        a[k] = b[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < npad * 16 && t < nt) {
          const float4* src = reinterpret_cast<const float4*>(
              o_lat + (static_cast<int64_t>(t0 + t) * kHeads + h) * kLatent + mk + u * 8);
          a[k] = src[0];
          b[k] = src[1];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = v0 + tid + k * kThreads, t = v >> 4, u = v & 15, c = u >> 3;
        if (v < npad * 16)
          *reinterpret_cast<uint4*>(sB + c * npad * 128 + sw128(t * 128 + (u & 7) * 16)) =
              make_uint4(pack_bf16x2(a[k].x, a[k].y), pack_bf16x2(a[k].z, a[k].w), pack_bf16x2(b[k].x, b[k].y),
                         pack_bf16x2(b[k].z, b[k].w));
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
      for (int k = 0; k < kKStep / 16; ++k) {
        const uint64_t ad = smem_desc(a0 + (k >> 2) * kAChunk + (k & 3) * 32, 16, 1024, kSw128);
        const uint64_t bd = smem_desc(b0 + (k >> 2) * npad * 128 + (k & 3) * 32, 16, 1024, kSw128);
        mma_ss(tmem, ad, bd, idesc, (step > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(bar));
    }
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), step & 1, status));  // stage reusable once the MMAs finished
    tc_fence_after();
  }

  if (ok) {
    const int d = warp * 32 + lane;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c0 = 0; c0 < npad; c0 += 16) {
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

}  // namespace

cudaError_t launch_out_absorb(const float* o_latent, const uint16_t* w_uv, uint16_t* out, int B, int n_q,
                              int* status, cudaStream_t stream) {
  const int T = B * n_q;
  if (T == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(out_absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(kHeads, (T + kNMax - 1) / kNMax);
  out_absorb_tc_kernel<<<grid, kThreads, smem_bytes_for(T), stream>>>(o_latent, w_uv, out, T, status);
  return cudaGetLastError();
}

}  // namespace mla
