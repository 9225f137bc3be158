// Value up-projection applied once to the latent output: O[t,h,d] = sum_m O'[t,h,m] W_UV[h,d,m].
//
// "MLA 矩阵吸收 …" section 2.1, V side (O = (Attn c) W_UV, done once, independent
// of the history length); "DeepSeek-MLA-Principle" value absorption
// o = W_UV[h] m; "DeepSeek MLA 架构详解" step 5 (einsum 'bhm,hdm->bhd').
//
// CUDA-core version: one block per (head, chunk of 16 query tokens).  O' is
// rounded to bf16 on the way into shared memory (the documented operand
// precision); each warp walks W_UV[h] rows with lanes along the latent axis and
// reduces across the warp.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kTokTile = 16;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
out_absorb_simt_kernel(const float* __restrict__ o_lat, const uint16_t* __restrict__ w_uv,
                       uint16_t* __restrict__ out, int T) {
  __shared__ float os[kTokTile][kLatent];
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kTokTile;
  const int nt = min(kTokTile, T - t0);
  for (int i = threadIdx.x; i < kTokTile * kLatent; i += kThreads) {
    const int t = i / kLatent, m = i % kLatent;
    float v = 0.f;
    if (t < nt) v = bf16_bits_to_f32(f32_to_bf16_bits(o_lat[(static_cast<int64_t>(t0 + t) * kHeads + h) * kLatent + m]));
    os[t][m] = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* wh = w_uv + static_cast<int64_t>(h) * kNope * kLatent;
  for (int d = warp; d < kNope; d += kThreads / 32) {
    float w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = bf16_bits_to_f32(wh[d * kLatent + k * 32 + lane]);
    for (int t = 0; t < nt; ++t) {
      float p = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) p = fmaf(w[k], os[t][k * 32 + lane], p);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      if (lane == 0) out[(static_cast<int64_t>(t0 + t) * kHeads + h) * kNope + d] = f32_to_bf16_bits(p);
    }
  }
}

}  // namespace

cudaError_t launch_out_absorb(const float* o_latent, const uint16_t* w_uv, uint16_t* out,
                              int B, int n_q, cudaStream_t stream) {
  const int T = B * n_q;
  if (T == 0) return cudaSuccess;
  dim3 grid(kHeads, (T + kTokTile - 1) / kTokTile);
  out_absorb_simt_kernel<<<grid, kThreads, 0, stream>>>(o_latent, w_uv, out, T);
  return cudaGetLastError();
}

}  // namespace mla
