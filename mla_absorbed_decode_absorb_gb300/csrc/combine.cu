// Split-KV merge by log-sum-exp, in float32 (the splits' partials O'_s arrive as bf16).
//
// "DeepSeek-MLA-Principle", FlashMLA point 3: the history is processed in
// blocks with the softmax normalisation updated online; splitting the blocks
// over CTAs needs this final merge.  With split outputs O'_s normalised within
// their split and natural log-sum-exps lse_s:
//   lse = log sum_s exp(lse_s),  O' = sum_s exp(lse_s - lse) O'_s.
// Empty splits carry lse_s = -inf and weigh nothing.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 128;  // 4 latent columns per thread

__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint16_t* __restrict__ o_part, const float* __restrict__ lse_part,
               int num_splits, float* __restrict__ o_latent, float* __restrict__ lse) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t row = blockIdx.x;  // (b*n_q + j)*128 + h
  const int64_t bj = row / kHeads;
  const int h = static_cast<int>(row % kHeads);
  float m = -INFINITY;
  for (int s = 0; s < num_splits; ++s) m = fmaxf(m, lse_part[(bj * num_splits + s) * kHeads + h]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float l = lse_part[(bj * num_splits + s) * kHeads + h];
      if (l == -INFINITY) continue;
      const float w = expf(l - m);
      z += w;
      const uint2 b = reinterpret_cast<const uint2*>(o_part + ((bj * num_splits + s) * kHeads + h) * kLatent)[threadIdx.x];
      const float4 v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                                   __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = 1.f / z;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
  }
  reinterpret_cast<float4*>(o_latent + row * kLatent)[threadIdx.x] = acc;
  if (lse != nullptr && threadIdx.x == 0) lse[row] = m == -INFINITY ? m : m + logf(z);
}

// dst[i] = bf16(src[i]), nearest even (the merged latent output as a bf16 GEMM operand)
__global__ void __launch_bounds__(256)
f32_to_bf16_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, int64_t n) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = f32_to_bf16_bits(src[i]);
}

}  // namespace

cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256;
  return launch_kernel(f32_to_bf16_kernel, dim3(static_cast<unsigned>(want < 8192 ? want : 8192)), dim3(256), 0,
                       stream, src, dst, n);
}

cudaError_t launch_combine(const uint16_t* o_part, const float* lse_part, int B, int n_q,
                           int num_splits, float* o_latent, float* lse, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * n_q * kHeads;
  if (rows == 0) return cudaSuccess;
  return launch_kernel(combine_kernel, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0, stream, o_part, lse_part,
                       num_splits, o_latent, lse);
}

}  // namespace mla
