// Absorbed query: q_abs[t,h,0:512] = sum_d q_nope[t,h,d] W_UK[h,d,:] and
// q_abs[t,h,512:576] = RoPE(q_rope[t,h,:], pos_t).
//
// "MLA 矩阵吸收 …" section 2.1 (Q' = Q W_UK^T, W_UK absorbed into the query);
// "DeepSeek-MLA-Principle" key absorption q~ = (W_UK[h])^T q^C and eq. (8);
// "DeepSeek MLA 架构详解" step 3 (einsum 'bhd,hdm->bhm').
//
// CUDA-core version: one block per (head, chunk of 32 query tokens); the
// block's query rows sit in shared memory as float32, each thread owns two of
// the 512 latent columns for all 32 tokens and streams its W_UK[h] column.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kTokTile = 32;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
absorb_q_simt_kernel(const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_rope,
                     const int32_t* __restrict__ lens, const uint16_t* __restrict__ w_uk,
                     const float* __restrict__ rope, int rope_max_pos,
                     uint16_t* __restrict__ q_abs, int T, int n_q, int* status) {
  __shared__ float qs[kTokTile][kNope];
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kTokTile;
  const int nt = min(kTokTile, T - t0);
  for (int i = threadIdx.x; i < kTokTile * kNope; i += kThreads) {
    const int t = i / kNope, d = i % kNope;
    qs[t][d] = t < nt ? bf16_bits_to_f32(q_nope[(static_cast<int64_t>(t0 + t) * kHeads + h) * kNope + d]) : 0.f;
  }
  __syncthreads();

  const int m0 = threadIdx.x, m1 = threadIdx.x + kThreads;
  float acc0[kTokTile], acc1[kTokTile];
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) acc0[t] = acc1[t] = 0.f;
  const uint16_t* w = w_uk + static_cast<int64_t>(h) * kNope * kLatent;
  for (int d = 0; d < kNope; ++d) {
    const float w0 = bf16_bits_to_f32(w[d * kLatent + m0]);
    const float w1 = bf16_bits_to_f32(w[d * kLatent + m1]);
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) {
      acc0[t] = fmaf(qs[t][d], w0, acc0[t]);
      acc1[t] = fmaf(qs[t][d], w1, acc1[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) {
    if (t < nt) {
      uint16_t* row = q_abs + (static_cast<int64_t>(t0 + t) * kHeads + h) * kRow;
      row[m0] = f32_to_bf16_bits(acc0[t]);
      row[m1] = f32_to_bf16_bits(acc1[t]);
    }
  }

  // RoPE of the query's position branch, one (token, frequency) pair per thread.
  for (int i = threadIdx.x; i < nt * kHalfRope; i += kThreads) {
    const int t = t0 + i / kHalfRope, f = i % kHalfRope;
    const int b = t / n_q, j = t % n_q;
    const int64_t pos = static_cast<int64_t>(lens[b]) + j;
    uint16_t* row = q_abs + (static_cast<int64_t>(t) * kHeads + h) * kRow + kLatent;
    if (pos < 0 || pos >= rope_max_pos) {
      record_status(status, MLA_ERR_BOUNDS);
      row[f] = row[f + kHalfRope] = 0;
      continue;
    }
    const uint16_t* x = q_rope + (static_cast<int64_t>(t) * kHeads + h) * kRope;
    const float x1 = bf16_bits_to_f32(x[f]), x2 = bf16_bits_to_f32(x[f + kHalfRope]);
    const float c = rope[pos * kRope + f], s = rope[pos * kRope + kHalfRope + f];
    row[f] = f32_to_bf16_bits(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s)));
    row[f + kHalfRope] = f32_to_bf16_bits(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s)));
  }
}

}  // namespace

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope,
                            const int32_t* seq_lens_before, const uint16_t* w_uk,
                            const float* rope_table, int rope_max_pos, uint16_t* q_abs,
                            int B, int n_q, int* status, cudaStream_t stream) {
  const int T = B * n_q;
  if (T == 0) return cudaSuccess;
  dim3 grid(kHeads, (T + kTokTile - 1) / kTokTile);
  absorb_q_simt_kernel<<<grid, kThreads, 0, stream>>>(q_nope, q_rope, seq_lens_before, w_uk,
                                                      rope_table, rope_max_pos, q_abs, T, n_q, status);
  return cudaGetLastError();
}

}  // namespace mla
