// Split-KV absorbed attention over the paged latent cache.
//
// Per (sequence b, query j, split s, head h), over the split's visible tokens t:
//   score_t = (q_abs[h,0:512] . c_t + q_abs[h,512:576] . kR_t) / sqrt(192)
//   O'_s[h] = sum_t softmax(score)_t c_t,  lse_s[h] = log sum_t exp(score_t)
// ("MLA 矩阵吸收 …" section 4.1, score = Q'_nope c^T + Q_rope k_rope^T, and the
//  V-side absorption O' = softmax . c; "DeepSeek-MLA-Principle" section 2 scale
//  1/sqrt(d_h + d_h^R) and eq. (10); FlashMLA point 3, online softmax by block.)
//
// CUDA-core version: one warp per head walks the split's tokens with an online
// softmax in the exp2 domain; lanes split the 576-wide row (16 latent + 2 RoPE
// scalars each) and reduce the dot product across the warp.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;  // heads per block

__global__ void __launch_bounds__(kWarps * 32)
decode_attn_simt_kernel(const uint16_t* __restrict__ q_abs, const uint16_t* __restrict__ cache,
                        int64_t num_pages, const int32_t* __restrict__ page_table, int pt_stride,
                        const int32_t* __restrict__ kv_lens, int n_q, int max_kv_len,
                        int split_pages, int num_splits, float* __restrict__ o_out,
                        float* __restrict__ lse_out, int* status) {
  const int split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWarps + warp;
  const int bj = blockIdx.z;
  const int b = bj / n_q, j = bj % n_q;
  const int64_t out_row = (static_cast<int64_t>(bj) * num_splits + split) * kHeads + h;

  const int kv = kv_lens[b];
  int t_begin = split * split_pages * kPage;
  int t_end = min(t_begin + split_pages * kPage, kv - n_q + j + 1);
  if (kv > max_kv_len || kv < n_q || (kv + kPage - 1) / kPage > pt_stride) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    t_end = t_begin;  // write an empty split
  }

  const uint16_t* qrow = q_abs + (static_cast<int64_t>(bj) * kHeads + h) * kRow;
  float qc[16], qr[2];
  {
    const uint4* q4 = reinterpret_cast<const uint4*>(qrow + lane * 16);
    const uint4 a = q4[0], c = q4[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      qc[2 * k] = __uint_as_float(w[k] << 16);
      qc[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
    const uint32_t r = reinterpret_cast<const uint32_t*>(qrow + kLatent)[lane];
    qr[0] = __uint_as_float(r << 16);
    qr[1] = __uint_as_float(r & 0xffff0000u);
  }

  float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;

  for (int t = t_begin; t < t_end; ++t) {
    const int page = page_table[static_cast<int64_t>(b) * pt_stride + t / kPage];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
      break;
    }
    const uint16_t* row = cache + (static_cast<int64_t>(page) * kPage + t % kPage) * kRow;
    const uint4* r4 = reinterpret_cast<const uint4*>(row + lane * 16);
    const uint4 a = r4[0], c = r4[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    float cv[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cv[2 * k] = __uint_as_float(w[k] << 16);
      cv[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
    const uint32_t rr = reinterpret_cast<const uint32_t*>(row + kLatent)[lane];
    float p = qr[0] * __uint_as_float(rr << 16) + qr[1] * __uint_as_float(rr & 0xffff0000u);
#pragma unroll
    for (int k = 0; k < 16; ++k) p = fmaf(qc[k], cv[k], p);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
    const float s = p * kScaleLog2;
    const float m_new = fmaxf(m, s);
    const float corr = exp2f(m - m_new);
    const float e = exp2f(s - m_new);
    l = l * corr + e;
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = fmaf(e, cv[k], acc[k] * corr);
    m = m_new;
  }

  float* orow = o_out + out_row * kLatent + lane * 16;
  if (l > 0.f) {
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < 16; k += 4)
      *reinterpret_cast<float4*>(orow + k) = make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
    if (lse_out != nullptr && lane == 0) lse_out[out_row] = (m + log2f(l)) * kLn2;
  } else {
#pragma unroll
    for (int k = 0; k < 16; k += 4) *reinterpret_cast<float4*>(orow + k) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_out != nullptr && lane == 0) lse_out[out_row] = -INFINITY;
  }
}

}  // namespace

cudaError_t launch_decode_partial(const uint16_t* q_abs, const uint16_t* cache,
                                  int64_t num_pages, const int32_t* page_table, int pt_stride,
                                  const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                  const SplitPlan& plan, float* o_out, float* lse_out,
                                  int* status, cudaStream_t stream) {
  if (B * n_q == 0) return cudaSuccess;
  dim3 grid(plan.num_splits, kHeads / kWarps, B * n_q);
  decode_attn_simt_kernel<<<grid, kWarps * 32, 0, stream>>>(
      q_abs, cache, num_pages, page_table, pt_stride, kv_lens, n_q, max_kv_len,
      plan.split_pages, plan.num_splits, o_out, lse_out, status);
  return cudaGetLastError();
}

}  // namespace mla
