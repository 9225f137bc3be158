// Paged append of the new tokens' cache rows: [c_kv ; RoPE(k_pe, pos)].
//
// "DeepSeek MLA 架构详解" decode listing, step 1: the shared RoPE key is rotated
// at the token's position and appended next to the latent; "DeepSeek-MLA-Principle"
// eq. (3) and FlashMLA point 4 (paged cache, block table); page size 64 from
// "MLA 矩阵吸收 …" section 6.
//
// One warp per token.  The 512-wide latent is a straight 1 KB copy (two 16-byte
// vectors per lane); lane i rotates the pair (x_i, x_{i+32}) with the float32
// cos/sin of the caller's table, each product and sum rounded separately so the
// bf16 result is reproducible bit for bit.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
append_kv_kernel(const uint16_t* __restrict__ c_new, const uint16_t* __restrict__ k_new,
                 const int32_t* __restrict__ lens, const int32_t* __restrict__ page_table,
                 int pt_stride, const float* __restrict__ rope, int rope_max_pos,
                 uint16_t* __restrict__ cache, int64_t num_pages, int B, int n_new,
                 int* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
  if (token >= static_cast<int64_t>(B) * n_new) return;
  const int b = static_cast<int>(token / n_new);
  const int j = static_cast<int>(token % n_new);
  const int64_t pos = static_cast<int64_t>(lens[b]) + j;
  if (pos < 0 || pos >= rope_max_pos || pos / kPage >= pt_stride) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  const int page = page_table[static_cast<int64_t>(b) * pt_stride + pos / kPage];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  uint16_t* dst = cache + (static_cast<int64_t>(page) * kPage + pos % kPage) * kRow;
  const uint4* src = reinterpret_cast<const uint4*>(c_new + token * kLatent);
  uint4* dst4 = reinterpret_cast<uint4*>(dst);
  dst4[lane] = src[lane];
  dst4[lane + 32] = src[lane + 32];

  const uint16_t* kp = k_new + token * kRope;
  const float x1 = bf16_bits_to_f32(kp[lane]);
  const float x2 = bf16_bits_to_f32(kp[lane + kHalfRope]);
  const float c = rope[pos * kRope + lane];
  const float s = rope[pos * kRope + kHalfRope + lane];
  const float r1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
  const float r2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
  dst[kLatent + lane] = f32_to_bf16_bits(r1);
  dst[kLatent + kHalfRope + lane] = f32_to_bf16_bits(r2);
}

}  // namespace

cudaError_t launch_append_kv(const uint16_t* c_kv_new, const uint16_t* k_pe_new,
                             const int32_t* seq_lens_before, const int32_t* page_table,
                             int pt_stride, const float* rope_table, int rope_max_pos,
                             uint16_t* cache, int64_t num_pages, int B, int n_new,
                             int* status, cudaStream_t stream) {
  const int64_t tokens = static_cast<int64_t>(B) * n_new;
  if (tokens == 0) return cudaSuccess;
  const int64_t blocks = (tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_kernel(append_kv_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarpsPerBlock * 32), 0, stream,
                       c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
                       cache, num_pages, B, n_new, status);
}

}  // namespace mla
