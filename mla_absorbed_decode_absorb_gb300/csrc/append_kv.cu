// Paged append of the new tokens' cache rows: [c_kv ; RoPE(k_pe, pos)].
//
// "DeepSeek MLA 架构详解" decode listing, step 1: the shared RoPE key is rotated
// at the token's position and appended next to the latent; "DeepSeek-MLA-Principle"
// eq. (3) and FlashMLA point 4 (paged cache, block table); page size 64 from
// "MLA 矩阵吸收 …" section 6.
//
// One warp per token (the row itself is written by append_token_bf16 or
// append_token_fp8).
#include <cuda_fp16.h>

#include "append_row.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
append_kv_kernel(const AppendArgs a, int* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (token >= static_cast<int64_t>(a.B) * a.n_new) return;
  append_token_bf16(a, token, threadIdx.x & 31, status);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
append_kv_fp8_kernel(const AppendArgs a, int* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (token >= static_cast<int64_t>(a.B) * a.n_new) return;
  append_token_fp8(a, token, threadIdx.x & 31, status);
}

}  // namespace

cudaError_t launch_append_kv_fp8(const uint16_t* c_kv_new, const uint16_t* k_pe_new,
                                 const int32_t* seq_lens_before, const int32_t* page_table,
                                 int pt_stride, const float* rope_table, int rope_max_pos,
                                 uint8_t* c8, float* scale, uint16_t* kr, int64_t num_pages, int B, int n_new,
                                 int* status, cudaStream_t stream) {
  const int64_t tokens = static_cast<int64_t>(B) * n_new;
  if (tokens == 0) return cudaSuccess;
  const int64_t blocks = (tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  AppendArgs a{c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
               nullptr, num_pages, B, n_new, c8, scale, kr};
  return launch_kernel(append_kv_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarpsPerBlock * 32), 0,
                       stream, a, status);
}

cudaError_t launch_append_kv(const uint16_t* c_kv_new, const uint16_t* k_pe_new,
                             const int32_t* seq_lens_before, const int32_t* page_table,
                             int pt_stride, const float* rope_table, int rope_max_pos,
                             uint16_t* cache, int64_t num_pages, int B, int n_new,
                             int* status, cudaStream_t stream) {
  const int64_t tokens = static_cast<int64_t>(B) * n_new;
  if (tokens == 0) return cudaSuccess;
  const int64_t blocks = (tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const AppendArgs a{c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
                     cache, num_pages, B, n_new};
  return launch_kernel(append_kv_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarpsPerBlock * 32), 0, stream,
                       a, status);
}

}  // namespace mla
