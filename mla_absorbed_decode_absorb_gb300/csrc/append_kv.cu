// Paged append of the new tokens' cache rows: [c_kv ; RoPE(k_pe, pos)].
//
// "DeepSeek MLA 架构详解" decode listing, step 1: the shared RoPE key is rotated
// at the token's position and appended next to the latent; "DeepSeek-MLA-Principle"
// eq. (3) and FlashMLA point 4 (paged cache, block table); page size 64 from
// "MLA 矩阵吸收 …" section 6.
//
// One warp per token (the row itself is written by append_token_bf16).
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

// FP8 cache variant (one warp per token): the latent as E4M3 codes of c / s with
// one float32 scale per token, s = max(amax / 448, 2^-10), and the rotated key
// as float16 of r / s.  Every value passes through the same float32 steps as
// the recipe the cache image is checked against: amax of the bf16 inputs, one
// IEEE division for s, one per code (then nearest-even E4M3 with saturation),
// the rotation as above, one division per key value, then nearest-even f16.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;  // lo in the low byte (the lower address)
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
append_kv_fp8_kernel(const uint16_t* __restrict__ c_new, const uint16_t* __restrict__ k_new,
                     const int32_t* __restrict__ lens, const int32_t* __restrict__ page_table,
                     int pt_stride, const float* __restrict__ rope, int rope_max_pos,
                     uint8_t* __restrict__ c8, float* __restrict__ scale, uint16_t* __restrict__ kr,
                     int64_t num_pages, int B, int n_new, int* status) {
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
  const int64_t slot = static_cast<int64_t>(page) * kPage + pos % kPage;
  // lane holds latent values [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8)
  const uint4* src = reinterpret_cast<const uint4*>(c_new + token * kLatent);
  const uint4 v0 = src[lane], v1 = src[lane + 32];
  float x[16];
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = fmaxf(__fdiv_rn(amax, 448.f), 0.0009765625f);  // floor 2^-10
  uint16_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = e4m3x2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
  uint8_t* dst = c8 + slot * kLatent;
  *reinterpret_cast<uint2*>(dst + 8 * lane) =
      make_uint2(q[0] | (static_cast<uint32_t>(q[1]) << 16), q[2] | (static_cast<uint32_t>(q[3]) << 16));
  *reinterpret_cast<uint2*>(dst + 256 + 8 * lane) =
      make_uint2(q[4] | (static_cast<uint32_t>(q[5]) << 16), q[6] | (static_cast<uint32_t>(q[7]) << 16));
  if (lane == 0) scale[slot] = s;

  const uint16_t* kp = k_new + token * kRope;
  const float x1 = bf16_bits_to_f32(kp[lane]);
  const float x2 = bf16_bits_to_f32(kp[lane + kHalfRope]);
  const float c = rope[pos * kRope + lane];
  const float sn = rope[pos * kRope + kHalfRope + lane];
  const float r1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn));
  const float r2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn));
  uint16_t* kd = kr + slot * kRope;
  kd[lane] = __half_as_ushort(__float2half_rn(__fdiv_rn(r1, s)));
  kd[kHalfRope + lane] = __half_as_ushort(__float2half_rn(__fdiv_rn(r2, s)));
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
  return launch_kernel(append_kv_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarpsPerBlock * 32), 0,
                       stream, c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table, rope_max_pos,
                       c8, scale, kr, num_pages, B, n_new, status);
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
