// One new token's cache row, written by one warp: [c_kv ; RoPE(k_pe, pos)].
//
// "DeepSeek MLA 架构详解" decode listing, step 1 (the shared RoPE key is rotated
// at the token's position and appended next to the latent); "DeepSeek-MLA-
// Principle" eq. (3) and FlashMLA point 4 (paged cache, block table).  The
// 512-wide latent is a straight 1 KB copy (two 16-byte vectors per lane); lane
// i rotates the pair (x_i, x_{i+32}) with the float32 cos/sin of the caller's
// table, each product and sum rounded separately so the bf16 result is
// reproducible bit for bit.  Used by the append kernels and by the absorbed-query
// kernel when it also performs the step's append.
#pragma once

#include <cuda_fp16.h>

#include "internal.cuh"

namespace mla {

struct AppendArgs {
  const uint16_t* c_new;   // [B * n_new, 512] bf16
  const uint16_t* k_new;   // [B * n_new, 64] bf16
  const int32_t* lens;     // [B] tokens already cached per sequence
  const int32_t* page_table;
  int pt_stride;
  const float* rope;       // [rope_max_pos, 64] float32 (cos | sin)
  int rope_max_pos;
  uint16_t* cache;         // [num_pages, 64, 576] bf16 (nullptr: the FP8 cache below)
  int64_t num_pages;
  int B, n_new;
  uint8_t* c8;             // FP8 cache: [num_pages, 64, 512] E4M3 codes,
  float* scale;            //   [num_pages, 64] float32 per-token scales,
  uint16_t* kr;            //   [num_pages, 64, 64] f16 rotated keys / scale
};

// Token `token` (= b * n_new + j) of the step; every lane of the warp calls it.
// A position or page outside the table records MLA_ERR_BOUNDS and writes nothing.
__device__ __forceinline__ void append_token_bf16(const AppendArgs& a, int64_t token, int lane, int* status) {
  const int b = static_cast<int>(token / a.n_new);
  const int j = static_cast<int>(token % a.n_new);
  const int64_t pos = static_cast<int64_t>(a.lens[b]) + j;
  if (pos < 0 || pos >= a.rope_max_pos || pos / kPage >= a.pt_stride) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  const int page = a.page_table[static_cast<int64_t>(b) * a.pt_stride + pos / kPage];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  uint16_t* dst = a.cache + (static_cast<int64_t>(page) * kPage + pos % kPage) * kRow;
  const uint4* src = reinterpret_cast<const uint4*>(a.c_new + token * kLatent);
  uint4* dst4 = reinterpret_cast<uint4*>(dst);
  dst4[lane] = src[lane];
  dst4[lane + 32] = src[lane + 32];

  const uint16_t* kp = a.k_new + token * kRope;
  const float x1 = bf16_bits_to_f32(kp[lane]);
  const float x2 = bf16_bits_to_f32(kp[lane + kHalfRope]);
  const float c = a.rope[pos * kRope + lane];
  const float s = a.rope[pos * kRope + kHalfRope + lane];
  const float r1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
  const float r2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
  dst[kLatent + lane] = f32_to_bf16_bits(r1);
  dst[kLatent + kHalfRope + lane] = f32_to_bf16_bits(r2);
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

__device__ __forceinline__ void append_token_fp8(const AppendArgs& a, int64_t token, int lane, int* status) {
  const int b = static_cast<int>(token / a.n_new);
  const int j = static_cast<int>(token % a.n_new);
  const int64_t pos = static_cast<int64_t>(a.lens[b]) + j;
  if (pos < 0 || pos >= a.rope_max_pos || pos / kPage >= a.pt_stride) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  const int page = a.page_table[static_cast<int64_t>(b) * a.pt_stride + pos / kPage];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) record_status(status, MLA_ERR_BOUNDS);
    return;
  }
  const int64_t slot = static_cast<int64_t>(page) * kPage + pos % kPage;
  // lane holds latent values [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8)
  const uint4* src = reinterpret_cast<const uint4*>(a.c_new + token * kLatent);
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
  uint8_t* dst = a.c8 + slot * kLatent;
  *reinterpret_cast<uint2*>(dst + 8 * lane) =
      make_uint2(q[0] | (static_cast<uint32_t>(q[1]) << 16), q[2] | (static_cast<uint32_t>(q[3]) << 16));
  *reinterpret_cast<uint2*>(dst + 256 + 8 * lane) =
      make_uint2(q[4] | (static_cast<uint32_t>(q[5]) << 16), q[6] | (static_cast<uint32_t>(q[7]) << 16));
  if (lane == 0) a.scale[slot] = s;

  const uint16_t* kp = a.k_new + token * kRope;
  const float x1 = bf16_bits_to_f32(kp[lane]);
  const float x2 = bf16_bits_to_f32(kp[lane + kHalfRope]);
  const float c = a.rope[pos * kRope + lane];
  const float sn = a.rope[pos * kRope + kHalfRope + lane];
  const float r1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn));
  const float r2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn));
  uint16_t* kd = a.kr + slot * kRope;
  kd[lane] = __half_as_ushort(__float2half_rn(__fdiv_rn(r1, s)));
  kd[kHalfRope + lane] = __half_as_ushort(__float2half_rn(__fdiv_rn(r2, s)));
}

}  // namespace mla
