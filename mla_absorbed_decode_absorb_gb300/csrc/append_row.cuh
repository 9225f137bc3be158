// One new token's cache row, written by one warp: [c_kv ; RoPE(k_pe, pos)].
//
// "DeepSeek MLA 架构详解" decode listing, step 1 (the shared RoPE key is rotated
// at the token's position and appended next to the latent); "DeepSeek-MLA-
// Principle" eq. (3) and FlashMLA point 4 (paged cache, block table).  The
// 512-wide latent is a straight 1 KB copy (two 16-byte vectors per lane); lane
// i rotates the pair (x_i, x_{i+32}) with the float32 cos/sin of the caller's
// table, each product and sum rounded separately so the bf16 result is
// reproducible bit for bit.  Used by the append kernel and by the absorbed-query
// kernel when it also performs the step's append.
#pragma once

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
  uint16_t* cache;         // [num_pages, 64, 576] bf16
  int64_t num_pages;
  int B, n_new;
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

}  // namespace mla
