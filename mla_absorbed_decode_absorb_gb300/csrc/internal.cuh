// Internal declarations shared by the CUDA translation units of libmla_decode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla {

constexpr int kHeads = MLA_N_HEADS;    // n_h
constexpr int kNope = MLA_D_NOPE;      // d_h
constexpr int kLatent = MLA_D_LATENT;  // d_c
constexpr int kRope = MLA_D_ROPE;      // d_h^R
constexpr int kRow = MLA_D_ROW;        // d_c + d_h^R
constexpr int kPage = MLA_PAGE;
constexpr int kHalfRope = kRope / 2;
// 1/sqrt(d_h + d_h^R) and that times log2(e): scores are exponentiated with exp2.
constexpr float kScale = 0.07216878364870323f;         // 1/sqrt(192)
constexpr float kScaleLog2 = 0.10411754627697264f;     // log2(e)/sqrt(192)
constexpr float kLn2 = 0.6931471805599453f;

// First fault code wins; later ones are dropped.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel of its
// stream is still running; grid_dep_wait() returns once that kernel has finished
// and its memory operations are visible (immediately when launched without the
// attribute).  Every kernel of this library touches global memory written or
// read by earlier stream work only after it.  grid_dep_launch() lets the next
// kernel's CTAs be scheduled once every CTA of this grid has executed it.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Split-KV layout shared by the attention kernel, the combine and the workspace.
// Short contexts: with an automatic split, at most kShortMaxUnits (sequence, query)
// units over at most kShortMaxKv cached tokens take the short-context kernel
// (csrc/decode_short.cu), one CTA per 8 heads and no split.
constexpr int kShortMaxKv = 1024;
constexpr int kShortMaxUnits = 2;

struct SplitPlan {
  int max_pages;    // ceil(max_kv_len / 64)
  int split_pages;  // pages per split
  int num_splits;   // ceil(max_pages / split_pages)
  bool short_path;  // the short-context kernel (then num_splits == 1)
  size_t o_part_bytes;
  size_t lse_part_bytes;
  size_t workspace_bytes;  // 0 when num_splits == 1
};

// ---- launchers (each defined in its own .cu; return cudaGetLastError()) ----
cudaError_t launch_append_kv(const uint16_t* c_kv_new, const uint16_t* k_pe_new,
                             const int32_t* seq_lens_before, const int32_t* page_table,
                             int pt_stride, const float* rope_table, int rope_max_pos,
                             uint16_t* cache, int64_t num_pages, int B, int n_new,
                             int* status, cudaStream_t stream);

cudaError_t launch_absorb_q(const uint16_t* q_nope, const uint16_t* q_rope,
                            const int32_t* seq_lens_before, const uint16_t* w_uk,
                            const float* rope_table, int rope_max_pos, uint16_t* q_abs,
                            int B, int n_q, int* status, cudaStream_t stream);

// absorb_q whose launch also appends the step's B * n_q new cache rows.
cudaError_t launch_append_absorb_q(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const uint16_t* q_nope,
                                   const uint16_t* q_rope, const int32_t* seq_lens_before, const int32_t* page_table,
                                   int pt_stride, const uint16_t* w_uk, const float* rope_table, int rope_max_pos,
                                   uint16_t* cache, int64_t num_pages, uint16_t* q_abs, int B, int n_q, int* status,
                                   cudaStream_t stream);
// The same with the FP8 latent cache (the rows as mla_append_kv_fp8 writes them).
cudaError_t launch_append_absorb_q_fp8(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const uint16_t* q_nope,
                                       const uint16_t* q_rope, const int32_t* seq_lens_before,
                                       const int32_t* page_table, int pt_stride, const uint16_t* w_uk,
                                       const float* rope_table, int rope_max_pos, uint8_t* c8, float* scale,
                                       uint16_t* kr, int64_t num_pages, uint16_t* q_abs, int B, int n_q, int* status,
                                       cudaStream_t stream);

// Clusters of the attention kernel that fit on the current device at once.
int decode_cluster_slots();

// The split-KV plan every decode entry point uses (false for invalid sizes), and
// the device address of the current device's status word (nullptr on failure).
bool split_plan(int B, int n_q, int max_kv_len, int split_pages, SplitPlan* plan);

// Launch overlap level (mla_set_launch_overlap): 0 plain stream order; 1 launch
// with programmatic stream serialization (prologues overlap the previous
// kernel); 2 as 1, and weight matrices are also read before grid_dep_wait().
int launch_overlap();

// The current device as an index into per-device tables of at most
// kMaxDevicesLocal entries, or -1.
constexpr int kMaxDevicesLocal = 64;
inline int current_device_index() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesLocal) return -1;
  return dev;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() > 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
int* device_status_word();

// SM-driven copy of `bytes` from src to dst, both device-addressable (csrc/copy.cu);
// `src_is_host`: the source is host memory, which no kernel writes.
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, bool src_is_host, cudaStream_t stream);

// One warp waiting on an mbarrier nothing completes, given up after limit_ns (csrc/selftest.cu).
cudaError_t launch_wait_timeout(int* status, uint64_t limit_ns, cudaStream_t stream);

// o_out: with one split the final O' (fp32 [B, n_q, 128, 512]); with several,
// the splits' partials O'_s as bf16 [B, n_q, splits, 128, 512] (the merge reads
// them; each is normalised within its split, so bf16 keeps its relative error
// at 2^-9 whatever the context length).  lse_out: fp32, per split likewise.
cudaError_t launch_decode_partial(const uint16_t* q_abs, const uint16_t* cache,
                                  int64_t num_pages, const int32_t* page_table, int pt_stride,
                                  const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                  const SplitPlan& plan, void* o_out, float* lse_out,
                                  int* status, cudaStream_t stream);

// One CTA per (sequence, query, 8 heads), warp-level MMAs, no split: O' and lse
// straight into o_out / lse_out (csrc/decode_short.cu); max_kv_len <= kShortMaxKv.
cudaError_t launch_decode_short(const uint16_t* q_abs, const uint16_t* cache, int64_t num_pages,
                                const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                int max_kv_len, float* o_out, float* lse_out, int* status, cudaStream_t stream);

// The attention a plan asks for: the short-context kernel when plan.short_path,
// else the 2-CTA split kernel (csrc/decode_short.cu).
cudaError_t launch_decode_planned(const uint16_t* q_abs, const uint16_t* cache, int64_t num_pages,
                                  const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                  int max_kv_len, const SplitPlan& plan, void* o_out, float* lse_out, int* status,
                                  cudaStream_t stream);

cudaError_t launch_decode_partial_fp8(const uint16_t* q_abs, const uint8_t* cache_c8, const float* cache_scale,
                                      const uint16_t* cache_kr, int64_t num_pages, const int32_t* page_table,
                                      int pt_stride, const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                      const SplitPlan& plan, void* o_out, float* lse_out, int* status,
                                      cudaStream_t stream);

cudaError_t launch_append_kv_fp8(const uint16_t* c_kv_new, const uint16_t* k_pe_new,
                                 const int32_t* seq_lens_before, const int32_t* page_table,
                                 int pt_stride, const float* rope_table, int rope_max_pos,
                                 uint8_t* c8, float* scale, uint16_t* kr, int64_t num_pages, int B, int n_new,
                                 int* status, cudaStream_t stream);

int linear_num_splits(int T, int K, int N);
size_t linear_workspace_bytes(int T, int K, int N, int N1 = 0);
cudaError_t launch_linear(const uint16_t* x, const uint16_t* w, uint16_t* y, int T, int K, int N, int64_t y_ld,
                          int seg, int seg_ld, float* part, int* status, cudaStream_t stream);
cudaError_t launch_linear_pair(const uint16_t* x, const uint16_t* w0, uint16_t* y0, int N0, const uint16_t* w1,
                               uint16_t* y1, int N1, int T, int K, float* part, int* status, cudaStream_t stream);
cudaError_t launch_rope_q(const uint16_t* q_rope, const int32_t* seq_lens_before, const float* rope_table,
                          int rope_max_pos, uint16_t* q_abs, int B, int n_q, int* status, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t stream);

// o_part: the bf16 partials of launch_decode_partial
cudaError_t launch_combine(const uint16_t* o_part, const float* lse_part, int B, int n_q,
                           int num_splits, float* o_latent, float* lse, cudaStream_t stream);

cudaError_t launch_out_absorb(const float* o_latent, const uint16_t* w_uv, uint16_t* out,
                              int B, int n_q, int* status, cudaStream_t stream);

cudaError_t launch_decompress_kv(const uint16_t* cache, int64_t num_pages, const int32_t* page_table, int pt_stride,
                                 const int32_t* kv_lens, int B, int max_kv_len, const uint16_t* w_uk,
                                 const uint16_t* w_uv, uint16_t* k_out, uint16_t* v_out, int* status,
                                 cudaStream_t stream);

cudaError_t launch_prefill_attn(const uint16_t* q_nope, const uint16_t* q_rope, const int32_t* seq_lens_before,
                                const float* rope_table, int rope_max_pos, const uint16_t* k_nope,
                                const uint16_t* v, int max_kv_len, const uint16_t* cache, int64_t num_pages,
                                const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                uint16_t* out, float* lse, int* status, cudaStream_t stream);

cudaError_t launch_combine_out_absorb(const uint16_t* o_part, const float* lse_part, int num_splits,
                                      const uint16_t* w_uv, uint16_t* out, float* lse, int B, int n_q,
                                      int* status, cudaStream_t stream);

}  // namespace mla
