// The C ABI of include/mla_decode.h: argument validation, split planning,
// the per-device status word, the RoPE table, and the launches.
#include <limits.h>
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.cuh"

// Per-device fault word written by the kernels (first code wins).
__device__ int g_mla_device_status;

namespace {

using namespace mla;

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
int* g_status_ptr[kMaxDevices];
std::atomic<int> g_launch_overlap{1};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Device address of the status word on the current device (nullptr on failure).
int* status_ptr() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mla_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The device address of [p, p + bytes) if the current device can address all of
// it: device memory of this device, managed memory, or pinned host memory
// mapped into the device's address space (`host` is then set).
bool device_view(const void* p, size_t bytes, void** out, bool* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  *host = false;
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != current_device()) return false;
      break;
    case cudaMemoryTypeManaged:
      break;
    case cudaMemoryTypeHost:
      *host = true;
      break;
    default:
      return false;  // pageable host memory
  }
  if (a.devicePointer == nullptr) return false;
  *out = a.devicePointer;
  // the whole range lies inside the one allocation (the driver entry point is looked
  // up once; a function-local static is initialised once even under concurrent calls)
  static const PFN_cuMemGetAddressRange_v3020 range = []() -> PFN_cuMemGetAddressRange_v3020 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 3020, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
  }();
  if (range == nullptr) return false;
  CUdeviceptr base = 0;
  size_t size = 0;
  if (range(&base, &size, reinterpret_cast<CUdeviceptr>(*out)) != CUDA_SUCCESS) return false;
  const uintptr_t start = reinterpret_cast<uintptr_t>(*out);
  return start >= base && bytes <= size && start - base <= size - bytes;
}

// Split-KV partition.  Automatic choice: the split count s per (sequence,
// query) that minimises waves(s) * (pages per split + 3), where a wave is as
// many units as attention clusters fit on the GPU at once and 3 pages stand for
// a unit's fixed cost (query load, pipeline fill, epilogue, partial write).
bool make_plan(int B, int n_q, int max_kv_len, int split_pages, SplitPlan* plan) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ || max_kv_len < n_q || split_pages < 0) return false;
  plan->max_pages = (max_kv_len + kPage - 1) / kPage;
  plan->short_path = split_pages == 0 && max_kv_len <= kShortMaxKv &&
                     static_cast<int64_t>(B) * n_q <= kShortMaxUnits;
  if (plan->short_path) split_pages = plan->max_pages;  // one split: no merge
  if (split_pages == 0) {
    const int64_t units = static_cast<int64_t>(B > 0 ? B : 1) * n_q;
    const int64_t slots = decode_cluster_slots();
    int64_t best_cost = -1;
    split_pages = plan->max_pages;
    for (int s = 1; s <= plan->max_pages && s <= 256; ++s) {
      const int sp = (plan->max_pages + s - 1) / s;
      const int s_eff = (plan->max_pages + sp - 1) / sp;
      const int64_t waves = (units * s_eff + slots - 1) / slots;
      const int64_t cost = waves * (sp + 3);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        split_pages = sp;
      }
    }
  }
  plan->split_pages = split_pages;
  plan->num_splits = (plan->max_pages + split_pages - 1) / split_pages;
  const size_t rows = static_cast<size_t>(B) * n_q * plan->num_splits * kHeads;
  plan->o_part_bytes = round_up(rows * kLatent * sizeof(uint16_t), 256);  // bf16 partials
  plan->lse_part_bytes = round_up(rows * sizeof(float), 256);
  plan->workspace_bytes = plan->num_splits > 1 ? plan->o_part_bytes + plan->lse_part_bytes : 0;
  return true;
}

}  // namespace

namespace mla {
// Shared with other translation units of the library.
bool split_plan(int B, int n_q, int max_kv_len, int split_pages, SplitPlan* plan) {
  return make_plan(B, n_q, max_kv_len, split_pages, plan);
}
int* device_status_word() { return status_ptr(); }
int launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed); }
}  // namespace mla

extern "C" {

int mla_abi_version(void) { return 1; }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null pointer, bad size or alignment";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape outside what the kernels handle";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA runtime call or launch failed";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded wait in a kernel ran out";
    case MLA_ERR_BOUNDS: return "MLA_ERR_BOUNDS: a page id or position was out of range";
    case MLA_ERR_RANGE: return "MLA_ERR_RANGE: a partial attention score exceeded the exchange range";
  }
  return "MLA_ERR_UNKNOWN";
}

size_t mla_rope_table_bytes(int max_positions) {
  return max_positions > 0 ? static_cast<size_t>(max_positions) * kRope * sizeof(float) : 0;
}

mla_status mla_rope_table_init(float* table, int max_positions, cudaStream_t stream) {
  if (table == nullptr || max_positions <= 0 || !aligned16(table)) return MLA_ERR_INVALID_ARG;
  std::vector<float> host(static_cast<size_t>(max_positions) * kRope);
  double inv_freq[kHalfRope];
  for (int i = 0; i < kHalfRope; ++i) inv_freq[i] = pow(10000.0, -static_cast<double>(i) / kHalfRope);
  for (int p = 0; p < max_positions; ++p) {
    float* row = host.data() + static_cast<size_t>(p) * kRope;
    for (int i = 0; i < kHalfRope; ++i) {
      const double a = static_cast<double>(p) * inv_freq[i];
      row[i] = static_cast<float>(cos(a));
      row[kHalfRope + i] = static_cast<float>(sin(a));
    }
  }
  cudaError_t e = cudaMemcpyAsync(table, host.data(), host.size() * sizeof(float),
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return from_cuda(e);
}

mla_status mla_append_kv(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                         const int32_t* seq_lens_before, const int32_t* page_table,
                         int pt_stride, const float* rope_table, int rope_max_pos,
                         mla_bf16* cache, int64_t num_pages, int B, int n_new,
                         cudaStream_t stream) {
  if (B < 0 || n_new < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return MLA_OK;
  if (!c_kv_new || !k_pe_new || !seq_lens_before || !page_table || !rope_table || !cache)
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < 1 || rope_max_pos < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv_new) || !aligned16(cache)) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_append_kv(c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride,
                                    rope_table, rope_max_pos, cache, num_pages, B, n_new, st, stream));
}

mla_status mla_append_kv_fp8(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                             const int32_t* seq_lens_before, const int32_t* page_table,
                             int pt_stride, const float* rope_table, int rope_max_pos,
                             uint8_t* cache_c8, float* cache_scale, uint16_t* cache_kr,
                             int64_t num_pages, int B, int n_new, cudaStream_t stream) {
  if (B < 0 || n_new < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return MLA_OK;
  if (!c_kv_new || !k_pe_new || !seq_lens_before || !page_table || !rope_table || !cache_c8 || !cache_scale ||
      !cache_kr)
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < 1 || rope_max_pos < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv_new) || !aligned16(cache_c8)) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_append_kv_fp8(c_kv_new, k_pe_new, seq_lens_before, page_table, pt_stride, rope_table,
                                        rope_max_pos, cache_c8, cache_scale, cache_kr, num_pages, B, n_new, st,
                                        stream));
}

mla_status mla_decode_attn_fp8_partial(const mla_bf16* q_abs, const uint8_t* cache_c8, const float* cache_scale,
                                       const uint16_t* cache_kr, int64_t num_pages, const int32_t* page_table,
                                       int pt_stride, const int32_t* kv_lens, int B, int n_q, int max_kv_len,
                                       int split_pages, void* workspace, size_t workspace_bytes,
                                       float* o_latent, float* lse, cudaStream_t stream) {
  SplitPlan plan;
  if (!make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_abs || !cache_c8 || !cache_scale || !cache_kr || !page_table || !kv_lens || !o_latent || num_pages < 1 ||
      pt_stride < 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache_c8) || !aligned16(cache_scale) || !aligned16(cache_kr) ||
      !aligned16(o_latent))
    return MLA_ERR_INVALID_ARG;
  if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
                                   !aligned16(workspace)))
    return MLA_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  void* o_out = o_latent;
  float* lse_out = lse;
  if (plan.num_splits > 1) {
    o_out = workspace;
    lse_out = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.o_part_bytes);
  }
  return from_cuda(launch_decode_partial_fp8(q_abs, cache_c8, cache_scale, cache_kr, num_pages, page_table,
                                             pt_stride, kv_lens, B, n_q, max_kv_len, plan, o_out, lse_out, st,
                                             stream));
}

mla_status mla_linear_workspace_size(int T, int K, int N, size_t* bytes) {
  if (bytes == nullptr || T < 1 || T > MLA_LINEAR_MAX_T || K < 64 || K % 64 != 0 || N < 1) return MLA_ERR_INVALID_ARG;
  *bytes = linear_workspace_bytes(T, K, N);
  return MLA_OK;
}

mla_status mla_linear_strided(const mla_bf16* x, const mla_bf16* w, mla_bf16* y, int T, int K, int N, int64_t y_ld,
                              int seg, int seg_ld, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (T < 1 || T > MLA_LINEAR_MAX_T || K < 64 || K % 64 != 0 || N < 1) return MLA_ERR_INVALID_ARG;
  if (!x || !w || !y || !aligned16(x) || !aligned16(w)) return MLA_ERR_INVALID_ARG;
  if (seg < 1 || N % seg != 0 || seg_ld < seg || y_ld < static_cast<int64_t>(N / seg) * seg_ld) return MLA_ERR_INVALID_ARG;
  const size_t need = linear_workspace_bytes(T, K, N);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))) return MLA_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_linear(x, w, y, T, K, N, y_ld, seg, seg_ld, static_cast<float*>(workspace), st, stream));
}

mla_status mla_linear(const mla_bf16* x, const mla_bf16* w, mla_bf16* y, int T, int K, int N, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
  return mla_linear_strided(x, w, y, T, K, N, N, N, N, workspace, workspace_bytes, stream);
}

mla_status mla_linear_pair_workspace_size(int T, int K, int N0, int N1, size_t* bytes) {
  if (bytes == nullptr || T < 1 || T > MLA_LINEAR_MAX_T || K < 64 || K % 64 != 0 || N0 < 1 || N1 < 1)
    return MLA_ERR_INVALID_ARG;
  *bytes = linear_workspace_bytes(T, K, N0, N1);
  return MLA_OK;
}

mla_status mla_linear_pair(const mla_bf16* x, int T, int K, const mla_bf16* w0, int N0, mla_bf16* y0,
                           const mla_bf16* w1, int N1, mla_bf16* y1, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  if (T < 1 || T > MLA_LINEAR_MAX_T || K < 64 || K % 64 != 0 || N0 < 1 || N1 < 1) return MLA_ERR_INVALID_ARG;
  if (!x || !w0 || !y0 || !w1 || !y1 || !aligned16(x) || !aligned16(w0) || !aligned16(w1)) return MLA_ERR_INVALID_ARG;
  const size_t need = linear_workspace_bytes(T, K, N0, N1);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))) return MLA_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_linear_pair(x, w0, y0, N0, w1, y1, N1, T, K, static_cast<float*>(workspace), st, stream));
}

mla_status mla_rope_q(const mla_bf16* q_rope, const int32_t* seq_lens_before, const float* rope_table,
                      int rope_max_pos, mla_bf16* q_abs, int B, int n_q, cudaStream_t stream) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_rope || !seq_lens_before || !rope_table || !q_abs || rope_max_pos < 1) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_rope_q(q_rope, seq_lens_before, rope_table, rope_max_pos, q_abs, B, n_q, st, stream));
}

mla_status mla_f32_to_bf16(const float* src, mla_bf16* dst, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!src || !dst))) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  return from_cuda(launch_f32_to_bf16(src, dst, n, stream));
}

mla_status mla_absorb_q(const mla_bf16* q_nope, const mla_bf16* q_rope,
                        const int32_t* seq_lens_before, const mla_bf16* w_uk,
                        const float* rope_table, int rope_max_pos, mla_bf16* q_abs,
                        int B, int n_q, cudaStream_t stream) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_rope || !seq_lens_before || !w_uk || !rope_table || !q_abs || rope_max_pos < 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_abs))
    return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_absorb_q(q_nope, q_rope, seq_lens_before, w_uk, rope_table, rope_max_pos,
                                   q_abs, B, n_q, st, stream));
}

mla_status mla_append_absorb_q(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                               const mla_bf16* q_nope, const mla_bf16* q_rope,
                               const int32_t* seq_lens_before, const int32_t* page_table,
                               int pt_stride, const mla_bf16* w_uk,
                               const float* rope_table, int rope_max_pos,
                               mla_bf16* cache, int64_t num_pages, mla_bf16* q_abs,
                               int B, int n_q, cudaStream_t stream) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!c_kv_new || !k_pe_new || !q_nope || !q_rope || !seq_lens_before || !page_table || !w_uk || !rope_table ||
      !cache || !q_abs)
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < 1 || rope_max_pos < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv_new) || !aligned16(cache) || !aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) ||
      !aligned16(q_abs))
    return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_append_absorb_q(c_kv_new, k_pe_new, q_nope, q_rope, seq_lens_before, page_table, pt_stride,
                                          w_uk, rope_table, rope_max_pos, cache, num_pages, q_abs, B, n_q, st,
                                          stream));
}

mla_status mla_append_absorb_q_fp8(const mla_bf16* c_kv_new, const mla_bf16* k_pe_new,
                                   const mla_bf16* q_nope, const mla_bf16* q_rope,
                                   const int32_t* seq_lens_before, const int32_t* page_table,
                                   int pt_stride, const mla_bf16* w_uk,
                                   const float* rope_table, int rope_max_pos,
                                   uint8_t* cache_c8, float* cache_scale, uint16_t* cache_kr,
                                   int64_t num_pages, mla_bf16* q_abs, int B, int n_q,
                                   cudaStream_t stream) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!c_kv_new || !k_pe_new || !q_nope || !q_rope || !seq_lens_before || !page_table || !w_uk || !rope_table ||
      !cache_c8 || !cache_scale || !cache_kr || !q_abs)
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < 1 || rope_max_pos < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv_new) || !aligned16(cache_c8) || !aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) ||
      !aligned16(q_abs))
    return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_append_absorb_q_fp8(c_kv_new, k_pe_new, q_nope, q_rope, seq_lens_before, page_table,
                                              pt_stride, w_uk, rope_table, rope_max_pos, cache_c8, cache_scale,
                                              cache_kr, num_pages, q_abs, B, n_q, st, stream));
}

// An output buffer that may be pinned host memory: its device address (the
// kernels store to it across the host link), or the pointer itself for device
// memory.  False for pageable host memory or a range outside the allocation.
bool output_view(void* p, size_t bytes, void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeUnregistered) {
    *out = p;
    return true;
  }
  bool host = false;
  return device_view(p, bytes, out, &host);
}

mla_status mla_selftest_wait_timeout(int64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000ll) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_wait_timeout(st, static_cast<uint64_t>(limit_ns), stream));
}

mla_status mla_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return MLA_OK;
  if (dst == nullptr || src == nullptr) return MLA_ERR_INVALID_ARG;
  void *d = nullptr, *s = nullptr;
  bool d_host = false, s_host = false;
  if (!device_view(dst, bytes, &d, &d_host) || !device_view(src, bytes, &s, &s_host)) return MLA_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(d), b = reinterpret_cast<uintptr_t>(s);
  if (a < b + bytes && b < a + bytes) return MLA_ERR_INVALID_ARG;  // overlapping ranges
  return from_cuda(launch_copy(d, s, bytes, s_host, stream));
}

mla_status mla_decode_workspace_size(int B, int n_q, int max_kv_len, int split_pages, size_t* bytes) {
  SplitPlan plan;
  if (bytes == nullptr || !make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  *bytes = plan.workspace_bytes;
  return MLA_OK;
}

mla_status mla_decode_num_splits(int B, int n_q, int max_kv_len, int split_pages, int* num_splits) {
  SplitPlan plan;
  if (num_splits == nullptr || !make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  *num_splits = plan.num_splits;
  return MLA_OK;
}

mla_status mla_decode_uses_short_path(int B, int n_q, int max_kv_len, int split_pages, int* is_short) {
  SplitPlan plan;
  if (is_short == nullptr || !make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  *is_short = plan.short_path ? 1 : 0;
  return MLA_OK;
}

mla_status mla_decode_attn_partial(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                                   const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                                   int B, int n_q, int max_kv_len, int split_pages,
                                   void* workspace, size_t workspace_bytes,
                                   float* o_latent, float* lse, cudaStream_t stream) {
  SplitPlan plan;
  if (!make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_abs || !cache || !page_table || !kv_lens || !o_latent || num_pages < 1 || pt_stride < 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(o_latent)) return MLA_ERR_INVALID_ARG;
  if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
                                   !aligned16(workspace)))
    return MLA_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  void* o_out = o_latent;
  float* lse_out = lse;
  if (plan.num_splits > 1) {
    o_out = workspace;
    lse_out = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.o_part_bytes);
  }
  return from_cuda(launch_decode_planned(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q,
                                         max_kv_len, plan, o_out, lse_out, st, stream));
}

mla_status mla_decode_combine(int B, int n_q, int max_kv_len, int split_pages,
                              const void* workspace, size_t workspace_bytes,
                              float* o_latent, float* lse, cudaStream_t stream) {
  SplitPlan plan;
  if (!make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  if (B == 0 || plan.num_splits == 1) return MLA_OK;
  if (!o_latent || !aligned16(o_latent)) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < plan.workspace_bytes || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  const uint16_t* o_part = static_cast<const uint16_t*>(workspace);
  const float* lse_part = reinterpret_cast<const float*>(static_cast<const char*>(workspace) + plan.o_part_bytes);
  return from_cuda(launch_combine(o_part, lse_part, B, n_q, plan.num_splits, o_latent, lse, stream));
}

mla_status mla_decode_attn(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                           const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                           int B, int n_q, int max_kv_len, int split_pages,
                           void* workspace, size_t workspace_bytes,
                           float* o_latent, float* lse, cudaStream_t stream) {
  mla_status s = mla_decode_attn_partial(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q,
                                         max_kv_len, split_pages, workspace, workspace_bytes, o_latent,
                                         lse, stream);
  if (s != MLA_OK) return s;
  return mla_decode_combine(B, n_q, max_kv_len, split_pages, workspace, workspace_bytes, o_latent, lse,
                            stream);
}

mla_status mla_out_absorb(const float* o_latent, const mla_bf16* w_uv, mla_bf16* out, int B, int n_q,
                          cudaStream_t stream) {
  if (B < 0 || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!o_latent || !w_uv || !out) return MLA_ERR_INVALID_ARG;
  void* od = nullptr;
  if (!output_view(out, static_cast<size_t>(B) * n_q * kHeads * kNope * 2, &od)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_latent) || !aligned16(w_uv) || !aligned16(od)) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_out_absorb(o_latent, w_uv, static_cast<uint16_t*>(od), B, n_q, st, stream));
}

mla_status mla_combine_out_absorb(int B, int n_q, int max_kv_len, int split_pages,
                                  const void* workspace, size_t workspace_bytes, const float* o_latent,
                                  const mla_bf16* w_uv, mla_bf16* out, float* lse, cudaStream_t stream) {
  SplitPlan plan;
  if (!make_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (plan.num_splits == 1) return mla_out_absorb(o_latent, w_uv, out, B, n_q, stream);
  if (!w_uv || !out) return MLA_ERR_INVALID_ARG;
  void* od = nullptr;
  if (!output_view(out, static_cast<size_t>(B) * n_q * kHeads * kNope * 2, &od)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w_uv) || !aligned16(od)) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < plan.workspace_bytes || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  const uint16_t* o_part = static_cast<const uint16_t*>(workspace);
  const float* lse_part = reinterpret_cast<const float*>(static_cast<const char*>(workspace) + plan.o_part_bytes);
  return from_cuda(launch_combine_out_absorb(o_part, lse_part, plan.num_splits, w_uv, static_cast<uint16_t*>(od), lse,
                                             B, n_q, st, stream));
}

mla_status mla_decompress_kv(const mla_bf16* cache, int64_t num_pages, const int32_t* page_table, int pt_stride,
                             const int32_t* kv_lens, int B, int max_kv_len, const mla_bf16* w_uk,
                             const mla_bf16* w_uv, mla_bf16* k_nope, mla_bf16* v, cudaStream_t stream) {
  if (B < 0 || max_kv_len < 0 || num_pages < 0 || pt_stride < 0) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * kHeads * (max_kv_len + kPage) > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (B == 0 || max_kv_len == 0) return MLA_OK;
  if (!cache || !page_table || !kv_lens || !w_uk || !w_uv || !k_nope || !v) return MLA_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(k_nope) || !aligned16(v))
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < (max_kv_len + kPage - 1) / kPage) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_decompress_kv(cache, num_pages, page_table, pt_stride, kv_lens, B, max_kv_len, w_uk, w_uv,
                                        k_nope, v, st, stream));
}

mla_status mla_prefill_attn(const mla_bf16* q_nope, const mla_bf16* q_rope, const int32_t* seq_lens_before,
                            const float* rope_table, int rope_max_pos, const mla_bf16* k_nope, const mla_bf16* v,
                            int max_kv_len, const mla_bf16* cache, int64_t num_pages, const int32_t* page_table,
                            int pt_stride, const int32_t* kv_lens, int B, int n_q, mla_bf16* out, float* lse,
                            cudaStream_t stream) {
  if (B < 0 || n_q < 0 || max_kv_len < n_q || num_pages < 0 || pt_stride < 0 || rope_max_pos < 0)
    return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * kHeads * (max_kv_len + 128) > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (B == 0 || n_q == 0) return MLA_OK;
  if (!q_nope || !q_rope || !seq_lens_before || !rope_table || !k_nope || !v || !cache || !page_table ||
      !kv_lens || !out)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(rope_table) || !aligned16(k_nope) || !aligned16(v) ||
      !aligned16(cache) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  if (pt_stride < (max_kv_len + kPage - 1) / kPage) return MLA_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  return from_cuda(launch_prefill_attn(q_nope, q_rope, seq_lens_before, rope_table, rope_max_pos, k_nope, v,
                                       max_kv_len, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q, out,
                                       lse, st, stream));
}

mla_status mla_set_launch_overlap(int level) {
  if (level < 0 || level > 2) return MLA_ERR_INVALID_ARG;
  g_launch_overlap.store(level, std::memory_order_relaxed);
  return MLA_OK;
}

int mla_get_launch_overlap(void) { return g_launch_overlap.load(std::memory_order_relaxed); }

mla_status mla_get_device_status(cudaStream_t stream) {
  int* st = status_ptr();
  if (st == nullptr) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ERR_CUDA;
  return static_cast<mla_status>(value);
}

}  // extern "C"
