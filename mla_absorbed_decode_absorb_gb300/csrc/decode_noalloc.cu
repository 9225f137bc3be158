// mla_decode_attn_noalloc: split-KV attention plus combine with the split
// partials kept in a fixed array inside this library instead of a caller-provided
// workspace.
//
// Some callers cannot allocate device memory when they call the decode step:
// code running inside an allocator-free runtime (an inference server whose
// memory pool is fully reserved up front, a plugin that may only use the
// buffers handed to it, an embedding that forbids cudaMalloc on its hot path).
// For them this entry point needs nothing but the inputs and outputs.  Its
// scratch is one file-scope device array of kNoallocScratchBytes (16 MiB), which
// every GPU that loads the library holds until the process exits.  Calls share
// that array, so calls that overlap on the GPU race with each other.
#include <mutex>

#include "internal.cuh"

namespace mla {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;

// Split partials (per-split O' and log-sum-exp) of calls to the entry point below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per
// device (the array's host-side name is not a device address).  A failed lookup
// clears the runtime's pending error, so that it is not reported later by an
// unrelated launch of this library.  The cached address belongs to the device's
// current context: after cudaDeviceReset it is stale, and this entry point must
// not be called again in that process.
void* scratch_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

extern "C" mla_status mla_decode_attn_noalloc(const mla_bf16* q_abs, const mla_bf16* cache, int64_t num_pages,
                                              const int32_t* page_table, int pt_stride, const int32_t* kv_lens,
                                              int B, int n_q, int max_kv_len, int split_pages, float* o_latent,
                                              float* lse, cudaStream_t stream) {
  using namespace mla;
  SplitPlan plan;
  if (!split_plan(B, n_q, max_kv_len, split_pages, &plan)) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_abs || !cache || !page_table || !kv_lens || !o_latent || num_pages < 1 || pt_stride < 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(o_latent)) return MLA_ERR_INVALID_ARG;
  if (plan.workspace_bytes > kNoallocScratchBytes) return MLA_ERR_WORKSPACE;
  int* st = device_status_word();
  if (st == nullptr) return MLA_ERR_CUDA;
  if (plan.num_splits == 1)
    return launch_decode_planned(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q, max_kv_len, plan,
                                 o_latent, lse, st, stream) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
  char* ws = static_cast<char*>(scratch_ptr());
  if (ws == nullptr) return MLA_ERR_CUDA;
  uint16_t* o_part = reinterpret_cast<uint16_t*>(ws);  // bf16 partials
  float* lse_part = reinterpret_cast<float*>(ws + plan.o_part_bytes);
  if (launch_decode_planned(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q, max_kv_len, plan, o_part,
                            lse_part, st, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  return launch_combine(o_part, lse_part, B, n_q, plan.num_splits, o_latent, lse, stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}
