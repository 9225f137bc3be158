// Copies between buffers the GPU addresses directly: device memory, or pinned
// host memory mapped into the device's address space (on an NVLink-C2C system
// the GPU reads and writes the host's pinned memory at link speed).  A decode
// step's inputs (about 1.6 MB at B = 32) and its output (1 MB) move by SM loads
// and stores spread over the whole GPU instead of the copy engines, and the
// copy joins the programmatic-dependent-launch chain of the step's kernels: an
// upload from host memory may read its source before the previous kernel of
// the stream has finished (only its stores wait), a download waits before it
// reads.  No counterpart on the MLA pages: this is the transport of the step.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per thread

// n16 vectors of 16 bytes, then `tail` (< 16) bytes after them.  With
// `early`, each thread's first kUnroll vectors are loaded before the wait for
// the previous kernel (the source is not written by any kernel).
__global__ void __launch_bounds__(kThreads)
copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n16, int tail, bool early) {
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  int64_t i = tid;
  if (early) {
    uint4 v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (i + k * nthreads < n16) v[k] = src[i + k * nthreads];
    grid_dep_wait();
    grid_dep_launch();
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (i + k * nthreads < n16) dst[i + k * nthreads] = v[k];
    i += kUnroll * nthreads;
  } else {
    grid_dep_wait();
    grid_dep_launch();
  }
  for (; i < n16; i += kUnroll * nthreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (i + k * nthreads < n16) v[k] = src[i + k * nthreads];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (i + k * nthreads < n16) dst[i + k * nthreads] = v[k];
  }
  if (tid < tail) {
    reinterpret_cast<uint8_t*>(dst + n16)[tid] = reinterpret_cast<const uint8_t*>(src + n16)[tid];
  }
}

// Any alignment: one byte per thread and step.
__global__ void __launch_bounds__(kThreads) copy1_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                        int64_t n) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kThreads)
    dst[i] = src[i];
}

int g_sms = 0;

}  // namespace

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, bool src_is_host, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || g_sms <= 0) g_sms = 148;
  }
  const int64_t most = 2ll * g_sms;  // two CTAs per SM
  const bool aligned = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
  if (aligned) {
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    const int tail = static_cast<int>(bytes % 16);
    const int64_t want = (n16 + static_cast<int64_t>(kThreads) * kUnroll - 1) / (static_cast<int64_t>(kThreads) * kUnroll);
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < most ? want : most));
    return launch_kernel(copy16_kernel, dim3(blocks), dim3(kThreads), 0, stream, static_cast<uint4*>(dst),
                         static_cast<const uint4*>(src), n16, tail, src_is_host && launch_overlap() >= 2);
  }
  const int64_t want = (static_cast<int64_t>(bytes) + kThreads - 1) / kThreads;
  const int blocks = static_cast<int>(want < most ? want : most);
  return launch_kernel(copy1_kernel, dim3(blocks), dim3(kThreads), 0, stream, static_cast<uint8_t*>(dst),
                       static_cast<const uint8_t*>(src), static_cast<int64_t>(bytes));
}

}  // namespace mla
