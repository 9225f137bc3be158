// y[T, N] = x[T, K] W[N, K]^T for a few tokens (T <= 256): the projections of
// the MLA layer around the attention ("DeepSeek MLA 架构详解", decode listing:
// W_DKV, W_KR, W_DQ, W_UQ, W_QR and W_O are nn.Linear layers; "DeepSeek-MLA-
// Principle" section 2 table, the dimension changes 7168 -> 512, 7168 -> 64,
// 7168 -> 1536, 1536 -> 128 x 128, 1536 -> 128 x 64 and 16384 -> 7168).
//
// With T this small the work is streaming W once from HBM.  Operands are
// swapped so the weight is the M = 128 side of the tcgen05 MMA: one CTA owns
// 128 output features and a range of K, and streams its W tile and the matching
// columns of x through a TMA ring (128-byte swizzle, 64 K per stage), one
// thread issuing 4 MMAs (K = 16) per stage into a TMEM accumulator of T
// columns.  K is split over CTAs so that the grid covers the GPU; a split
// launch writes fp32 partials and a second kernel adds them in split order.
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

// A stage holds kBoxes consecutive 64-wide K boxes of the CTA's 128 weight rows
// (and of x): the weight rows are read kBoxes * 128 contiguous bytes at a time.
constexpr int kBoxes = 2;
constexpr int kKB = 64 * kBoxes;  // K per stage
constexpr int kThreads = 128;     // warp 0: TMA, warp 1: MMA; all four: epilogue
constexpr int kWBox = 128 * 128;  // 128 W rows x 64 K (bf16)
constexpr int kSmemBudget = 200 * 1024;

__host__ __device__ inline int pad16(int t) { return (t + 15) & ~15; }
__host__ __device__ inline int stage_bytes(int tp) { return kBoxes * (kWBox + tp * 128); }
constexpr int kMaxStages = 12;
__host__ __device__ inline int num_stages(int tp) { return min(kMaxStages, kSmemBudget / stage_bytes(tp)); }
__host__ __device__ inline uint32_t tmem_cols_for(int tp) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(tp)) c <<= 1;
  return c;
}
inline int smem_bytes_for(int tp) { return num_stages(tp) * stage_bytes(tp) + 256 + 1024; }
static_assert((2 * kMaxStages + 1) * 8 + 4 <= 256, "barrier block");

// One or two projections of the same x: CTAs [0, tiles0) compute y = x W^T with
// N outputs, CTAs [tiles0, ..) y1 = x W1^T with N1 outputs (N1 = 0: one projection).
struct LinParams {
  uint16_t* y;        // bf16 out (no split): element (t, n) at t * y_ld + (n / seg) * seg_ld + n % seg
  uint16_t* y1;       // second projection's bf16 out: element (t, n) at t * y1_ld + n
  float* part;        // [ksplit, T, N + N1] fp32 (split)
  int* status;
  int T, K, N, N1;
  int tiles0;         // 128-row tiles of the first projection
  int kb_per_split;   // K blocks of kKB per CTA
  int64_t y_ld, y1_ld;
  int seg, seg_ld;
};

__device__ __forceinline__ int64_t y_index(const LinParams& p, int t, int n) {
  return static_cast<int64_t>(t) * p.y_ld + static_cast<int64_t>(n / p.seg) * p.seg_ld + n % p.seg;
}

__global__ void __launch_bounds__(kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_w1, const LinParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tp = pad16(p.T);
  const int S = num_stages(tp);
  const int SB = stage_bytes(tp);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
  uint64_t* empty = full + kMaxStages;
  uint64_t* done = empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const uint32_t tmem_cols = tmem_cols_for(tp);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool second = static_cast<int>(blockIdx.x) >= p.tiles0;  // this CTA's projection
  const CUtensorMap* tw = second ? &tm_w1 : &tm_w;
  const int n0 = (static_cast<int>(blockIdx.x) - (second ? p.tiles0 : 0)) * 128;
  const int Ng = second ? p.N1 : p.N;
  const int ncol = second ? p.N + n0 : n0;  // column of the partials' row [N + N1]
  const int kb0 = blockIdx.y * p.kb_per_split;
  const int nkb = min(p.kb_per_split, (p.K + kKB - 1) / kKB - kb0);  // K past the end reads as zeros

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      if (!mbar_wait(smem_u32(&empty[s]), ((i / S) & 1) ^ 1, p.status)) break;
      uint8_t* st = smem + s * SB;
      mbar_arrive_expect_tx(smem_u32(&full[s]), SB);
      const int k = (kb0 + i) * kKB;
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_2d(smem_u32(st + bx * kWBox), tw, k + 64 * bx, n0, smem_u32(&full[s]));
        tma_load_2d(smem_u32(st + kBoxes * kWBox + bx * tp * 128), &tm_x, k + 64 * bx, 0, smem_u32(&full[s]));
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_bf16(128, tp, /*a_mn=*/0, /*b_mn=*/0);
    bool ok = true;
    for (int i = 0; i < nkb && ok; ++i) {
      const int s = i % S;
      ok = mbar_wait(smem_u32(&full[s]), (i / S) & 1, p.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + s * SB), b0 = a0 + kBoxes * kWBox;
#pragma unroll
      for (int q = 0; q < kKB / 16; ++q)
        mma_ss(tmem, smem_desc(a0 + (q >> 2) * kWBox + (q & 3) * 32, 16, 1024, kSw128),
               smem_desc(b0 + (q >> 2) * tp * 128 + (q & 3) * 32, 16, 1024, kSw128), idesc, (i | q) ? 1u : 0u);
      mma_commit(smem_u32(&empty[s]));
    }
    if (ok) mma_commit(smem_u32(done));
    else mbar_arrive(smem_u32(done));  // no result (the status is set): release the epilogue
  }
  __syncwarp();

  // -------------------------------------------------------------------- epilogue
  // TMEM lane = output feature n0 + 32 warp + lane, column = token
  const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done), 0, p.status));
  tc_fence_after();
  const int n = n0 + warp * 32 + lane;
  const int64_t ntot = p.N + p.N1;
  const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  auto put = [&](int t, float v) {
    if (gridDim.y > 1)
      p.part[(static_cast<int64_t>(blockIdx.y) * p.T + t) * ntot + ncol + warp * 32 + lane] = v;
    else if (second)
      p.y1[static_cast<int64_t>(t) * p.y1_ld + n] = f32_to_bf16_bits(v);
    else
      p.y[y_index(p, t, n)] = f32_to_bf16_bits(v);
  };
  if (ok && nkb > 0) {
    for (int c0 = 0; c0 < tp; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
      if (n < Ng) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = c0 + i;
          if (t < p.T) put(t, __uint_as_float(r[i]));
        }
      }
    }
  } else if (n < Ng) {
    for (int t = 0; t < p.T; ++t) put(t, 0.f);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

// y(t, n) = bf16(sum over splits s in order of part[s, t, n])
__global__ void __launch_bounds__(256)
linear_reduce_kernel(const float* __restrict__ part, const LinParams p, int ksplit) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t ntot = p.N + p.N1;
  const int64_t elems = static_cast<int64_t>(p.T) * ntot;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < elems;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // the loads of eight splits are in flight together; the sum keeps split order
    float a = 0.f;
    int s = 0;
    for (; s + 8 <= ksplit; s += 8) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = part[(s + q) * elems + e];
#pragma unroll
      for (int q = 0; q < 8; ++q) a += v[q];
    }
    for (; s < ksplit; ++s) a += part[s * elems + e];
    const int t = static_cast<int>(e / ntot), c = static_cast<int>(e % ntot);
    if (c < p.N)
      p.y[y_index(p, t, c)] = f32_to_bf16_bits(a);
    else
      p.y1[static_cast<int64_t>(t) * p.y1_ld + (c - p.N)] = f32_to_bf16_bits(a);
  }
}

int g_sms = 0;

}  // namespace

// K split so that tiles x splits fills one wave of the GPU (one CTA per SM),
// each split keeping at least 256 of K: a second, partial wave of short
// weight streams cost more than it overlapped (W_O, K = 16384: 60.9 -> 55.4 us).
int linear_num_splits(int T, int K, int N) {
  (void)T;
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || g_sms <= 0) g_sms = 148;
  }
  const int tiles = (N + 127) / 128;
  const int kbs = (K + kKB - 1) / kKB;
  int split = max(1, g_sms / tiles);
  // long weight streams (over 128 K blocks per split in one wave) keep a second wave
  // busy: W_OV, K = 65536, streamed faster in two (166 against 183 us)
  if (kbs / split > 128) split = max(1, (2 * g_sms) / tiles);
  split = min(split, max(1, kbs / (4 / kBoxes)));  // at least 256 K per split
  const int per = (kbs + split - 1) / split;
  return (kbs + per - 1) / per;  // no empty split
}

size_t linear_workspace_bytes(int T, int K, int N, int N1) {
  const int tiles = (N + 127) / 128 + (N1 + 127) / 128;
  const int split = linear_num_splits(T, K, 128 * tiles);
  return split > 1 ? static_cast<size_t>(split) * T * (N + N1) * sizeof(float) : 0;
}

namespace {

cudaError_t launch_linear_any(const uint16_t* x, const uint16_t* w, uint16_t* y, int T, int K, int N, int64_t y_ld,
                              int seg, int seg_ld, const uint16_t* w1, uint16_t* y1, int N1, int64_t y1_ld,
                              float* part, int* status, cudaStream_t stream) {
  const int tp = pad16(T);
  static bool configured[kMaxDevicesLocal] = {};  // the attribute is per device
  const int dev_ = current_device_index();
  if (dev_ < 0) return cudaErrorInvalidDevice;
  if (!configured[dev_]) {
    int most = 0;
    for (int t = 16; t <= 256; t += 16) most = max(most, smem_bytes_for(t));
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    configured[dev_] = true;
  }
  const int tiles0 = (N + 127) / 128, tiles = tiles0 + (N1 + 127) / 128;
  const int split = linear_num_splits(T, K, 128 * tiles);
  const int kbs = (K + kKB - 1) / kKB;
  CUtensorMap tx, tw, tw1;
  if (!make_tmap_bf16_2d(&tx, x, T, K, K, 64, tp, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16_2d(&tw, w, N, K, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (N1 > 0) {
    if (!make_tmap_bf16_2d(&tw1, w1, N1, K, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  } else {
    tw1 = tw;  // not read
  }
  LinParams prm;
  prm.y = y;
  prm.y1 = y1;
  prm.part = part;
  prm.status = status;
  prm.T = T;
  prm.K = K;
  prm.N = N;
  prm.N1 = N1;
  prm.tiles0 = tiles0;
  prm.kb_per_split = (kbs + split - 1) / split;
  prm.y_ld = y_ld;
  prm.y1_ld = y1_ld;
  prm.seg = seg;
  prm.seg_ld = seg_ld;
  cudaError_t e = launch_kernel(linear_tc_kernel, dim3(tiles, split), dim3(kThreads), smem_bytes_for(tp), stream, tx,
                                tw, tw1, prm);
  if (e != cudaSuccess || split == 1) return e;
  const int64_t elems = static_cast<int64_t>(T) * (N + N1);
  const int64_t want = (elems + 255) / 256;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  return launch_kernel(linear_reduce_kernel, dim3(blocks), dim3(256), 0, stream, static_cast<const float*>(part), prm,
                       split);
}

}  // namespace

cudaError_t launch_linear(const uint16_t* x, const uint16_t* w, uint16_t* y, int T, int K, int N, int64_t y_ld,
                          int seg, int seg_ld, float* part, int* status, cudaStream_t stream) {
  return launch_linear_any(x, w, y, T, K, N, y_ld, seg, seg_ld, nullptr, nullptr, 0, 0, part, status, stream);
}

cudaError_t launch_linear_pair(const uint16_t* x, const uint16_t* w0, uint16_t* y0, int N0, const uint16_t* w1,
                               uint16_t* y1, int N1, int T, int K, float* part, int* status, cudaStream_t stream) {
  return launch_linear_any(x, w0, y0, T, K, N0, N0, N0, N0, w1, y1, N1, N1, part, status, stream);
}

}  // namespace mla
