// Absorbed decode attention for short contexts: one CTA per (sequence, query,
// group of 8 heads), warp-level tensor-core tiles, without a KV split.
//
// Per (sequence b, query j) and head h, over the visible tokens t:
//   score_t = (q_abs[h,0:512] . c_t + q_abs[h,512:576] . kR_t) / sqrt(192)
//   O'[h] = sum_t softmax(score)_t c_t,   lse[h] = log sum_t exp(score_t)
// ("MLA 矩阵吸收 …" section 4.1: score = Q'_nope c^T + Q_rope k_rope^T, and the
//  V-side absorption O' = softmax . c; "DeepSeek-MLA-Principle" section 2: scale
//  1/sqrt(d_h + d_h^R), eq. (10); FlashMLA point 3: online softmax by block;
//  point 4: paged cache.)
//
// For a few queries over a few hundred cached tokens the 2-CTA split kernel is all
// fixed cost: each unit moves the whole 128-head query into TMEM, stores a 128 x
// 512 fp32 tile of O' and, once the history is split to spread the units, needs a
// merge.  Here the sequence's pages are spread over a cluster of up to 8 CTAs
// (contiguous ranges), each CTA takes 8 heads of one query, and the cluster merges
// its partials through distributed shared memory before writing O' and lse.  Per
// 64-token page the two contractions are thin, S^T = C q^T (64 tokens
// x 8 heads, K = 576) and O'^T += C^T P (512 x 8, K = 64 tokens), so they run as
// warp-level m16n8k16 bf16 MMAs (fp32 accumulation): the 8 heads are N = 8, and a
// tcgen05 tile of that width would be bound by its per-instruction latency.
//   * A page lands by 16-byte asynchronous copies of all 256 threads (consecutive
//     threads on consecutive units of a row) at a 1168-byte row stride, so the
//     eight rows an 8 x 8 ldmatrix reads start in different banks; rows past the
//     visible tokens are zero-filled instead of read (the cache may hold anything
//     there).  Two page buffers: the next page loads during this one's MMAs.
//   * S: warp w takes tokens 16 (w % 4) .. + 15 and half of K; the two halves are
//     added in shared memory.
//   * softmax: warp w takes head w (two tokens per lane): running max and sum in
//     the exp2 domain, P rounded to bf16 (the row sum adds the rounded values).
//   * O': warp w owns latent rows 64 w .. + 63 (four 16-row tiles) for all 8
//     heads, rescaled by each head's factor before the page's P V.
//   * merge (clusters of more than one CTA): after a cluster barrier (every CTA is
//     done with its page buffers) every CTA writes its running maxima and sums, and
//     every CTA but 0 its unnormalised partial O' (512 x 8 fp32, in the MMA
//     fragment order: four 16-byte stores per thread), into CTA 0's idle page
//     buffers; after a second barrier each thread of CTA 0 adds the partials at its
//     own fragment positions to the one in its registers, in rank order, each
//     weighted by 2^(m_s - M) against the largest max M, and writes
//     O' = sum / (sum of weighted row sums) and the natural log-sum-exp.
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHG = 8;                               // heads per CTA (the MMAs' N)
constexpr int kRowBytes = kRow * 2;                  // 1152
constexpr int kStride = kRowBytes + 16;              // padded row in shared memory
constexpr int kMaxPages = kShortMaxKv / kPage;       // 16
constexpr int kPStride = kPage + 8;                  // bf16 P row (per head), padded
static_assert(kHeads % kHG == 0, "head groups");
static_assert(kWarps == kHG, "one softmax warp per head");
static_assert(kLatent == kWarps * 64, "64 latent rows per warp");

struct Smem {
  alignas(128) uint8_t page[2][kPage * kStride];   // 2 x 74,752 B
  alignas(16) uint8_t q[kHG * kStride];            // the 8 heads' query rows
  float s[2][kPage][kHG];                          // S halves (K split over warp pairs)
  alignas(16) uint16_t p[kHG][kPStride];           // P (bf16) per head
  float fac[kHG];                                  // per-head rescale of O' for this page
  float l[kHG], m[kHG];                            // final row sums and maxima
  int page_ids[kMaxPages];
};

struct Params {
  const uint16_t* q_abs;
  const uint16_t* cache;
  const int32_t* page_table;
  const int32_t* kv_lens;
  float* o_out;
  float* lse_out;
  int* status;
  int64_t num_pages;
  int pt_stride;
  int n_q;
  int max_kv_len;
  int n_split;   // CTAs per cluster: the pages of a (sequence, query) in contiguous ranges
};

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D (16 x 8, fp32) += A (16 x 16, bf16, row-major) B (16 x 8, bf16, column-major)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) decode_short_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;  // MMA fragment coordinates
  constexpr int kGroups = kHeads / kHG;
  const int S = p.n_split;
  const int split = static_cast<int>(blockIdx.x) % S;        // the CTA's rank in its cluster
  const int rest = static_cast<int>(blockIdx.x) / S;
  const int h0 = (rest % kGroups) * kHG;
  const int unit = rest / kGroups;  // b * n_q + j
  const int b = unit / p.n_q, j = unit % p.n_q;

  grid_dep_wait();
  grid_dep_launch();
  // the 8 query rows (72 sixteen-byte units each), this thread's page id and the
  // length, all requested before anything is stored: none depends on another (an
  // invalid sequence's outputs are zeros whatever the query holds), and a store
  // through a byte pointer would keep every later load behind it
  constexpr int kQUnits = kHG * (kRowBytes / 16);  // 576
  const uint4* qsrc = reinterpret_cast<const uint4*>(p.q_abs + (static_cast<int64_t>(unit) * kHeads + h0) * kRow);
  uint4 qv[(kQUnits + kThreads - 1) / kThreads];
#pragma unroll
  for (int k = 0; k < (kQUnits + kThreads - 1) / kThreads; ++k)
    qv[k] = tid + kThreads * k < kQUnits ? __ldg(qsrc + tid + kThreads * k) : make_uint4(0, 0, 0, 0);
  const int pg_raw = tid < kMaxPages && tid < p.pt_stride ? p.page_table[static_cast<int64_t>(b) * p.pt_stride + tid] : 0;
  const int kv = p.kv_lens[b];
#pragma unroll
  for (int k = 0; k < (kQUnits + kThreads - 1) / kThreads; ++k) {
    const int u = tid + kThreads * k;
    if (u < kQUnits) *reinterpret_cast<uint4*>(sm.q + (u / (kRowBytes / 16)) * kStride + 16 * (u % (kRowBytes / 16))) = qv[k];
  }
  const bool bad = kv > p.max_kv_len || kv < p.n_q || (kv + kPage - 1) / kPage > p.pt_stride;
  const int n_vis = bad ? 0 : kv - p.n_q + j + 1;  // query j sees tokens 0 .. n_vis - 1
  const int n_pages = (n_vis + kPage - 1) / kPage;
  const int ppc = (n_pages + S - 1) / S;                     // pages per CTA of the cluster
  const int pb = min(n_pages, split * ppc), my_pages = min(n_pages, pb + ppc) - pb;  // pages pb .. pb + my_pages - 1
  if (tid == 0 && bad && j == 0 && h0 == 0) record_status(p.status, MLA_ERR_BOUNDS);
  if (tid < n_pages) {
    int pg = pg_raw;
    if (pg < 0 || pg >= p.num_pages) {
      record_status(p.status, MLA_ERR_BOUNDS);
      pg = 0;  // stay in bounds; the result of this row is not meaningful
    }
    sm.page_ids[tid] = pg;
  }
  __syncthreads();  // page ids and query in place

  // page i into buffer i & 1 (one commit group per call, empty past the last page):
  // thread tid copies units tid + 256 k of the page's 64 x 72 sixteen-byte units
  auto issue = [&](int i) {  // the CTA's i-th page
    if (i < my_pages) {
      const int nt = min(kPage, n_vis - (pb + i) * kPage);
      const uint8_t* src = reinterpret_cast<const uint8_t*>(p.cache + static_cast<int64_t>(sm.page_ids[pb + i]) * kPage * kRow);
      const uint32_t dst = smem_u32(sm.page[i & 1]);
      for (int u = tid; u < kPage * (kRowBytes / 16); u += kThreads) {
        const int r = u / (kRowBytes / 16), c = u % (kRowBytes / 16);
        cp_async16_zfill(dst + r * kStride + 16 * c, src + (r < nt ? r * kRowBytes + 16 * c : 0), r < nt ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  issue(0);
  issue(1);

  const uint32_t q_base = smem_u32(sm.q);
  static_assert(2 * kPage * kStride >= (7 * kHG * kLatent + 2 * 8 * kHG) * 4, "merge staging fits the page buffers");
  float o[4][4] = {};                      // O'^T tiles: latent rows 64 warp + 16 i, heads 2 t4, 2 t4 + 1
  float m_run = -INFINITY, l_run = 0.f;    // head `warp` (softmax warp)
  for (int i = 0; i < my_pages; ++i) {
    cp_async_wait_group<1>();  // this thread's copies of page i (page i + 1 may still be in flight)
    __syncthreads();           // everyone's
    const uint32_t pg_base = smem_u32(sm.page[i & 1]);
    const int nt = min(kPage, n_vis - (pb + i) * kPage);  // visible tokens of the page (the rest are zeros)
    // S^T (tokens x heads): warp w -> tokens 16 (w & 3) .. + 15, K half w >> 2 (18 steps of 16)
    {
      const int t0 = 16 * (warp & 3), k0 = (warp >> 2) * (kRow / 2);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t a_addr = pg_base + (t0 + (lane & 7) + ((lane >> 3) & 1) * 8) * kStride + (lane >> 4) * 16;
      const uint32_t b_addr = q_base + (lane & 7) * kStride + (lane >> 3) * 16;
#pragma unroll 3
      for (int kk = 0; kk < kRow / 2; kk += 32) {  // two K steps per B load
        uint32_t a0[4], a1[4], bq[4];
        ldsm_x4(a_addr + 2 * (k0 + kk), a0);
        ldsm_x4(a_addr + 2 * (k0 + kk + 16), a1);
        ldsm_x4(b_addr + 2 * (k0 + kk), bq);
        mma_16816(acc, a0, bq[0], bq[1]);
        mma_16816(acc, a1, bq[2], bq[3]);
      }
      float* sh = &sm.s[warp >> 2][0][0];
      sh[(t0 + g) * kHG + 2 * t4] = acc[0];
      sh[(t0 + g) * kHG + 2 * t4 + 1] = acc[1];
      sh[(t0 + g + 8) * kHG + 2 * t4] = acc[2];
      sh[(t0 + g + 8) * kHG + 2 * t4 + 1] = acc[3];
    }
    __syncthreads();
    // online softmax of head `warp` over the page's tokens (lane, lane + 32)
    {
      const int hh = warp;
      float v0 = (sm.s[0][lane][hh] + sm.s[1][lane][hh]) * kScaleLog2;
      float v1 = (sm.s[0][lane + 32][hh] + sm.s[1][lane + 32][hh]) * kScaleLog2;
      if (lane >= nt) v0 = -INFINITY;
      if (lane + 32 >= nt) v1 = -INFINITY;
      const float m_new = fmaxf(m_run, warp_max(fmaxf(v0, v1)));  // finite: the page has a visible token
      const float factor = ex2_approx(m_run - m_new);              // 0 on the first page
      const uint16_t p0 = f32_to_bf16_bits(ex2_approx(v0 - m_new));  // exp2(-inf) = 0 past the tokens
      const uint16_t p1 = f32_to_bf16_bits(ex2_approx(v1 - m_new));
      sm.p[hh][lane] = p0;
      sm.p[hh][lane + 32] = p1;
      l_run = l_run * factor + warp_sum(__uint_as_float(static_cast<uint32_t>(p0) << 16) +
                                        __uint_as_float(static_cast<uint32_t>(p1) << 16));
      m_run = m_new;
      if (lane == 0) sm.fac[hh] = factor;
    }
    __syncthreads();
    // O'^T += C^T P: warp w -> latent rows 64 w + 16 mi .. + 15, all 8 heads, K = 64 tokens
    {
      const float f0 = sm.fac[2 * t4], f1 = sm.fac[2 * t4 + 1];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        o[mi][0] *= f0;
        o[mi][1] *= f1;
        o[mi][2] *= f0;
        o[mi][3] *= f1;
      }
      const uint32_t a_addr = pg_base + ((lane & 7) + (lane >> 4) * 8) * kStride + (64 * warp + ((lane >> 3) & 1) * 8) * 2;
#pragma unroll
      for (int kk = 0; kk < kPage; kk += 16) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&sm.p[g][kk + 2 * t4]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&sm.p[g][kk + 8 + 2 * t4]);
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
          uint32_t a[4];
          ldsm_x4_t(a_addr + kk * kStride + mi * 32, a);
          mma_16816(o[mi], a, b0, b1);
        }
      }
    }
    __syncthreads();  // the page buffer, S and P may be reused
    issue(i + 2);
  }
  cp_async_wait_group<0>();

  const bool valid = n_vis > 0;
  if (S == 1) {
    if (lane == 0) {
      sm.l[warp] = l_run;
      sm.m[warp] = m_run;
    }
    __syncthreads();
    const float inv0 = valid ? 1.f / sm.l[2 * t4] : 0.f, inv1 = valid ? 1.f / sm.l[2 * t4 + 1] : 0.f;
    float* out0 = p.o_out + (static_cast<int64_t>(unit) * kHeads + h0 + 2 * t4) * kLatent;
    float* out1 = out0 + kLatent;
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      const int m = 64 * warp + 16 * mi + g;
      out0[m] = o[mi][0] * inv0;
      out1[m] = o[mi][1] * inv1;
      out0[m + 8] = o[mi][2] * inv0;
      out1[m + 8] = o[mi][3] * inv1;
    }
    if (tid < kHG && p.lse_out != nullptr)
      p.lse_out[static_cast<int64_t>(unit) * kHeads + h0 + tid] =
          valid ? (sm.m[tid] + log2f(sm.l[tid])) * kLn2 : -INFINITY;
    return;
  }
  // cluster merge: CTA 0's page buffers hold the partial O' of CTAs 1 .. S - 1 as
  // [S - 1][4 tiles][256 threads][4], then [S][8] maxima and [S][8] row sums
  float* stage = reinterpret_cast<float*>(sm.page[0]);
  constexpr int kPart = kHG * kLatent;
  float* ms = stage + 7 * kPart;
  float* ls = ms + 8 * kHG;
  cluster_sync();  // every CTA of the cluster is done with its page buffers
  {
    const uint32_t st0 = mapa(smem_u32(stage), 0);
    if (split > 0) {
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
        st_cluster_v4(st0 + 4 * ((split - 1) * kPart + (mi * kThreads + tid) * 4), o[mi][0], o[mi][1], o[mi][2],
                      o[mi][3]);
    }
    if (lane == 0) {
      st_cluster_f32(mapa(smem_u32(ms + split * kHG + warp), 0), m_run);
      st_cluster_f32(mapa(smem_u32(ls + split * kHG + warp), 0), l_run);
    }
  }
  cluster_sync();  // the partials are in CTA 0
  if (split != 0) return;
  {
    // heads 2 t4 and 2 t4 + 1 of this thread's fragments: weights of every CTA's partial
    float M[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < S) {
        M[0] = fmaxf(M[0], ms[k * kHG + 2 * t4]);
        M[1] = fmaxf(M[1], ms[k * kHG + 2 * t4 + 1]);
      }
    float w[8][2], lsum[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        w[k][e] = k < S && valid ? ex2_approx(ms[k * kHG + 2 * t4 + e] - M[e]) : 0.f;  // 0 for a CTA without pages
        if (k < S) lsum[e] += w[k][e] * ls[k * kHG + 2 * t4 + e];
      }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mi][e] *= w[0][e & 1];
#pragma unroll
    for (int k = 1; k < 8; ++k) {
      if (k >= S) break;
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const float4 x = *reinterpret_cast<const float4*>(stage + (k - 1) * kPart + (mi * kThreads + tid) * 4);
        o[mi][0] += w[k][0] * x.x;
        o[mi][1] += w[k][1] * x.y;
        o[mi][2] += w[k][0] * x.z;
        o[mi][3] += w[k][1] * x.w;
      }
    }
    const float inv0 = valid ? 1.f / lsum[0] : 0.f, inv1 = valid ? 1.f / lsum[1] : 0.f;
    float* out0 = p.o_out + (static_cast<int64_t>(unit) * kHeads + h0 + 2 * t4) * kLatent;
    float* out1 = out0 + kLatent;
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      const int m = 64 * warp + 16 * mi + g;
      out0[m] = o[mi][0] * inv0;
      out1[m] = o[mi][1] * inv1;
      out0[m + 8] = o[mi][2] * inv0;
      out1[m + 8] = o[mi][3] * inv1;
    }
    if (warp == 0 && g == 0 && p.lse_out != nullptr) {
      float* lse = p.lse_out + static_cast<int64_t>(unit) * kHeads + h0 + 2 * t4;
      lse[0] = valid ? (M[0] + log2f(lsum[0])) * kLn2 : -INFINITY;
      lse[1] = valid ? (M[1] + log2f(lsum[1])) * kLn2 : -INFINITY;
    }
  }
}

bool g_configured[kMaxDevicesLocal];
int g_sms[kMaxDevicesLocal];

}  // namespace

cudaError_t launch_decode_short(const uint16_t* q_abs, const uint16_t* cache, int64_t num_pages,
                                const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                int max_kv_len, float* o_out, float* lse_out, int* status, cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(B) * n_q;
  if (units == 0) return cudaSuccess;
  if (max_kv_len > kShortMaxKv) return cudaErrorInvalidValue;
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  const size_t smem = sizeof(Smem) + 128;
  if (!g_configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_configured[dev] = true;
  }
  // spread the pages over a cluster while the CTAs stay within about one wave
  const int64_t groups = units * (kHeads / kHG);
  const int max_pages = (max_kv_len + kPage - 1) / kPage;
  int64_t s = (g_sms[dev] * 4 / 5) / groups;
  s = s < 1 ? 1 : (s > 8 ? 8 : s);
  if (s > max_pages) s = max_pages > 0 ? max_pages : 1;
  Params prm;
  prm.q_abs = q_abs;
  prm.cache = cache;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.o_out = o_out;
  prm.lse_out = lse_out;
  prm.status = status;
  prm.num_pages = num_pages;
  prm.pt_stride = pt_stride;
  prm.n_q = n_q;
  prm.max_kv_len = max_kv_len;
  prm.n_split = static_cast<int>(s);
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = static_cast<unsigned>(s);
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (launch_overlap() > 0) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups * s));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_short_kernel, prm);
}

cudaError_t launch_decode_planned(const uint16_t* q_abs, const uint16_t* cache, int64_t num_pages,
                                  const int32_t* page_table, int pt_stride, const int32_t* kv_lens, int B, int n_q,
                                  int max_kv_len, const SplitPlan& plan, void* o_out, float* lse_out, int* status,
                                  cudaStream_t stream) {
  if (plan.short_path)  // a single split: o_out is the final fp32 O'
    return launch_decode_short(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q, max_kv_len,
                               static_cast<float*>(o_out), lse_out, status, stream);
  return launch_decode_partial(q_abs, cache, num_pages, page_table, pt_stride, kv_lens, B, n_q, max_kv_len, plan,
                               o_out, lse_out, status, stream);
}

}  // namespace mla
