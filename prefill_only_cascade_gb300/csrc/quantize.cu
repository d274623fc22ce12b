// quantize.cu - per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of
// the qwen3-4b-fp8 model in the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
// GPU"). scale = amax / 448 (1 when amax == 0, IEEE fp32 division); code =
// e4m3_rn_satfinite(y) with y the correctly rounded fp32 quotient x / scale.
//
// Two calls:
//  * quail_quantize_kv_fp8 (kv_quantize_kernel): the scales are not known. Persistent
//    clusters of 8 CTAs (one CTA per SM, 8 warps) take slabs = (anchor, group of KV heads
//    with up to 256 contiguous bytes of every token row); the cluster splits the slab's
//    rows into 8 contiguous parts, and each warp of a CTA TMA-loads 32-row chunks of its
//    part into buffers of its own (3 x 8 KB). The slab stays in shared memory: each warp
//    forms the max |x| of its chunks as they land, the CTA maxima meet in CTA 0's shared
//    memory (distributed shared memory), and one cluster barrier later every thread
//    quantises its chunks from shared memory and stores the codes. HBM sees one read and
//    one write per element. A slab longer than the cluster's buffers (more than 24
//    chunks per CTA: anchors above 6,144 tokens at 256-byte rows) is read twice, in
//    rounds. Each warp issues the first round of its next slab as soon as its chunks of
//    the current slab are quantised.
//  * quail_quantize_kv_fp8_with_scales (kv_quantize_scaled_kernel): the amax of every
//    (anchor, KV head) is given (as the causal prefill emits it); a grid-stride stream of
//    16-byte loads and 8-byte stores, one read and one write per element.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kMaxHeadsPerSlab = 2;  // heads per 256-byte row (d >= 64)

// 8-byte store of codes with an L2 eviction policy (the codes are not re-read here)
__device__ __forceinline__ void st_hint_8(uint2* p, uint2 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x),
               "r"(v.y), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float absmax_bf16x8(const uint4& raw) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
  return m;
}

inline bool hkv_divides(int hkv, int n) { return hkv % n == 0; }

__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// x / s correctly rounded in fp32, given r = RN(1/s): q = RN(x r), then one correction
// with the exact residual x - q s (Markstein's division by reciprocal with an FMA
// correction: P. Markstein, "IA-64 and Elementary Functions", 2000). It can differ from
// the IEEE quotient only when the quotient underflows fp32, where the E4M3 code is a
// signed zero either way; the GPU tests compare it bit for bit with __fdiv_rn over every
// bf16 input for many scales.
__device__ __forceinline__ float div_by_recip(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q, s, x);
  // s > 0: the quotient has the sign of x (this keeps -0 / s = -0)
  return copysignf(__fmaf_rn(e, r, q), x);
}

// Eight bf16 -> eight E4M3 codes: e4m3_rn_satfinite(x / s), the quotient fp32.
__device__ __forceinline__ uint2 quantize_bf16x8(const uint4& raw, float s, float r) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 qv = make_float2(div_by_recip(__uint_as_float(w[k] << 16), s, r),
                                  div_by_recip(__uint_as_float(w[k] & 0xFFFF0000u), s, r));
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
    packed[k >> 1] |= static_cast<uint32_t>(c) << (16 * (k & 1));
  }
  return make_uint2(packed[0], packed[1]);
}

constexpr int kCluster = 8;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 32;              // rows per chunk
constexpr int kBufs = 3;               // chunk buffers per warp
constexpr int kChunkBytes = kRows * 256;
constexpr int kChunksPerRound = kWarps * kBufs;  // per CTA
constexpr int kSmemBytes = kWarps * kBufs * kChunkBytes + 1024;  // + alignment slack

struct __align__(8) QBars {
  uint64_t full[kWarps][kBufs];
  float warp_max[kWarps][kMaxHeadsPerSlab];
  float part[2][kCluster][kMaxHeadsPerSlab];  // CTA maxima, in CTA 0
  int abort_flag;
};

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* m, uint64_t* bar, void* dst, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Geometry of slab `slab` for CTA `rank` of the cluster.
struct Slab {
  int a, c;          // anchor, head group
  int64_t lo;        // first row of this CTA's part
  int rows;          // rows of this CTA's part
  int chunks;        // ceil(rows / kRows)
  int rounds;        // ceil(chunks / kChunksPerRound)
};
__device__ __forceinline__ Slab slab_geometry(int64_t slab, int groups, uint32_t rank,
                                              const int32_t* ao, int64_t T) {
  Slab g;
  g.a = static_cast<int>(slab / groups);
  g.c = static_cast<int>(slab % groups);
  // offsets clamped into [0, T]: inconsistent ones cannot address out of bounds
  const int64_t lo = min(max(static_cast<int64_t>(__ldg(ao + g.a)), int64_t{0}), T);
  const int64_t hi = min(max(static_cast<int64_t>(__ldg(ao + g.a + 1)), lo), T);
  const int64_t len = hi - lo;
  // rows per CTA: a multiple of kRows so that chunks never straddle two CTAs' parts
  const int64_t per = ((len + kCluster - 1) / kCluster + kRows - 1) / kRows * kRows;
  const int64_t start = min(static_cast<int64_t>(rank) * per, len);
  g.lo = lo + start;
  g.rows = static_cast<int>(min(per, len - start));
  g.chunks = (g.rows + kRows - 1) / kRows;
  g.rounds = (g.chunks + kChunksPerRound - 1) / kChunksPerRound;
  return g;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
kv_quantize_kernel(const __grid_constant__ CUtensorMap map, int num_anchors, int64_t T,
                   int hkv, int d, int hg, const int32_t* __restrict__ ao,
                   uint8_t* __restrict__ codes, float* __restrict__ scale, unsigned* err_word,
                   uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf0 = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ QBars bars;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = hg * d * 2;         // 128 or 256
  const int vpr = row_bytes / 16;           // 16-byte vectors per row: 8 or 16
  const int vph = d / 8;                    // vectors per head
  const int chunk_bytes = kRows * row_bytes;
  const int vec_per_lane = kRows * vpr / 32;  // 8 or 16
  const int col = lane & (vpr - 1);          // vpr divides 32: the lane's column is fixed
  const int my_head = col / vph;             // within the slab
  const int row_step = 32 / vpr;             // rows between a lane's vectors
  const int lane_row = lane / vpr;
  const int groups = hkv / hg;
  const int64_t slabs = static_cast<int64_t>(num_anchors) * groups;
  const int64_t n_clusters = gridDim.x / kCluster;
  const int64_t row_codes = static_cast<int64_t>(hkv) * d;  // code bytes per token row
  const uint64_t pol = l2_policy_evict_first();              // each byte is read once

  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int b = 0; b < kBufs; ++b) mbar_init(&bars.full[w][b], 1);
    bars.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map);
  }
  __syncthreads();
  WaitCtl wc;
  wc.timeout_ns = timeout_ns;
  wc.abort_flag = &bars.abort_flag;
  wc.err_word = err_word;

  uint32_t fills[kBufs] = {0, 0, 0};  // loads issued into each of this warp's buffers
  auto buf = [&](int b) { return buf0 + (warp * kBufs + b) * kChunkBytes; };
  // Issue this warp's chunks of round r of slab g (chunk j of the CTA's part is owned by
  // warp j % kWarps, buffer (j / kWarps) % kBufs).
  auto issue_round = [&](const Slab& g, int r) {
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads first
    for (int b = 0; b < kBufs; ++b) {
      const int j = r * kChunksPerRound + b * kWarps + warp;
      if (j < g.chunks) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.full[warp][b], chunk_bytes);
          tma_load_2d(&map, &bars.full[warp][b], buf(b), g.c * hg * d,
                      static_cast<int>(g.lo + static_cast<int64_t>(j) * kRows), pol);
        }
        ++fills[b];
      }
    }
    __syncwarp();
  };
  // Wait for this warp's buffer b (its latest load).
  auto wait_buf = [&](int b) { return wait_parity_warp(wc, &bars.full[warp][b], (fills[b] - 1) & 1u); };

  int64_t slab = blockIdx.x / kCluster;
  if (slab < slabs) issue_round(slab_geometry(slab, groups, rank, ao, T), 0);
  int parity = 0;
  for (; slab < slabs; slab += n_clusters) {
    const Slab g = slab_geometry(slab, groups, rank, ao, T);
    // pass 1: max |x| of this lane's head over this warp's chunks
    float m = 0.f;
    for (int r = 0; r < g.rounds; ++r) {
      if (r > 0) issue_round(g, r);  // round 0 was issued ahead
      for (int b = 0; b < kBufs; ++b) {
        const int j = r * kChunksPerRound + b * kWarps + warp;
        if (j >= g.chunks) continue;
        wait_buf(b);
        const int nrows = min(kRows, g.rows - j * kRows);
        const uint32_t base = smem_u32(buf(b));
        for (int i = 0; i < vec_per_lane; ++i) {
          const int row = lane_row + i * row_step;
          if (row < nrows)
            m = fmaxf(m, absmax_bf16x8(ld_shared_16(base + (row * vpr + col) * 16)));
        }
      }
    }
    // lanes with the same head: the vph-lane group, repeated every vpr lanes
    for (int off = 1; off < vph; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    for (int off = vpr; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane < vpr && lane % vph == 0) bars.warp_max[warp][my_head] = m;
    __syncthreads();
    if (threadIdx.x < hg) {
      float cm = bars.warp_max[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) cm = fmaxf(cm, bars.warp_max[w][threadIdx.x]);
      st_cluster_f32(cluster_map(&bars.part[parity][rank][threadIdx.x], 0), cm);
    }
    cluster_sync();
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < kCluster; ++r)
      amax = fmaxf(amax, ld_cluster_f32(cluster_map(&bars.part[parity][r][my_head], 0)));
    const float s = scale_from_amax(amax);
    const float rs = __frcp_rn(s);
    if (rank == 0 && warp == 0 && lane < vpr && lane % vph == 0)
      scale[static_cast<int64_t>(g.a) * hkv + g.c * hg + my_head] = s;
    // pass 2: quantise from shared memory (a slab held on chip), or read again in rounds
    for (int r = 0; r < g.rounds; ++r) {
      if (g.rounds > 1) issue_round(g, r);
      for (int b = 0; b < kBufs; ++b) {
        const int j = r * kChunksPerRound + b * kWarps + warp;
        if (j >= g.chunks) continue;
        if (g.rounds > 1) wait_buf(b);
        const int nrows = min(kRows, g.rows - j * kRows);
        const uint32_t base = smem_u32(buf(b));
        uint2* dst = reinterpret_cast<uint2*>(codes + (g.lo + j * kRows) * row_codes +
                                              static_cast<int64_t>(g.c) * hg * d) + col;
        for (int i = 0; i < vec_per_lane; ++i) {
          const int row = lane_row + i * row_step;
          if (row < nrows)
            st_hint_8(dst + row * (row_codes / 8),
                      quantize_bf16x8(ld_shared_16(base + (row * vpr + col) * 16), s, rs), pol);
        }
      }
    }
    // the first round of this cluster's next slab goes out while the others finish
    if (slab + n_clusters < slabs)
      issue_round(slab_geometry(slab + n_clusters, groups, rank, ao, T), 0);
    parity ^= 1;  // the next slab's maxima go to the other buffer (see the barrier note)
  }
  // CTA 0's shared memory must outlive every CTA's reads of it. (Within the loop, the
  // partials of slab k + 2 reuse slab k's buffer only after every CTA has passed slab
  // k + 1's barrier, hence after its reads of slab k.)
  cluster_sync();
}

// Given amax: codes of 8 elements per thread step (one 16-byte load, one 8-byte store),
// grid-stride over all T * Hkv * d elements; the (anchor, head) of a vector comes from
// its row (anchor: binary search of the offsets, cached per thread) and column.
__global__ void __launch_bounds__(256) kv_quantize_scaled_kernel(
    int num_anchors, int64_t T, int hkv, int d, const int32_t* __restrict__ ao,
    const float* __restrict__ amax, const __nv_bfloat16* __restrict__ x,
    uint8_t* __restrict__ codes, float* __restrict__ scale) {
  const int64_t vpr = static_cast<int64_t>(hkv) * d / 8;  // vectors per token row
  const int64_t total = T * vpr;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint64_t pol = l2_policy_evict_first();
  // scales: scale[a, g] from amax[a, g]
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < static_cast<int64_t>(num_anchors) * hkv; i += step)
    scale[i] = amax != nullptr ? scale_from_amax(__ldg(amax + i)) : 1.0f;  // no rows: 1
  int a = 0;
  int64_t a_lo = 0, a_hi = -1;  // rows of the cached anchor
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += step) {
    const int64_t row = v / vpr;
    if (row < a_lo || row >= a_hi) {  // the anchor holding this row (anchors are sorted)
      int lo = 0, hi = num_anchors - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(ao + mid) <= row) lo = mid; else hi = mid - 1;
      }
      a = lo;
      a_lo = __ldg(ao + a);
      a_hi = __ldg(ao + a + 1);
    }
    const int head = static_cast<int>((v % vpr) / (d / 8));
    const float s = scale_from_amax(__ldg(amax + static_cast<int64_t>(a) * hkv + head));
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x) + v);
    st_hint_8(reinterpret_cast<uint2*>(codes) + v, quantize_bf16x8(raw, s, __frcp_rn(s)), pol);
  }
}

}  // namespace

int quantize_heads_per_slab(int num_kv_heads, int head_dim) {
  // the largest power of two dividing Hkv with HG * d * 2 <= 256 bytes per token row
  int hg = 1;
  while (hg * 2 <= kMaxHeadsPerSlab && hkv_divides(num_kv_heads, hg * 2) &&
         hg * 2 * head_dim * 2 <= 256)
    hg *= 2;
  return hg;
}

cudaError_t launch_quantize_kv_fp8(const QuantArgs& q, int num_sms, cudaStream_t stream) {
  if (q.num_anchors == 0) return cudaSuccess;
  const int hg = quantize_heads_per_slab(q.num_kv_heads, q.head_dim);
  const int64_t slabs = static_cast<int64_t>(q.num_anchors) * (q.num_kv_heads / hg);
  cudaError_t e = cudaFuncSetAttribute(kv_quantize_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // persistent: as many clusters as can be resident at once (one CTA per SM)
  int max_clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / kCluster * kCluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kv_quantize_kernel, &cfg) != cudaSuccess ||
        max_clusters <= 0) {
      cudaGetLastError();
      max_clusters = num_sms / kCluster;
    }
  }
  const int64_t clusters = slabs < max_clusters ? slabs : max_clusters;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  kv_quantize_kernel<<<static_cast<unsigned>(clusters * kCluster), kThreads, kSmemBytes,
                       stream>>>(q.map, q.num_anchors, q.total_tokens, q.num_kv_heads,
                                 q.head_dim, hg, q.anchor_offsets, static_cast<uint8_t*>(q.codes),
                                 q.scale, q.err_word, q.timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv_fp8_scaled(const QuantArgs& q, const float* amax, int num_sms,
                                          cudaStream_t stream) {
  if (q.num_anchors == 0) return cudaSuccess;
  const int64_t vec = q.total_tokens * q.num_kv_heads * q.head_dim / 8;
  const int64_t need = (std::max<int64_t>(vec, int64_t{q.num_anchors} * q.num_kv_heads) + 255) / 256;
  const int blocks = static_cast<int>(std::min<int64_t>(need, int64_t{num_sms} * 8));
  kv_quantize_scaled_kernel<<<blocks, 256, 0, stream>>>(
      q.num_anchors, q.total_tokens, q.num_kv_heads, q.head_dim, q.anchor_offsets, amax,
      static_cast<const __nv_bfloat16*>(q.kv), static_cast<uint8_t*>(q.codes), q.scale);
  return cudaGetLastError();
}

}  // namespace quail
