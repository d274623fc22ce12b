// quantize.cu - per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of
// the qwen3-4b-fp8 model in the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
// GPU"). scale = amax / 448 (1 when amax == 0, IEEE fp32 division); code =
// e4m3_rn_satfinite(y) with y the correctly rounded fp32 quotient x / scale.
//
// Persistent clusters of 8 CTAs (3 CTAs per SM) take slabs = (anchor, group of up to
// 256 / (2 d) KV heads: up to 256 contiguous bytes of every token row). Pass 1 reads the
// slab and forms each head's max |x|; the CTA maxima meet in CTA 0's shared memory
// (distributed shared memory) and one cluster barrier later every CTA has the scales;
// pass 2 reads the slab again - largely from L2 - and writes the codes. Loads go through
// shared memory with cp.async (two rounds of 8 x 16 bytes per thread in flight, no
// registers held), each thread reading back only what it copied.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kClusterCtas = 8;
constexpr int kQWarps = 8;
constexpr int kQThreads = kQWarps * 32;
constexpr int kQCtasPerSm = 3;
constexpr int kVecPerRound = 8;  // 16-byte vectors per thread per round
constexpr int kQStages = 2;      // rounds in flight (cp.async into shared memory)
constexpr int kQSmemBytes = kQStages * kVecPerRound * kQThreads * 16;  // 64 KB
constexpr int kMaxHeadsPerSlab = 4;

// 16-byte asynchronous copy global -> shared (no registers held while in flight), with
// an L2 eviction policy.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
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

// Slab (a, c): rows ao[a] .. ao[a+1], heads c*HG .. c*HG + HG - 1: cvec = HG * d / 8
// 16-byte vectors per row (a divisor of 32). Vector f of the slab is row f / cvec, column
// f % cvec. The cluster reads 16,384 vectors per round; warp w of the cluster (0..63)
// takes f = round_base + (w * 8 + i) * 32 + lane for i < 8, so a lane's column, and head,
// is fixed: lane % cvec.
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kQThreads, kQCtasPerSm)
kv_quantize_kernel(int num_anchors, int64_t T, int hkv, int d, int hg,
                   const int32_t* __restrict__ ao, const __nv_bfloat16* __restrict__ x,
                   uint8_t* __restrict__ codes, float* __restrict__ scale) {
  __shared__ float part[2][kClusterCtas][kMaxHeadsPerSlab];  // CTA maxima, in CTA 0
  __shared__ float warp_max[kQWarps][kMaxHeadsPerSlab];
  extern __shared__ __align__(16) uint8_t stage_buf[];  // [kQStages][kVecPerRound][threads] x 16 B
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vph = d / 8;
  const int cvec = hg * vph;
  const int my_head = (lane % cvec) / vph;  // within the slab (fixed per lane)
  const int chunks = hkv / hg;
  const int64_t slabs = static_cast<int64_t>(num_anchors) * chunks;
  const int64_t n_clusters = gridDim.x / kClusterCtas;
  // cvec is a power of two dividing 32: vector f = (w * 8 + i) * 32 + lane of a round is
  // row (w * 8 + i) * (32 / cvec) + lane / cvec, column lane % cvec
  const int lc = __ffs(cvec) - 1;
  const int w_c = static_cast<int>(rank) * kQWarps + warp;  // warp within the cluster
  const int lane_row = lane >> lc, col = lane & (cvec - 1);
  const int rows_per_32 = 32 >> lc;
  const int row0 = w_c * kVecPerRound * rows_per_32 + lane_row;  // row of i = 0 in a round
  const int rows_per_round = kClusterCtas * kQWarps * kVecPerRound * rows_per_32;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint2* cv = reinterpret_cast<uint2*>(codes);
  const int64_t row_vec = static_cast<int64_t>(hkv) * vph;  // 16-byte vectors per token row
  const uint64_t keep = l2_policy_evict_last(), last_use = l2_policy_evict_first();
  // this thread's 16-byte slot i of stage st (consecutive threads: consecutive slots)
  const uint32_t slot0 = smem_u32(stage_buf) + threadIdx.x * 16u;
  auto slot = [&](int st, int i) {
    return slot0 + static_cast<uint32_t>((st * kVecPerRound + i) * kQThreads * 16);
  };
  int parity = 0;
  for (int64_t slab = blockIdx.x / kClusterCtas; slab < slabs; slab += n_clusters) {
    const int a = static_cast<int>(slab / chunks), c = static_cast<int>(slab % chunks);
    // offsets clamped into [0, T]: inconsistent ones cannot address out of bounds
    const int64_t lo = min(max(static_cast<int64_t>(__ldg(ao + a)), int64_t{0}), T);
    const int64_t hi = min(max(static_cast<int64_t>(__ldg(ao + a + 1)), lo), T);
    const int64_t nrows = hi - lo;
    const int64_t col_off = static_cast<int64_t>(c) * cvec + col;
    auto at = [&](int64_t row) {  // 16-byte index (8-byte index for the codes)
      return (lo + row) * row_vec + col_off;
    };
    const int rounds = static_cast<int>((nrows + rows_per_round - 1) / rows_per_round);
    // Round r of a pass: this thread's vectors (row r * rows_per_round + row0 + i * 32 /
    // cvec) copied into stage r % kQStages, one commit group per round (empty past the
    // end). A thread reads back only what it copied, so no block barrier is needed.
    auto issue = [&](int r, uint64_t pol) {
      if (r < rounds) {
#pragma unroll
        for (int i = 0; i < kVecPerRound; ++i) {
          const int64_t row = static_cast<int64_t>(r) * rows_per_round + row0 + i * rows_per_32;
          if (row < nrows) cp_async_16(slot(r % kQStages, i), xv + at(row), pol);
        }
      }
      cp_async_commit();
    };
    // pass 1: max |x| of this lane's head (the slab is kept in L2 for pass 2)
    float m = 0.f;
#pragma unroll
    for (int r = 0; r < kQStages; ++r) issue(r, keep);
    for (int r = 0; r < rounds; ++r) {
      cp_async_wait<kQStages - 1>();
#pragma unroll
      for (int i = 0; i < kVecPerRound; ++i) {
        const int64_t row = static_cast<int64_t>(r) * rows_per_round + row0 + i * rows_per_32;
        if (row < nrows) m = fmaxf(m, absmax_bf16x8(ld_shared_16(slot(r % kQStages, i))));
      }
      issue(r + kQStages, keep);
    }
    cp_async_wait<0>();
    // lanes with the same head: the vph-lane group, repeated every cvec lanes
    for (int off = 1; off < vph; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    for (int off = cvec; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane < cvec && lane % vph == 0) warp_max[warp][my_head] = m;
    __syncthreads();
    if (threadIdx.x < hg) {
      float cm = warp_max[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kQWarps; ++w) cm = fmaxf(cm, warp_max[w][threadIdx.x]);
      st_cluster_f32(cluster_map(&part[parity][rank][threadIdx.x], 0), cm);
    }
    cluster_sync();
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < kClusterCtas; ++r)
      amax = fmaxf(amax, ld_cluster_f32(cluster_map(&part[parity][r][my_head], 0)));
    const float s = scale_from_amax(amax);
    const float rs = __frcp_rn(s);
    if (rank == 0 && lane < cvec && lane % vph == 0 && warp == 0)
      scale[static_cast<int64_t>(a) * hkv + c * hg + my_head] = s;
    // pass 2: the slab again (mostly from L2; last use), quantised
#pragma unroll
    for (int r = 0; r < kQStages; ++r) issue(r, last_use);
    for (int r = 0; r < rounds; ++r) {
      cp_async_wait<kQStages - 1>();
#pragma unroll
      for (int i = 0; i < kVecPerRound; ++i) {
        const int64_t row = static_cast<int64_t>(r) * rows_per_round + row0 + i * rows_per_32;
        if (row < nrows)
          st_hint_8(cv + at(row), quantize_bf16x8(ld_shared_16(slot(r % kQStages, i)), s, rs),
                    last_use);
      }
      issue(r + kQStages, last_use);
    }
    cp_async_wait<0>();
    parity ^= 1;  // the next slab's maxima go to the other buffer (see the barrier note)
  }
  // CTA 0's shared memory must outlive every CTA's reads of it. (Within the loop, the
  // partials of slab k + 2 reuse slab k's buffer only after every CTA has passed slab
  // k + 1's barrier, hence after its reads of slab k.)
  cluster_sync();
}

}  // namespace

cudaError_t launch_quantize_kv_fp8(const QuantArgs& q, int num_sms, cudaStream_t stream) {
  if (q.num_anchors == 0) return cudaSuccess;
  // heads per slab: the largest power of two dividing Hkv with HG * d * 2 <= 256 bytes
  // (smaller slabs stay in L2 between the passes more often)
  int hg = 1;
  while (hg * 2 <= kMaxHeadsPerSlab && hkv_divides(q.num_kv_heads, hg * 2) &&
         hg * 2 * q.head_dim * 2 <= 256)
    hg *= 2;
  const int64_t slabs = static_cast<int64_t>(q.num_anchors) * (q.num_kv_heads / hg);
  const int64_t max_clusters = static_cast<int64_t>(num_sms) * kQCtasPerSm / kClusterCtas;
  const int64_t clusters = slabs < max_clusters ? slabs : max_clusters;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kv_quantize_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
  if (e != cudaSuccess) return e;
  kv_quantize_kernel<<<static_cast<unsigned>(clusters * kClusterCtas), kQThreads, kQSmemBytes,
                       stream>>>(
      q.num_anchors, q.total_tokens, q.num_kv_heads, q.head_dim, hg, q.anchor_offsets,
      static_cast<const __nv_bfloat16*>(q.kv), static_cast<uint8_t*>(q.codes), q.scale);
  return cudaGetLastError();
}

}  // namespace quail
