// quantize.cu - per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of
// the qwen3-4b-fp8 model in the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
// GPU"). scale = amax / 448 (1 when amax == 0); code = e4m3_rn_satfinite(x / scale),
// both divisions IEEE fp32.
//
// Bandwidth-bound steps on one stream: (1) zero the scale array, (2) amax of each
// (anchor, head) into it (fp32 bit patterns of non-negative values order like unsigned
// integers, so atomicMax on the bits is a float max), (3) quantise every element with the
// scale derived from the amax, (4) turn the amax entries into scales in place.
// Requires Hkv * d <= 4096 (checked on the host).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kQThreads = 256;
constexpr int kRowsPerBlock = 64;   // token rows per block (8 warps, one row per warp step)
constexpr int kMaxVecPerLane = 16;  // (Hkv * d / 8) / 32: Hkv * d <= 4096

__device__ __forceinline__ int find_anchor(const int32_t* __restrict__ ao, int A, int64_t row) {
  int lo = 0, hi = A - 1;  // largest a with ao[a] <= row (anchors may be empty)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(ao[mid]) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
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

// A block covers 64 consecutive token rows; its first anchor is found once. Warps take
// rows round-robin and keep, per 16-byte vector slot of the row, the running max of the
// current anchor; when a warp's row moves to the next anchor (rare) and at the end, the
// maxima are reduced over the lanes of each head and merged with one atomicMax per
// (anchor, head) (fp32 bit patterns of non-negative values order like unsigned ints).
__global__ void __launch_bounds__(kQThreads)
kv_amax_kernel(int A, const int32_t* __restrict__ ao, int64_t T, int hkv, int d,
               const __nv_bfloat16* __restrict__ x, unsigned* __restrict__ amax_bits) {
  __shared__ int a_first;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int64_t r1 = min(r0 + kRowsPerBlock, T);
  if (threadIdx.x == 0) a_first = find_anchor(ao, A, r0);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vpr = hkv * d / 8;  // 16-byte vectors per row
  const int vph = d / 8;        // vectors per head: 8 or 16, divides 32
  float m[kMaxVecPerLane];
#pragma unroll
  for (int i = 0; i < kMaxVecPerLane; ++i) m[i] = 0.f;
  auto flush = [&](int a) {
#pragma unroll
    for (int i = 0; i < kMaxVecPerLane; ++i) {
      if (i * 32 >= vpr) break;
      float v = m[i];
      for (int off = vph >> 1; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
      const int vec = i * 32 + lane;
      if (vec < vpr && (lane & (vph - 1)) == 0 && v > 0.f)
        atomicMax(amax_bits + static_cast<int64_t>(a) * hkv + vec / vph, __float_as_uint(v));
      m[i] = 0.f;
    }
  };
  int a = a_first;
  bool any = false;
  for (int64_t r = r0 + warp; r < r1; r += kQThreads / 32) {
    while (static_cast<int64_t>(__ldg(ao + a + 1)) <= r) {  // warp-uniform
      if (any) flush(a);
      any = false;
      ++a;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + r * hkv * d);
#pragma unroll
    for (int i = 0; i < kMaxVecPerLane; ++i) {
      const int vec = i * 32 + lane;
      if (i * 32 < vpr && vec < vpr) m[i] = fmaxf(m[i], absmax_bf16x8(__ldg(row + vec)));
    }
    any = true;
  }
  if (any) flush(a);
}

__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// Same row partition; every element becomes e4m3_rn_satfinite(x / scale) with the scale
// of its (anchor, head), both divisions IEEE fp32.
__global__ void __launch_bounds__(kQThreads)
kv_quantize_kernel(int A, const int32_t* __restrict__ ao, int64_t T, int hkv, int d,
                   const __nv_bfloat16* __restrict__ x, const float* __restrict__ amax,
                   uint8_t* __restrict__ codes) {
  __shared__ int a_first;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int64_t r1 = min(r0 + kRowsPerBlock, T);
  if (threadIdx.x == 0) a_first = find_anchor(ao, A, r0);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vpr = hkv * d / 8;
  const int vph = d / 8;
  int a = a_first;
  for (int64_t r = r0 + warp; r < r1; r += kQThreads / 32) {
    while (static_cast<int64_t>(__ldg(ao + a + 1)) <= r) ++a;
    const uint4* row = reinterpret_cast<const uint4*>(x + r * hkv * d);
    uint2* out = reinterpret_cast<uint2*>(codes + r * hkv * d);
#pragma unroll
    for (int i = 0; i < kMaxVecPerLane; ++i) {
      const int vec = i * 32 + lane;
      if (i * 32 >= vpr || vec >= vpr) continue;
      const float s = scale_from_amax(__ldg(amax + static_cast<int64_t>(a) * hkv + vec / vph));
      const uint4 raw = __ldg(row + vec);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 qv = make_float2(__fdiv_rn(__uint_as_float(w[k] << 16), s),
                                      __fdiv_rn(__uint_as_float(w[k] & 0xFFFF0000u), s));
        const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
        packed[k >> 1] |= static_cast<uint32_t>(c) << (16 * (k & 1));
      }
      out[vec] = make_uint2(packed[0], packed[1]);
    }
  }
}

__global__ void amax_to_scale_kernel(int64_t n, float* __restrict__ s) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) s[i] = scale_from_amax(s[i]);
}

}  // namespace

cudaError_t launch_quantize_kv_fp8(const QuantArgs& q, int num_sms, cudaStream_t stream) {
  const int64_t n_scale = static_cast<int64_t>(q.num_anchors) * q.num_kv_heads;
  if (n_scale == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(q.scale, 0, n_scale * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t T = q.total_tokens;
  if (T > 0) {
    const int64_t blocks = (T + kRowsPerBlock - 1) / kRowsPerBlock;
    kv_amax_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, stream>>>(
        q.num_anchors, q.anchor_offsets, T, q.num_kv_heads, q.head_dim,
        static_cast<const __nv_bfloat16*>(q.kv), reinterpret_cast<unsigned*>(q.scale));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kv_quantize_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, stream>>>(
        q.num_anchors, q.anchor_offsets, T, q.num_kv_heads, q.head_dim,
        static_cast<const __nv_bfloat16*>(q.kv), q.scale, static_cast<uint8_t*>(q.codes));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  amax_to_scale_kernel<<<static_cast<unsigned>((n_scale + 255) / 256), 256, 0, stream>>>(
      n_scale, q.scale);
  return cudaGetLastError();
}

}  // namespace quail
