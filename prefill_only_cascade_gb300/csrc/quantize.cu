// quantize.cu - per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of
// the qwen3-4b-fp8 model in the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
// GPU"). scale = amax / 448 (1 when amax == 0); code = e4m3_rn_satfinite(x / scale),
// both divisions IEEE fp32.
//
// Three bandwidth-bound steps on one stream: (1) zero the scale array, (2) amax of each
// (anchor, head) into it (fp32 bit patterns of non-negative values order like unsigned
// integers, so atomicMax on the bits is a float max), (3) quantise every element with the
// scale derived from the amax, (4) turn the amax entries into scales in place.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kQThreads = 256;
constexpr int kRowsPerBlock = 16;  // token rows per amax block

__device__ __forceinline__ int find_anchor(const int32_t* __restrict__ ao, int A, int64_t row) {
  int lo = 0, hi = A - 1;  // largest a with ao[a] <= row (anchors may be empty)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(ao[mid]) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kQThreads)
kv_amax_kernel(int A, const int32_t* __restrict__ ao, int64_t T, int hkv, int d,
               const __nv_bfloat16* __restrict__ x, unsigned* __restrict__ amax_bits) {
  // A block covers kRowsPerBlock token rows; each thread reduces 8-element vectors.
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  const int vec_per_row = hkv * d / 8;
  const int vec_per_head = d / 8;
  const int64_t nvec = static_cast<int64_t>(kRowsPerBlock) * vec_per_row;
  for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int64_t row = row0 + v / vec_per_row;
    const bool valid = row < T;  // no early exit: every lane takes part in the shuffles
    const int head = static_cast<int>((v % vec_per_row) / vec_per_head);
    const uint4 raw = valid ? *reinterpret_cast<const uint4*>(
                                  x + (row * vec_per_row + v % vec_per_row) * 8)
                            : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    // lanes holding the same head of the same row are contiguous groups of d/8 lanes
    // when d/8 divides 32; reduce inside the group before the atomic.
    const int grp = vec_per_head < 32 ? vec_per_head : 32;
    for (int off = grp >> 1; off > 0; off >>= 1)
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (valid && (threadIdx.x & (grp - 1)) == 0 && m > 0.f) {
      const int a = find_anchor(ao, A, row);
      atomicMax(amax_bits + static_cast<int64_t>(a) * hkv + head, __float_as_uint(m));
    }
  }
}

__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

__global__ void __launch_bounds__(kQThreads)
kv_quantize_kernel(int A, const int32_t* __restrict__ ao, int64_t T, int hkv, int d,
                   const __nv_bfloat16* __restrict__ x, const float* __restrict__ amax,
                   uint8_t* __restrict__ codes) {
  const int vec_per_row = hkv * d / 8;
  const int64_t nvec = T * vec_per_row;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = v / vec_per_row;
    const int head = static_cast<int>((v % vec_per_row) / (d / 8));
    const int a = find_anchor(ao, A, row);
    const float s = scale_from_amax(amax[static_cast<int64_t>(a) * hkv + head]);
    const uint4 raw = *reinterpret_cast<const uint4*>(x + v * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q = make_float2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                                   __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
      const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
      packed[i >> 1] |= static_cast<uint32_t>(c) << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(codes + v * 8) = make_uint2(packed[0], packed[1]);
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
    const int64_t nvec = T * q.num_kv_heads * q.head_dim / 8;
    int64_t grid = (nvec + kQThreads - 1) / kQThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    kv_quantize_kernel<<<static_cast<unsigned>(grid), kQThreads, 0, stream>>>(
        q.num_anchors, q.anchor_offsets, T, q.num_kv_heads, q.head_dim,
        static_cast<const __nv_bfloat16*>(q.kv), q.scale, static_cast<uint8_t*>(q.codes));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  amax_to_scale_kernel<<<static_cast<unsigned>((n_scale + 255) / 256), 256, 0, stream>>>(
      n_scale, q.scale);
  return cudaGetLastError();
}

}  // namespace quail
